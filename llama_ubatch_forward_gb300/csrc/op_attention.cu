// lcx_attention: the attention step of the forward as a stand-alone call over caller-owned
// buffers (one layer of a paged f16 KV cache), running the same split-K kernel lcx_decode uses.
#include <cstring>
#include <string>

#include "../../include/lcx.h"
#include "lcx_internal.h"

using namespace lcx;

namespace lcx {
void set_error_text(const char *msg);
}

static bool attn_args_ok(int32_t T, int32_t n_head, int32_t n_head_kv, int32_t head_dim, const float *q,
                         const void *k_cache, const void *v_cache, int32_t n_pages, const int32_t *page_table,
                         int32_t max_pages, const int32_t *pos, const int32_t *seq, int32_t max_pos, const float *out) {
    if (T <= 0 || n_head <= 0 || n_head_kv <= 0 || n_head % n_head_kv) return false;
    const int g = n_head / n_head_kv;
    if (g != 1 && g != 2 && g != 4 && g != 8) return false;
    if (head_dim != 64 && head_dim != 128) return false;
    if (!q || !k_cache || !v_cache || !page_table || !pos || !seq || !out) return false;
    if (n_pages <= 0 || max_pages <= 0 || max_pos < 0 || (int64_t)max_pos >= (int64_t)max_pages * kPage) return false;
    return true;
}

namespace lcx {
FwdArgs attn_fwd_args(int32_t T, int32_t n_head, int32_t n_head_kv, int32_t head_dim, const float *q,
                      const void *k_cache, const void *v_cache, int32_t n_pages, const int32_t *page_table,
                      int32_t max_pages, const int32_t *pos, const int32_t *seq, float *out) {
    FwdArgs a{};
    a.H = n_head;
    a.KV = n_head_kv;
    a.hd = head_dim;
    a.T = T;
    a.q = const_cast<float *>(q);
    a.kc = (__half *)k_cache;
    a.vc = (__half *)v_cache;
    a.n_pages = n_pages;
    a.pt = const_cast<int32_t *>(page_table);
    a.max_pages_per_seq = max_pages;
    a.ub.pos = pos;
    a.ub.seq = seq;
    a.o32 = out;
    a.att_max_split = 64;
    return a;
}
}  // namespace lcx

extern "C" size_t lcx_attention_workspace_size(int32_t T, int32_t n_head, int32_t n_head_kv, int32_t head_dim,
                                              int32_t max_pos) {
    if (T <= 0 || n_head <= 0 || n_head_kv <= 0 || max_pos < 0) return 0;
    FwdArgs a{};
    a.H = n_head;
    a.KV = n_head_kv;
    a.hd = head_dim;
    a.T = T;
    a.att_max_split = 64;
    return attention_scratch_bytes(a, max_pos + 1, nullptr);
}

extern "C" int32_t lcx_attention(int32_t T, int32_t n_head, int32_t n_head_kv, int32_t head_dim, const float *q,
                                 const void *k_cache, const void *v_cache, int32_t n_pages, const int32_t *page_table,
                                 int32_t max_pages, const int32_t *pos, const int32_t *seq, int32_t max_pos, float *out,
                                 void *workspace, size_t workspace_bytes, void *cuda_stream) {
    if (!attn_args_ok(T, n_head, n_head_kv, head_dim, q, k_cache, v_cache, n_pages, page_table, max_pages, pos, seq,
                      max_pos, out))
        return LCX_INVALID;
    FwdArgs a = attn_fwd_args(T, n_head, n_head_kv, head_dim, q, k_cache, v_cache, n_pages, page_table, max_pages, pos,
                              seq, out);
    size_t cnt_off = 0;
    const size_t need = attention_scratch_bytes(a, max_pos + 1, &cnt_off);
    if (need > 0 && (!workspace || workspace_bytes < need)) {
        set_error_text("lcx_attention: workspace smaller than lcx_attention_workspace_size()");
        return LCX_INVALID;
    }
    cudaStream_t s = (cudaStream_t)cuda_stream;
    cudaError_t e = cudaSuccess;
    if (need > 0) {
        a.att_part = (float *)workspace;
        a.att_cnt = (int32_t *)((uint8_t *)workspace + cnt_off);
        e = cudaMemsetAsync(a.att_cnt, 0, (size_t)T * n_head_kv * sizeof(int32_t), s);
    }
    int64_t launches = 0;
    if (e == cudaSuccess) e = launch_attention(a, 0, max_pos + 1, false, s, launches);
    if (e != cudaSuccess) {
        set_error_text(cudaGetErrorString(e));
        return LCX_COMPUTE_FAILED;
    }
    return LCX_OK;
}
