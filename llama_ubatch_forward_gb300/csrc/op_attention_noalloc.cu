// lcx_attention_noalloc: lcx_attention for callers that cannot allocate device memory.
//
// Some callers have no way to hand the library a workspace: a plugin whose host application
// owns every device allocation, a process whose device memory is already fully reserved by a
// framework's caching allocator, or a latency-critical path that cannot afford cudaMalloc's
// implicit device synchronisation. For them the split-K partials and arrival counters live in
// a fixed file-scope device array instead of a caller buffer. That array exists on every GPU
// that loads this library, for the life of the process.
#include <mutex>

#include "../../include/lcx.h"
#include "lcx_internal.h"

using namespace lcx;

namespace lcx {
void set_error_text(const char *msg);
FwdArgs attn_fwd_args(int32_t T, int32_t n_head, int32_t n_head_kv, int32_t head_dim, const float *q,
                      const void *k_cache, const void *v_cache, int32_t n_pages, const int32_t *page_table,
                      int32_t max_pages, const int32_t *pos, const int32_t *seq, float *out);
}  // namespace lcx

namespace {

// Partials first, then the arrival counters (the same layout lcx_attention uses in a workspace).
static __device__ __align__(256) unsigned char g_attn_scratch[LCX_ATTENTION_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of g_attn_scratch on the current device. In host code the symbol is only a
// host-side stand-in, so the address is looked up once per device (with it current) and kept.
cudaError_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_attn_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" int32_t lcx_attention_noalloc(int32_t T, int32_t n_head, int32_t n_head_kv, int32_t head_dim,
                                         const float *q, const void *k_cache, const void *v_cache, int32_t n_pages,
                                         const int32_t *page_table, int32_t max_pages, const int32_t *pos,
                                         const int32_t *seq, int32_t max_pos, float *out, void *cuda_stream) {
    if (T <= 0 || n_head <= 0 || n_head_kv <= 0 || n_head % n_head_kv || (head_dim != 64 && head_dim != 128))
        return LCX_INVALID;
    const int g = n_head / n_head_kv;
    if (g != 1 && g != 2 && g != 4 && g != 8) return LCX_INVALID;
    if (!q || !k_cache || !v_cache || !page_table || !pos || !seq || !out) return LCX_INVALID;
    if (n_pages <= 0 || max_pages <= 0 || max_pos < 0 || (int64_t)max_pos >= (int64_t)max_pages * kPage)
        return LCX_INVALID;
    FwdArgs a = attn_fwd_args(T, n_head, n_head_kv, head_dim, q, k_cache, v_cache, n_pages, page_table, max_pages,
                              pos, seq, out);
    size_t cnt_off = 0;
    const size_t need = attention_scratch_bytes(a, max_pos + 1, &cnt_off);
    if (need > (size_t)LCX_ATTENTION_NOALLOC_SCRATCH_BYTES) {
        set_error_text("lcx_attention_noalloc: this call needs more scratch than the fixed "
                       "LCX_ATTENTION_NOALLOC_SCRATCH_BYTES; use lcx_attention with a workspace");
        return LCX_INVALID;
    }
    cudaStream_t s = (cudaStream_t)cuda_stream;
    cudaError_t e = cudaSuccess;
    if (need > 0) {
        void *base = nullptr;
        e = scratch_address(&base);
        if (e == cudaSuccess) {
            a.att_part = (float *)base;
            a.att_cnt = (int32_t *)((uint8_t *)base + cnt_off);
            // the array keeps the previous call's contents: the counters must start at zero
            e = cudaMemsetAsync(a.att_cnt, 0, (size_t)T * n_head_kv * sizeof(int32_t), s);
        }
    }
    int64_t launches = 0;
    if (e == cudaSuccess) e = launch_attention(a, 0, max_pos + 1, false, s, launches);
    if (e != cudaSuccess) {
        set_error_text(cudaGetErrorString(e));
        return LCX_COMPUTE_FAILED;
    }
    return LCX_OK;
}
