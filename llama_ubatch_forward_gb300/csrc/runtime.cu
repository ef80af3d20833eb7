// Host runtime of the lcx C ABI (include/lcx.h): model re-layout, context and KV-cell
// bookkeeping, batch validation and filling, ubatch split, and the per-ubatch kernel plan.
//
// The flow of lcx_decode follows steps 11-13 of the article "How inference works in
// llama.cpp": the batch is validated and its positions / output flags filled
// (llama_batch_allocr::init), the whole batch is cut into ubatches of at most n_ubatch
// consecutive tokens and cells are reserved for all of them before any runs (init_batch,
// split_simple, prepare: return 1 with nothing committed when they do not fit), then each
// ubatch is run in order (process_ubatch) and its logits rows are appended in batch order.
// A failed or aborted ubatch releases its cells and those of later ubatches.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <set>
#include <tuple>
#include <string>
#include <vector>

#include "../../include/lcx.h"
#include "lcx_internal.h"

using namespace lcx;

namespace {

std::mutex g_err_mu;
std::string g_err;

void set_err(const char *what, cudaError_t e) {
    std::lock_guard<std::mutex> lk(g_err_mu);
    g_err = std::string(what) + ": " + cudaGetErrorString(e);
}

int round_up(int x, int m) { return (x + m - 1) / m * m; }

}  // namespace

namespace lcx {
void set_error_text(const char *msg) {
    std::lock_guard<std::mutex> lk(g_err_mu);
    g_err = msg;
}

namespace {
std::mutex g_attr_mu;
std::set<std::tuple<const void *, int, int>> g_attr_done;   // (kernel, device, attribute)
std::map<int, int> g_sm_count;                               // device -> SMs
}  // namespace

cudaError_t func_attr_once(const void *kern, cudaFuncAttribute attr, int value) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(g_attr_mu);
    const auto key = std::make_tuple(kern, dev, (int)attr);
    if (g_attr_done.count(key)) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, attr, value);
    if (e == cudaSuccess) g_attr_done.insert(key);
    return e;
}

int device_sm_count() {
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lk(g_attr_mu);
    auto it = g_sm_count.find(dev);
    if (it != g_sm_count.end()) return it->second;
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) return 1;
    g_sm_count[dev] = n;
    return n;
}
}  // namespace lcx

namespace {

bool valid_block_type(int t) { return t == LCX_Q4_0 || t == LCX_Q8_0; }

}  // namespace

// =========================================================================== model
struct lcx_model {
    lcx_hparams hp{};
    int device = 0;
    int F_pad = 0;
    const void *tok_embd = nullptr;
    const float *output_norm = nullptr;
    std::vector<DevLayer> layers;
    QMat head;
    void *arena = nullptr;
    size_t arena_bytes = 0;
};

static bool check_hparams(const lcx_hparams *hp) {
    if (!hp) return false;
    if (hp->n_vocab <= 0 || hp->n_embd <= 0 || hp->n_layer <= 0 || hp->n_head <= 0 || hp->n_head_kv <= 0 ||
        hp->head_dim <= 0 || hp->n_ff <= 0)
        return false;
    if (hp->n_embd % 64 || hp->head_dim % 2 || (hp->n_head * hp->head_dim) % 64) return false;
    if (hp->head_dim != 64 && hp->head_dim != 128) return false;
    if (hp->n_head % hp->n_head_kv) return false;
    const int g = hp->n_head / hp->n_head_kv;
    if (g != 1 && g != 2 && g != 4 && g != 8) return false;
    if (!valid_block_type(hp->t_linear)) return false;
    if (hp->t_embd != LCX_F16 && !valid_block_type(hp->t_embd)) return false;
    if (!(hp->rms_eps >= 0.f) || !(hp->rope_theta > 0.f)) return false;
    return true;
}

static void plan_qmat(QMat &q, int type, int N, int N_pad, int K_pad) {
    q.type = type;
    q.N = N;
    q.N_pad = N_pad;
    q.K = K_pad;
    q.nb = K_pad / 32;
}

extern "C" lcx_model *lcx_model_create(const lcx_hparams *hp, const lcx_weights *w, int32_t *err) {
    if (err) *err = LCX_OK;
    if (!check_hparams(hp) || !w || !w->tok_embd || !w->output_norm || !w->layers) {
        if (err) *err = LCX_INVALID;
        return nullptr;
    }
    const int t_out = w->output ? hp->t_out : hp->t_embd;
    if (!valid_block_type(t_out)) {
        if (err) *err = LCX_INVALID;
        return nullptr;
    }
    for (int l = 0; l < hp->n_layer; ++l) {
        const lcx_layer_w &L = w->layers[l];
        if (!L.attn_norm || !L.wq || !L.wk || !L.wv || !L.wo || !L.ffn_norm || !L.w_gate || !L.w_up || !L.w_down) {
            if (err) *err = LCX_INVALID;
            return nullptr;
        }
    }
    lcx_model *m = new lcx_model;
    m->hp = *hp;
    cudaGetDevice(&m->device);
    m->tok_embd = w->tok_embd;
    m->output_norm = (const float *)w->output_norm;
    const int d = hp->n_embd, hd = hp->head_dim, H = hp->n_head, KV = hp->n_head_kv, F = hp->n_ff;
    m->F_pad = round_up(F, kRowTile);
    m->layers.resize(hp->n_layer);
    size_t total = 0;
    std::vector<QMat *> mats;
    for (int l = 0; l < hp->n_layer; ++l) {
        DevLayer &D = m->layers[l];
        D.attn_norm = (const float *)w->layers[l].attn_norm;
        D.ffn_norm = (const float *)w->layers[l].ffn_norm;
        const int nqkv = (H + 2 * KV) * hd;
        plan_qmat(D.qkv, hp->t_linear, nqkv, round_up(nqkv, kRowTile), d);
        plan_qmat(D.wo, hp->t_linear, d, round_up(d, kRowTile), H * hd);
        plan_qmat(D.gateup, hp->t_linear, 2 * m->F_pad, 2 * m->F_pad, d);
        plan_qmat(D.down, hp->t_linear, d, round_up(d, kRowTile), m->F_pad);
        mats.push_back(&D.qkv);
        mats.push_back(&D.wo);
        mats.push_back(&D.gateup);
        mats.push_back(&D.down);
    }
    plan_qmat(m->head, t_out, hp->n_vocab, round_up(hp->n_vocab, kRowTile), d);
    mats.push_back(&m->head);
    for (QMat *q : mats) total += (q->bytes() + 255) / 256 * 256;
    cudaError_t e = cudaMalloc(&m->arena, total);
    if (e != cudaSuccess) {
        set_err("model arena", e);
        delete m;
        if (err) *err = LCX_ALLOC_FAILED;
        return nullptr;
    }
    m->arena_bytes = total;
    uint8_t *p = (uint8_t *)m->arena;
    for (QMat *q : mats) {
        q->w = p;
        p += (q->bytes() + 255) / 256 * 256;
    }
    cudaStream_t s = nullptr;
    e = cudaMemsetAsync(m->arena, 0, total, s);
    for (int l = 0; l < hp->n_layer && e == cudaSuccess; ++l) {
        DevLayer &D = m->layers[l];
        const lcx_layer_w &L = w->layers[l];
        const int nbd = d / 32;
        if (e == cudaSuccess) e = launch_repack(L.wq, hp->t_linear, H * hd, nbd, D.qkv, 0, 0, s);
        if (e == cudaSuccess) e = launch_repack(L.wk, hp->t_linear, KV * hd, nbd, D.qkv, H * hd, 0, s);
        if (e == cudaSuccess) e = launch_repack(L.wv, hp->t_linear, KV * hd, nbd, D.qkv, (H + KV) * hd, 0, s);
        if (e == cudaSuccess) e = launch_repack(L.wo, hp->t_linear, d, (H * hd) / 32, D.wo, 0, 0, s);
        if (e == cudaSuccess) e = launch_repack(L.w_gate, hp->t_linear, F, nbd, D.gateup, 0, 1, s);
        if (e == cudaSuccess) e = launch_repack(L.w_up, hp->t_linear, F, nbd, D.gateup, 4, 1, s);
        if (e == cudaSuccess) e = launch_repack(L.w_down, hp->t_linear, d, (F + 31) / 32, D.down, 0, 0, s);
    }
    if (e == cudaSuccess)
        e = launch_repack(w->output ? w->output : w->tok_embd, t_out, hp->n_vocab, d / 32, m->head, 0, 0, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    for (QMat *q : mats)
        if (e == cudaSuccess && !make_weight_maps(*q)) e = cudaErrorInvalidValue;
    if (e != cudaSuccess) {
        set_err("model re-layout", e);
        cudaFree(m->arena);
        delete m;
        if (err) *err = LCX_COMPUTE_FAILED;
        return nullptr;
    }
    return m;
}

extern "C" void lcx_model_free(lcx_model *m) {
    if (!m) return;
    if (m->arena) cudaFree(m->arena);
    delete m;
}

// =========================================================================== context
namespace {

struct Plan {                    // one validated, filled batch
    std::vector<int32_t> tok, pos, seq, cell;
    std::vector<int8_t> flag;
    std::vector<int32_t> pt_idx, pt_page, pt_tok;   // page-table updates and the first token that uses each
};

struct SeqState {
    std::vector<int32_t> pages;  // page ids in position order
    int32_t len = 0;             // cells used = last position + 1
};

}  // namespace

struct lcx_ctx {
    lcx_model *m = nullptr;
    lcx_hparams hp{};
    bool host_only = false;
    int fail_ubatch = -1;   // host-only contexts: this ubatch of the next lcx_decode fails (-3)
    bool kv_unified = true; // one cell store for all sequences; else a stream of n_ctx / n_seq_max per sequence
    uint32_t n_ctx = 0, n_seq_max = 0, n_ubatch = 0;
    cudaStream_t stream = nullptr;
    int n_pages = 0, max_pages_per_seq = 0;
    std::vector<int32_t> free_pages;
    std::vector<SeqState> seqs;
    int64_t cells_used = 0;
    int (*abort_cb)(void *) = nullptr;
    void *abort_ud = nullptr;
    lcx_stats st{};
    int32_t n_outputs_last = 0;

    // device state
    __half *kc = nullptr, *vc = nullptr;
    int32_t *pt = nullptr;
    float2 *rope = nullptr;
    void *ws = nullptr;          // workspace arena
    FwdArgs base{};              // pointers into ws
    int32_t *amax_dev = nullptr; // [cap] argmax per output row of a call
    int meta_cap = 0;            // int32 slots of the metadata region
    int32_t *meta_dev = nullptr;
    int32_t *meta_host = nullptr;  // pinned staging (2 halves, each meta_cap)
    cudaEvent_t meta_ev[2] = {nullptr, nullptr};
    int meta_slot = 0;
    int32_t *amax_host = nullptr;  // pinned argmax staging
    int32_t *status_host = nullptr; // pinned copy of the device error and non-finite words
    int amax_cap = 0;
    int max_att_split = 64;
    DecodeStep step;             // persistent one-token decode step, prepared at first use
    // profiling
    bool prof_on = false;
    std::vector<cudaEvent_t> prof_ev;      // pairs
    struct ProfRec { int cls; double bytes, flops; };
    std::vector<ProfRec> prof_rec;
    lcx_profile prof{};
    // in-kernel launch timeline (lcx_set_profiling mode 2)
    unsigned long long *trace = nullptr;
    int trace_cap = 0, trace_used = 0;
};

static void prof_resolve(lcx_ctx *c);
static int32_t trace_on(lcx_ctx *c);

static void free_ctx_device(lcx_ctx *c) {
    decode_step_release(c->step);
    for (auto e : c->prof_ev) cudaEventDestroy(e);
    c->prof_ev.clear();
    if (c->trace) cudaFree(c->trace);
    if (c->kc) cudaFree(c->kc);
    if (c->vc) cudaFree(c->vc);
    if (c->pt) cudaFree(c->pt);
    if (c->rope) cudaFree(c->rope);
    if (c->ws) cudaFree(c->ws);
    if (c->meta_dev) cudaFree(c->meta_dev);
    if (c->meta_host) cudaFreeHost(c->meta_host);
    if (c->amax_host) cudaFreeHost(c->amax_host);
    if (c->status_host) cudaFreeHost(c->status_host);
    for (auto &e : c->meta_ev)
        if (e) cudaEventDestroy(e);
}

static void init_cells(lcx_ctx *c) {
    c->n_pages = (int)((c->n_ctx + kPage - 1) / kPage) + (int)c->n_seq_max;
    c->max_pages_per_seq = (int)((c->n_ctx + kPage - 1) / kPage);
    c->free_pages.clear();
    for (int p = c->n_pages - 1; p >= 0; --p) c->free_pages.push_back(p);
    c->seqs.assign(c->n_seq_max, SeqState{});
    c->cells_used = 0;
    c->st.n_ctx = c->n_ctx;
    c->st.n_pages = (uint32_t)c->n_pages;
}

static lcx_ctx *make_ctx_common(const lcx_hparams *hp, uint32_t n_ctx, uint32_t n_seq_max, uint32_t n_ubatch) {
    if (!check_hparams(hp) || n_ctx == 0 || n_seq_max == 0 || n_ubatch == 0) return nullptr;
    if (n_ctx > (1u << 24) || n_seq_max > 65536 || n_ubatch > 65536) return nullptr;
    lcx_ctx *c = new lcx_ctx;
    c->hp = *hp;
    c->n_ctx = (n_ctx + 255u) / 256u * 256u;   // rounded up to a multiple of 256 (step 7)
    c->n_seq_max = n_seq_max;
    c->n_ubatch = std::min(n_ubatch, c->n_ctx);  // n_ubatch <= n_batch = n_ctx for a causal model
    init_cells(c);
    return c;
}

extern "C" lcx_ctx *lcx_ctx_create_host_only(const lcx_hparams *hp, uint32_t n_ctx, uint32_t n_seq_max,
                                             uint32_t n_ubatch) {
    lcx_ctx *c = make_ctx_common(hp, n_ctx, n_seq_max, n_ubatch);
    if (c) c->host_only = true;
    return c;
}

extern "C" int32_t lcx_ctx_inject_failure(lcx_ctx *c, int32_t ubatch) {
    if (!c || !c->host_only) return LCX_INVALID;
    c->fail_ubatch = ubatch;
    return LCX_OK;
}

template <class T>
static T *carve(uint8_t *&p, size_t n) {
    T *r = (T *)p;
    p += (n * sizeof(T) + 255) / 256 * 256;
    return r;
}

extern "C" lcx_ctx *lcx_ctx_create(lcx_model *m, uint32_t n_ctx, uint32_t n_seq_max, uint32_t n_ubatch,
                                   void *cuda_stream) {
    if (!m) return nullptr;
    lcx_ctx *c = make_ctx_common(&m->hp, n_ctx, n_seq_max, n_ubatch);
    if (!c) return nullptr;
    c->m = m;
    c->stream = (cudaStream_t)cuda_stream;
    const lcx_hparams &hp = m->hp;
    const int d = hp.n_embd, H = hp.n_head, KV = hp.n_head_kv, hd = hp.head_dim, L = hp.n_layer;
    const int T = (int)c->n_ubatch, V = hp.n_vocab, Fp = m->F_pad;
    const size_t kv_elems = (size_t)L * c->n_pages * KV * kPage * hd;
    cudaError_t e = cudaSuccess;
    auto ok = [&](cudaError_t r, const char *what) {
        if (r != cudaSuccess && e == cudaSuccess) {
            e = r;
            set_err(what, r);
        }
        return e == cudaSuccess;
    };
    ok(cudaMalloc(&c->kc, kv_elems * sizeof(__half)), "kv cache");
    if (e == cudaSuccess) ok(cudaMalloc(&c->vc, kv_elems * sizeof(__half)), "kv cache");
    // finite contents everywhere: the prefill attention reads whole pages and gives the cells past
    // a query's position a weight of exactly 0
    if (e == cudaSuccess) ok(cudaMemsetAsync(c->kc, 0, kv_elems * sizeof(__half), c->stream), "kv cache");
    if (e == cudaSuccess) ok(cudaMemsetAsync(c->vc, 0, kv_elems * sizeof(__half), c->stream), "kv cache");
    if (e == cudaSuccess)
        ok(cudaMalloc(&c->pt, (size_t)c->n_seq_max * c->max_pages_per_seq * sizeof(int32_t)), "page table");
    if (e == cudaSuccess) ok(cudaMalloc(&c->rope, (size_t)c->n_ctx * (hd / 2) * sizeof(float2)), "rope table");
    // workspace
    int n_sm = 0;
    cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, m->device);
    // attention partials: the split-K attention's (max, sum, acc) rows, see attention_splits
    const size_t part_rows = std::max<size_t>((size_t)2 * 4 * (n_sm > 0 ? n_sm : 160) + (size_t)T * KV,
                                              std::min<size_t>((size_t)T * KV * 16, 16384));
    const int G = H / KV;
    size_t ws = 0;
    const size_t sizes[] = {
        (size_t)T * d * 4,                   // x
        (size_t)T * d * 2,                   // xh
        (size_t)T * d * 2,                   // xh_lo
        (size_t)T * H * hd * 4,              // q
        (size_t)T * H * hd * 4,              // o32
        (size_t)T * H * hd * 2,              // o16
        (size_t)T * H * hd * 2,              // o16_lo
        (size_t)T * Fp * 4,                  // h32
        (size_t)T * Fp * 2,                  // h16
        (size_t)T * Fp * 2,                  // h16_lo
        (size_t)T * V * 4,                   // logits scratch
        (size_t)T * 8,                       // argmax keys
        part_rows * G * (hd + 2) * 4,        // attention partials
        (size_t)T * KV * 4,                  // attention counters
        (size_t)std::max<int>(T, 4096) * 4,  // argmax per output row
        256,                                 // device error word
        T > kGemvMaxT ? kGemmPartBytes : 0,  // split-K partial sums of the tensor-core GEMM
        T > kGemvMaxT ? (size_t)kGemmMaxTiles * 4 : 0,   // their per-tile counters
    };
    for (size_t s : sizes) ws += (s + 255) / 256 * 256;
    if (e == cudaSuccess) ok(cudaMalloc(&c->ws, ws), "workspace");
    if (e == cudaSuccess) ok(cudaMemsetAsync(c->ws, 0, ws, c->stream), "workspace");
    if (e == cudaSuccess) {
        uint8_t *p = (uint8_t *)c->ws;
        FwdArgs &a = c->base;
        a.x = carve<float>(p, (size_t)T * d);
        a.xh = carve<__half>(p, (size_t)T * d);
        a.xh_lo = carve<__half>(p, (size_t)T * d);
        a.q = carve<float>(p, (size_t)T * H * hd);
        a.o32 = carve<float>(p, (size_t)T * H * hd);
        a.o16 = carve<__half>(p, (size_t)T * H * hd);
        a.o16_lo = carve<__half>(p, (size_t)T * H * hd);
        a.h32 = carve<float>(p, (size_t)T * Fp);
        a.h16 = carve<__half>(p, (size_t)T * Fp);
        a.h16_lo = carve<__half>(p, (size_t)T * Fp);
        a.logits = carve<float>(p, (size_t)T * V);
        a.amax_key = carve<unsigned long long>(p, (size_t)T);
        a.att_part = carve<float>(p, part_rows * G * (hd + 2));
        a.att_cnt = carve<int32_t>(p, (size_t)T * KV);
        c->amax_dev = carve<int32_t>(p, (size_t)std::max<int>(T, 4096));
        a.err = carve<int32_t>(p, 64);
        a.nonfinite = a.err + 1;
        a.tag = 1;
        if (T > kGemvMaxT) {
            a.gemm_part = carve<float>(p, kGemmPartBytes / 4);
            a.gemm_part_bytes = kGemmPartBytes;
            a.gemm_cnt = carve<int32_t>(p, kGemmMaxTiles);
        }
        a.d = d; a.H = H; a.KV = KV; a.hd = hd; a.F = hp.n_ff; a.F_pad = Fp; a.V = V; a.L = L;
        a.eps = hp.rms_eps;
        a.kc = c->kc; a.vc = c->vc; a.n_pages = c->n_pages;
        a.pt = c->pt; a.max_pages_per_seq = c->max_pages_per_seq;
        a.rope = c->rope;
        a.att_max_split = c->max_att_split;
        a.att_max_chunk = 512;
        a.att_rows_cap = (int)part_rows;
        a.pdl = true;
    }
    // metadata: per token tok, pos, seq, cell, out_row + up to 2 page-table updates (2 ints each)
    c->meta_cap = 12 * std::max<int>(T, 4096) + 64;
    if (e == cudaSuccess) ok(cudaMalloc(&c->meta_dev, (size_t)c->meta_cap * 4), "metadata");
    if (e == cudaSuccess) ok(cudaHostAlloc((void **)&c->meta_host, (size_t)2 * c->meta_cap * 4, cudaHostAllocDefault), "pinned");
    c->amax_cap = std::max<int>(T, 4096);
    if (e == cudaSuccess) ok(cudaHostAlloc((void **)&c->amax_host, (size_t)c->amax_cap * 4, cudaHostAllocDefault), "pinned");
    if (e == cudaSuccess) ok(cudaHostAlloc((void **)&c->status_host, 2 * sizeof(int32_t), cudaHostAllocDefault), "pinned");
    for (auto &ev : c->meta_ev)
        if (e == cudaSuccess) ok(cudaEventCreateWithFlags(&ev, cudaEventDisableTiming), "event");
    if (e == cudaSuccess) ok(launch_rope_table(c->rope, (int)c->n_ctx, hd, (double)hp.rope_theta, c->stream), "rope table");
    if (e == cudaSuccess) ok(cudaStreamSynchronize(c->stream), "ctx init");
    if (e != cudaSuccess) {
        free_ctx_device(c);
        delete c;
        return nullptr;
    }
    return c;
}

extern "C" void lcx_ctx_free(lcx_ctx *c) {
    if (!c) return;
    if (!c->host_only) {
        cudaStreamSynchronize(c->stream);
        free_ctx_device(c);
    }
    delete c;
}

extern "C" void lcx_kv_clear(lcx_ctx *c) {
    if (!c) return;
    init_cells(c);
}

extern "C" int32_t lcx_seq_pos_max(const lcx_ctx *c, int32_t seq) {
    if (!c || seq < 0 || (uint32_t)seq >= c->n_seq_max) return -1;
    return c->seqs[seq].len - 1;
}

extern "C" int32_t lcx_n_outputs(const lcx_ctx *c) { return c ? c->n_outputs_last : 0; }

extern "C" void lcx_set_abort(lcx_ctx *c, int (*cb)(void *), void *ud) {
    if (!c) return;
    c->abort_cb = cb;
    c->abort_ud = ud;
}

extern "C" void lcx_get_stats(const lcx_ctx *c, lcx_stats *out) {
    if (!c || !out) return;
    *out = c->st;
    out->n_cells_used = c->cells_used;
}

extern "C" int32_t lcx_kv_read(lcx_ctx *c, int32_t layer, int32_t seq, int32_t pos, uint16_t *k_out, uint16_t *v_out) {
    if (!c || c->host_only || !k_out || !v_out) return LCX_INVALID;
    if (layer < 0 || layer >= c->hp.n_layer || seq < 0 || (uint32_t)seq >= c->n_seq_max) return LCX_INVALID;
    const SeqState &S = c->seqs[seq];
    if (pos < 0 || pos >= S.len) return LCX_INVALID;
    const int KV = c->hp.n_head_kv, hd = c->hp.head_dim;
    const int page = S.pages[pos / kPage], slot = pos % kPage;
    cudaError_t e = cudaStreamSynchronize(c->stream);
    for (int h = 0; h < KV && e == cudaSuccess; ++h) {
        const size_t off = ((((size_t)layer * c->n_pages + page) * KV + h) * kPage + slot) * hd;
        e = cudaMemcpy(k_out + (size_t)h * hd, c->kc + off, (size_t)hd * 2, cudaMemcpyDeviceToHost);
        if (e == cudaSuccess) e = cudaMemcpy(v_out + (size_t)h * hd, c->vc + off, (size_t)hd * 2, cudaMemcpyDeviceToHost);
    }
    if (e != cudaSuccess) {
        set_err("kv read", e);
        return LCX_COMPUTE_FAILED;
    }
    return LCX_OK;
}

extern "C" const char *lcx_last_error(void) {
    std::lock_guard<std::mutex> lk(g_err_mu);
    return g_err.c_str();
}

// --------------------------------------------------------------------- batch rules
// Validates and fills the batch (llama_batch_allocr::init): -1 on an invalid batch.
static int32_t fill_batch(const lcx_ctx *c, const lcx_batch &b, Plan &P) {
    if (b.n_tokens <= 0 || !b.token) return LCX_INVALID;
    const int n = b.n_tokens;
    P.tok.assign(b.token, b.token + n);
    P.seq.resize(n);
    P.pos.resize(n);
    P.flag.resize(n);
    std::vector<int32_t> next(c->n_seq_max);
    for (uint32_t s = 0; s < c->n_seq_max; ++s) next[s] = c->seqs[s].len;
    for (int i = 0; i < n; ++i) {
        if (P.tok[i] < 0 || P.tok[i] >= c->hp.n_vocab) return LCX_INVALID;
        const int32_t s = b.seq_id ? b.seq_id[i] : 0;
        if (s < 0 || (uint32_t)s >= c->n_seq_max) return LCX_INVALID;
        P.seq[i] = s;
        const int32_t expect = next[s]++;
        const int32_t p = b.pos ? b.pos[i] : expect;
        if (p != expect) return LCX_INVALID;
        P.pos[i] = p;
        P.flag[i] = b.logits ? (int8_t)(b.logits[i] != 0) : (int8_t)(i == n - 1);
    }
    return LCX_OK;
}

// Reserves a cell for every token (all or nothing): 1 if the cache cannot hold the batch.
static int32_t reserve_cells(lcx_ctx *c, Plan &P) {
    const int n = (int)P.tok.size();
    if (c->kv_unified) {
        if (c->cells_used + n > (int64_t)c->n_ctx) return LCX_NO_KV_SLOT;
    } else {   // a stream per sequence: n_ctx_seq = n_ctx / n_seq_max cells each (step 10)
        const int64_t n_ctx_seq = (int64_t)c->n_ctx / c->n_seq_max;
        std::vector<int64_t> len(c->n_seq_max);
        for (uint32_t q = 0; q < c->n_seq_max; ++q) len[q] = c->seqs[q].len;
        for (int i = 0; i < n; ++i)
            if (++len[P.seq[i]] > n_ctx_seq) return LCX_NO_KV_SLOT;
    }
    P.cell.resize(n);
    P.pt_idx.clear();
    P.pt_page.clear();
    P.pt_tok.clear();
    for (int i = 0; i < n; ++i) {
        SeqState &S = c->seqs[P.seq[i]];
        const int32_t p = P.pos[i];
        if (p % kPage == 0) {
            if (c->free_pages.empty()) return LCX_NO_KV_SLOT;   // cannot happen: pages cover n_ctx + slack
            const int32_t page = c->free_pages.back();
            c->free_pages.pop_back();
            S.pages.push_back(page);
            P.pt_idx.push_back(P.seq[i] * c->max_pages_per_seq + p / kPage);
            P.pt_page.push_back(page);
            P.pt_tok.push_back(i);
        }
        P.cell[i] = S.pages[p / kPage] * kPage + p % kPage;
        S.len = p + 1;
    }
    c->cells_used += n;
    return LCX_OK;
}

// Releases the cells of the plan's tokens marked in `rel` (for each sequence a tail of its
// tokens: ubatches take every sequence's tokens in position order).
static void release_tokens(lcx_ctx *c, const Plan &P, const std::vector<char> &rel) {
    std::vector<int32_t> len(c->n_seq_max, -1);
    int cnt = 0;
    for (size_t i = 0; i < rel.size(); ++i)
        if (rel[i]) {
            const int32_t q = P.seq[i];
            if (len[q] < 0 || P.pos[i] < len[q]) len[q] = P.pos[i];
            ++cnt;
        }
    for (uint32_t q = 0; q < c->n_seq_max; ++q) {
        if (len[q] < 0) continue;
        SeqState &S = c->seqs[q];
        S.len = len[q];
        while ((int)S.pages.size() * kPage > S.len + (kPage - 1) && !S.pages.empty()) {
            c->free_pages.push_back(S.pages.back());
            S.pages.pop_back();
        }
    }
    c->cells_used -= cnt;
}

// Releases the cells of tokens [from, n) of the plan (their sequences' tails).
static void release_cells(lcx_ctx *c, const Plan &P, int from) {
    std::vector<char> rel(P.tok.size(), 0);
    for (size_t i = (size_t)from; i < rel.size(); ++i) rel[i] = 1;
    release_tokens(c, P, rel);
}

// --------------------------------------------------------------------- forward of one ubatch
namespace {

struct Ub {
    std::vector<int> idx;   // the plan's tokens in this ubatch, in ubatch order
    int T = 0, n_out = 0;   // tokens and output rows
    int row0 = 0;           // batch-order output row of its first flagged token
    bool contig = true;     // its flagged tokens' batch rows are row0, row0 + 1, ... in ubatch order
    std::vector<int> rows;  // batch-order output row of each flagged token, in ubatch order
};

bool is_device_ptr(const void *p) {
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged;
}

// Writes the ubatch's metadata into pinned staging and queues its upload. Returns the
// device UbDev view.
cudaError_t upload_meta(lcx_ctx *c, const Plan &P, const Ub &u, UbDev &ub) {
    const int T = u.T;
    const std::vector<int> &x = u.idx;
    // updates whose first token lies in this ubatch
    std::vector<char> mine(P.tok.size(), 0);
    for (int i : x) mine[i] = 1;
    std::vector<int> upd;
    for (size_t k = 0; k < P.pt_tok.size(); ++k)
        if (mine[P.pt_tok[k]]) upd.push_back((int)k);
    // query tiles: runs of consecutive positions of one sequence, cut every 64 tokens
    std::vector<int32_t> tiles;
    for (int i = 0; i < T;) {
        int n = 1;
        while (i + n < T && n < 64 && P.seq[x[i + n]] == P.seq[x[i]] && P.pos[x[i + n]] == P.pos[x[i]] + n) ++n;
        tiles.insert(tiles.end(), {i, n, P.seq[x[i]], P.pos[x[i]]});
        i += n;
    }
    const int ntiles = (int)tiles.size() / 4;
    const int tiles_off = (5 * T + 2 * (int)upd.size() + 3) / 4 * 4;   // int4-aligned
    const int need = tiles_off + 4 * ntiles;
    if (need > c->meta_cap) return cudaErrorInvalidValue;
    const int slot = c->meta_slot;
    c->meta_slot ^= 1;
    cudaError_t e = cudaEventSynchronize(c->meta_ev[slot]);
    if (e != cudaSuccess) return e;
    int32_t *h = c->meta_host + (size_t)slot * c->meta_cap;
    int32_t *tok = h, *pos = h + T, *seq = h + 2 * T, *cell = h + 3 * T, *orow = h + 4 * T, *pu = h + 5 * T;
    int no = 0;
    for (int i = 0; i < T; ++i) {
        tok[i] = P.tok[x[i]];
        pos[i] = P.pos[x[i]];
        seq[i] = P.seq[x[i]];
        cell[i] = P.cell[x[i]];
        if (P.flag[x[i]]) orow[no++] = i;
    }
    for (size_t k = 0; k < upd.size(); ++k) {
        pu[2 * k] = P.pt_idx[upd[k]];
        pu[2 * k + 1] = P.pt_page[upd[k]];
    }
    std::memcpy(h + tiles_off, tiles.data(), tiles.size() * 4);
    e = cudaMemcpyAsync(c->meta_dev, h, (size_t)need * 4, cudaMemcpyHostToDevice, c->stream);
    if (e == cudaSuccess) e = cudaEventRecord(c->meta_ev[slot], c->stream);
    int32_t *d = c->meta_dev;
    ub.tok = d;
    ub.pos = d + T;
    ub.seq = d + 2 * T;
    ub.cell = d + 3 * T;
    ub.out_rows = d + 4 * T;
    ub.pt_upd = d + 5 * T;
    ub.n_upd = (int)upd.size();
    ub.qtiles = reinterpret_cast<const int4 *>(d + tiles_off);
    ub.n_qtiles = ntiles;
    return e;
}

enum { PC_GEMV = 0, PC_GEMM = 1, PC_ATTN = 2, PC_OTHER = 3 };

// The tensor-core (tcgen05) prefill attention wherever its shape fits (4 query heads per KV head,
// head_dim 64 or 128): measured faster than the mma.sync kernel at every length of the named
// workloads (1B shape, 512-token prompt: 19 vs 27 us a layer; 8B shape, ubatches of 512 up to
// position 2048: 4.9 vs 9.4 ms for the prompt; 32768-token prompt: 0.61 vs 1.35 s).
// LCX_ATTN_MMA_SYNC=1 selects the mma.sync kernel everywhere (same results up to summation order),
// for cross-checking the two on a device.
static bool attention_prefill_tc(const FwdArgs &a) {
    static const bool mma_sync = [] {
        const char *e = getenv("LCX_ATTN_MMA_SYNC");
        return e && e[0] == '1';
    }();
    return !mma_sync && attention_prefill_tc_fits(a);
}

// Brackets one launch with events when profiling is on; in trace mode gives the launch a slot of
// the in-kernel timeline instead.
struct ProfScope {
    lcx_ctx *c;
    int cls;
    double bytes, flops;
    ProfScope(lcx_ctx *c_, int cls_, double bytes_, double flops_, FwdArgs *a = nullptr)
        : c(c_), cls(cls_), bytes(bytes_), flops(flops_) {
        if (a) {
            a->trace = nullptr;
            if (c->trace && c->trace_used < c->trace_cap) {
                a->trace = c->trace;
                a->trace_slot = c->trace_used++;
            }
        }
        if (!c->prof_on) return;
        if (c->prof_rec.size() * 2 + 2 > c->prof_ev.size()) prof_resolve(c);
        cudaEventRecord(c->prof_ev[c->prof_rec.size() * 2], c->stream);
    }
    ~ProfScope() {
        if (!c->prof_on) return;
        cudaEventRecord(c->prof_ev[c->prof_rec.size() * 2 + 1], c->stream);
        c->prof_rec.push_back({cls, bytes, flops});
    }
};

// algorithmic bytes of a weight matrix as stored: its logical rows and stored blocks
double qmat_bytes(const QMat &W, int rows, int k_logical) {
    return (double)rows * ((k_logical + 31) / 32) * (W.type == Q4 ? 18.0 : 34.0);
}

cudaError_t run_forward(lcx_ctx *c, FwdArgs &a, int max_natt, double att_cells, int32_t *amax_dst) {
    lcx_model *m = c->m;
    const lcx_hparams &hp = m->hp;
    cudaStream_t s = c->stream;
    int64_t &nl = c->st.n_kernels;
    int64_t *wide = &c->st.n_gemm_wide;
    const double T = a.T, d = a.d, qw = (double)a.H * a.hd, kvw = (double)a.KV * a.hd, F = a.F;
    cudaError_t e;
    // a one-token ubatch runs as one persistent launch where the step kernel applies
    if (a.T == 1 && a.n_out <= 1) {
        if (!c->step.tried) {
            e = decode_step_prepare(c->step, m->layers.data(), hp.n_layer, m->head, m->output_norm, c->base);
            if (e != cudaSuccess) return e;
        }
        if (c->step.ok) {
            const double kvw = (double)a.KV * a.hd;
            const double bytes = c->step.weight_bytes + (a.n_out ? c->step.head_bytes : 0.0) +
                                 att_cells * kvw * 2 * 2 * hp.n_layer;
            const double flops = 2.0 * (c->step.weight_bytes + (a.n_out ? c->step.head_bytes : 0.0)) * 32.0 /
                                     (m->layers[0].qkv.type == Q4 ? 18.0 : 34.0) +
                                 att_cells * 4.0 * a.H * a.hd * hp.n_layer;
            a.trace = nullptr;
            const int n_slots = 5 * hp.n_layer + 2;
            if (c->trace && c->trace_used + n_slots <= c->trace_cap) {
                a.trace = c->trace;
                a.trace_slot = c->trace_used;
                c->trace_used += n_slots;
            }
            ProfScope ps(c, PC_GEMV, bytes, flops);
            return launch_decode_step(c->step, a, m->tok_embd, hp.t_embd, amax_dst, max_natt, s, nl);
        }
    }
    {
        ProfScope ps(c, PC_OTHER, T * (d * (hp.t_embd == LCX_F16 ? 2.0 : 34.0 / 32.0) + d * 4), 0);
        e = launch_embed(a, hp.t_embd, m->tok_embd, s, nl);
    }
    if (e != cudaSuccess) return e;
    const DevLayer &L0 = m->layers[0];
    const bool gemv = gemv_fits(L0.qkv, a.T) && gemv_fits(L0.wo, a.T) && gemv_fits(L0.gateup, a.T) &&
                      gemv_fits(L0.down, a.T);
    const int cls = gemv ? PC_GEMV : PC_GEMM;
    const double ab = gemv ? 4.0 : 2.0;   // activation bytes per element read by the matmul
    const double w_qkv = qmat_bytes(L0.qkv, (int)(qw + 2 * kvw), a.d), w_o = qmat_bytes(L0.wo, a.d, (int)qw);
    const double w_gu = qmat_bytes(L0.gateup, 2 * a.F, a.d), w_dn = qmat_bytes(L0.down, a.d, a.F);
    const double att_bytes = att_cells * kvw * 2 * 2 + T * qw * (4 + ab);
    const double att_flops = att_cells * 4.0 * qw;
    for (int l = 0; l < hp.n_layer && e == cudaSuccess; ++l) {
        const DevLayer &D = m->layers[l];
        if (!gemv) {
            ProfScope ps(c, PC_OTHER, T * d * 6, 0);
            e = launch_rmsnorm_h(a.x, nullptr, a.T, a.d, D.attn_norm, a.eps, a.xh, a.xh_lo, s, nl);
        }
        if (e == cudaSuccess) {
            ProfScope ps(c, cls, w_qkv + T * d * ab + T * (qw * 4 + kvw * 4), 2 * T * (qw + 2 * kvw) * d, &a);
            e = gemv ? launch_gemv(D.qkv, EPI_QKV, a.T, GemvIn{a.x, nullptr, D.attn_norm}, a, l, s, nl)
                     : launch_gemm(D.qkv, EPI_QKV, a.T, a.xh, a.xh_lo, a, l, s, nl, wide);
        }
        if (e == cudaSuccess) {
            ProfScope ps(c, PC_ATTN, att_bytes, att_flops, &a);
            // long runs of one sequence (prefill): tensor-core tiles; single tokens: split-K
            const bool tiles = !gemv && a.ub.n_qtiles > 0 && a.ub.n_qtiles * 8 <= a.T;
            e = !tiles ? launch_attention(a, l, max_natt, !gemv, s, nl)
                : attention_prefill_tc(a) ? launch_attention_prefill_tc(a, l, s, nl)
                                          : launch_attention_prefill(a, l, s, nl);
        }
        if (e == cudaSuccess) {
            ProfScope ps(c, cls, w_o + T * qw * ab + T * d * 8, 2 * T * d * qw, &a);
            e = gemv ? launch_gemv(D.wo, EPI_RESID, a.T, GemvIn{a.o32, nullptr, nullptr}, a, l, s, nl)
                     : launch_gemm(D.wo, EPI_RESID, a.T, a.o16, a.o16_lo, a, l, s, nl, wide);
        }
        if (e == cudaSuccess && !gemv) {
            ProfScope ps(c, PC_OTHER, T * d * 6, 0);
            e = launch_rmsnorm_h(a.x, nullptr, a.T, a.d, D.ffn_norm, a.eps, a.xh, a.xh_lo, s, nl);
        }
        if (e == cudaSuccess) {
            ProfScope ps(c, cls, w_gu + T * d * ab + T * F * ab, 2 * T * 2 * F * d, &a);
            e = gemv ? launch_gemv(D.gateup, EPI_SWIGLU, a.T, GemvIn{a.x, nullptr, D.ffn_norm}, a, l, s, nl)
                     : launch_gemm(D.gateup, EPI_SWIGLU, a.T, a.xh, a.xh_lo, a, l, s, nl, wide);
        }
        if (e == cudaSuccess) {
            ProfScope ps(c, cls, w_dn + T * F * ab + T * d * 8, 2 * T * d * F, &a);
            e = gemv ? launch_gemv(D.down, EPI_RESID, a.T, GemvIn{a.h32, nullptr, nullptr}, a, l, s, nl)
                     : launch_gemm(D.down, EPI_RESID, a.T, a.h16, a.h16_lo, a, l, s, nl, wide);
        }
    }
    if (e != cudaSuccess || a.n_out == 0) return e;
    const double no = a.n_out, w_head = qmat_bytes(m->head, a.V, a.d);
    if (gemv_fits(m->head, a.n_out)) {
        ProfScope ps(c, PC_GEMV, w_head + no * d * 4 + no * a.V * 4, 2 * no * a.V * d, &a);
        e = launch_gemv(m->head, EPI_LOGITS, a.n_out, GemvIn{a.x, a.ub.out_rows, m->output_norm}, a, -1, s, nl);
    } else {
        {
            ProfScope ps(c, PC_OTHER, no * d * 6, 0);
            e = launch_rmsnorm_h(a.x, a.ub.out_rows, a.n_out, a.d, m->output_norm, a.eps, a.xh, a.xh_lo, s, nl);
        }
        if (e == cudaSuccess) {
            // the logits GEMM reads the gathered rows as its tokens
            ProfScope ps(c, PC_GEMM, w_head + no * d * 2 + no * a.V * 4, 2 * no * a.V * d);
            e = launch_gemm(m->head, EPI_LOGITS, a.n_out, a.xh, a.xh_lo, a, -1, s, nl, wide);
        }
    }
    if (e == cudaSuccess) {
        ProfScope ps(c, PC_OTHER, no * 12, 0);
        e = launch_argmax_final(a, amax_dst, s, nl);
    }
    return e;
}

}  // namespace

// Queues the copy of the device status words (after `extra`, if any, a queued copy) and
// synchronizes the stream. Returns the first failing tag of the call: 0 when every ubatch (or step)
// succeeded, the tag of the first whose logits were not all finite, or -1 when a kernel's bounded
// wait timed out (which ubatch is unknown) or the stream failed. Clears the words it found set.
static int32_t read_status(lcx_ctx *c) {
    cudaError_t e = cudaMemcpyAsync(c->status_host, c->base.err, 2 * sizeof(int32_t), cudaMemcpyDeviceToHost, c->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(c->stream);
    if (e != cudaSuccess) {
        set_err("decode", e);
        return -1;
    }
    const int32_t timed_out = c->status_host[0], nf = c->status_host[1];
    if (!timed_out && !nf) return 0;
    cudaMemsetAsync(c->base.err, 0, 2 * sizeof(int32_t), c->stream);
    if (timed_out) decode_step_reset(c->step, c->base, c->stream);   // counters a stopped step may have left
    cudaStreamSynchronize(c->stream);
    if (timed_out) {
        set_error_text("a kernel's bounded wait timed out");
        return -1;
    }
    set_error_text("a logits row holds a value that is not finite");
    return nf;
}

// The ubatches of a validated batch (step 12, init_batch): with one cell store, consecutive chunks
// of n_ubatch tokens (split_simple); with a stream per sequence, split_equal: each ubatch takes the
// same number of next tokens from every sequence that has tokens left (the lowest sequence ids
// first, at most n_ubatch sequences) -- as many as the shortest of them has left and at most
// n_ubatch divided by their number -- sequence by sequence in position order. Output rows stay in
// batch order: row of a flagged token = flagged tokens before it in the batch.
static std::vector<Ub> split_batch(const lcx_ctx *c, const Plan &P) {
    const int n = (int)P.tok.size();
    std::vector<int> brow(n, -1);
    int n_rows = 0;
    for (int i = 0; i < n; ++i)
        if (P.flag[i]) brow[i] = n_rows++;
    std::vector<Ub> ubs;
    if (c->kv_unified) {
        for (int i0 = 0; i0 < n; i0 += (int)c->n_ubatch) {
            Ub u;
            for (int i = i0; i < n && i < i0 + (int)c->n_ubatch; ++i) u.idx.push_back(i);
            ubs.push_back(std::move(u));
        }
    } else {
        std::vector<std::vector<int>> left(c->n_seq_max);
        for (int i = 0; i < n; ++i) left[P.seq[i]].push_back(i);
        std::vector<size_t> taken(c->n_seq_max, 0);
        for (;;) {
            std::vector<uint32_t> ss;
            for (uint32_t q = 0; q < c->n_seq_max && ss.size() < c->n_ubatch; ++q)
                if (taken[q] < left[q].size()) ss.push_back(q);
            if (ss.empty()) break;
            size_t k = c->n_ubatch / ss.size();
            for (uint32_t q : ss) k = std::min(k, left[q].size() - taken[q]);
            Ub u;
            for (uint32_t q : ss)
                for (size_t j = 0; j < k; ++j) u.idx.push_back(left[q][taken[q] + j]);
            for (uint32_t q : ss) taken[q] += k;
            ubs.push_back(std::move(u));
        }
    }
    for (Ub &u : ubs) {
        u.T = (int)u.idx.size();
        for (int i : u.idx)
            if (P.flag[i]) u.rows.push_back(brow[i]);
        u.n_out = (int)u.rows.size();
        u.row0 = u.n_out ? u.rows[0] : 0;
        for (int j = 0; j < u.n_out; ++j) u.contig = u.contig && u.rows[j] == u.row0 + j;
    }
    return ubs;
}

// Releases the cells of ubatch k and of every later one.
static void release_ubatches(lcx_ctx *c, const Plan &P, const std::vector<Ub> &ubs, size_t k) {
    std::vector<char> rel(P.tok.size(), 0);
    for (size_t j = k; j < ubs.size(); ++j)
        for (int i : ubs[j].idx) rel[i] = 1;
    release_tokens(c, P, rel);
}

// Rows kept after the batch stopped before ubatch k: with one store the ubatches ran in batch order,
// so the rows before k's are the batch's first rows; with a stream per sequence they are not a
// prefix of the batch's rows, and none is reported.
static int rows_kept(const lcx_ctx *c, const std::vector<Ub> &ubs, size_t k) {
    return c->kv_unified ? ubs[k].row0 : 0;
}

// Copies rows [0, n) of a ubatch's outputs (scratch) to their batch-order rows, one copy per run
// of consecutive rows: `w` elements of `esz` bytes per row.
static cudaError_t scatter_rows(const Ub &u, const void *src, void *dst, size_t w, size_t esz, cudaMemcpyKind kind,
                                cudaStream_t s) {
    cudaError_t e = cudaSuccess;
    for (int j = 0; j < u.n_out && e == cudaSuccess;) {
        int r = 1;
        while (j + r < u.n_out && u.rows[j + r] == u.rows[j] + r) ++r;
        e = cudaMemcpyAsync((uint8_t *)dst + (size_t)u.rows[j] * w * esz, (const uint8_t *)src + (size_t)j * w * esz,
                            (size_t)r * w * esz, kind, s);
        j += r;
    }
    return e;
}

extern "C" int32_t lcx_decode(lcx_ctx *c, lcx_batch batch, float *logits_out, int32_t *argmax_out) {
    if (!c) return LCX_INVALID;
    c->n_outputs_last = 0;
    Plan P;
    int32_t rc = fill_batch(c, batch, P);
    if (rc != LCX_OK) return rc;
    if (c->host_only && logits_out) return LCX_INVALID;
    rc = reserve_cells(c, P);
    if (rc != LCX_OK) return rc;
    std::vector<Ub> ubs = split_batch(c, P);
    int n_out_total = 0;
    for (const Ub &u : ubs) n_out_total += u.n_out;
    const bool amax_dev = argmax_out && !c->host_only && is_device_ptr(argmax_out);
    const bool host_am = argmax_out && !amax_dev && !c->host_only;
    if (host_am && n_out_total > c->amax_cap) {
        int32_t *nh = nullptr;
        if (cudaHostAlloc((void **)&nh, (size_t)n_out_total * 4, cudaHostAllocDefault) != cudaSuccess) {
            release_cells(c, P, 0);
            return LCX_ALLOC_FAILED;
        }
        cudaFreeHost(c->amax_host);
        c->amax_host = nh;
        c->amax_cap = n_out_total;
    }
    auto stop = [&](size_t k, int32_t code) {
        release_ubatches(c, P, ubs, k);
        c->st.n_decode++;
        c->st.n_ubatch_last = (int32_t)k;
        c->st.n_outputs_last = rows_kept(c, ubs, k);
        c->n_outputs_last = c->st.n_outputs_last;
        return code;
    };
    int done = 0;
    for (size_t k = 0; k < ubs.size(); ++k) {
        const Ub &u = ubs[k];
        if (k > 0 && c->abort_cb && c->abort_cb(c->abort_ud)) return stop(k, LCX_ABORTED);
        if (c->host_only && (int)k == c->fail_ubatch) {   // as a failed launch below
            c->fail_ubatch = -1;
            return stop(k, LCX_COMPUTE_FAILED);
        }
        if (!c->host_only) {
            FwdArgs a = c->base;
            a.T = u.T;
            a.n_out = u.n_out;
            a.tag = (int32_t)k + 1;
            cudaError_t e = upload_meta(c, P, u, a.ub);
            a.tok_src = a.ub.tok;
            // rows in batch order: written in place when they are consecutive, else through the
            // context's scratch and copied to their rows
            const bool direct = u.contig;
            if (logits_out && direct) a.logits = logits_out + (size_t)u.row0 * c->hp.n_vocab;
            int max_natt = 0;
            double cells = 0;
            for (int i : u.idx) {
                max_natt = std::max(max_natt, P.pos[i] + 1);
                cells += P.pos[i] + 1;
            }
            int32_t *dst = amax_dev && direct ? argmax_out + u.row0 : c->amax_dev;
            if (e == cudaSuccess) e = run_forward(c, a, max_natt, cells, dst);
            if (e == cudaSuccess && u.n_out > 0) {
                if (logits_out && !direct)
                    e = scatter_rows(u, c->base.logits, logits_out, c->hp.n_vocab, 4, cudaMemcpyDeviceToDevice, c->stream);
                if (e == cudaSuccess && amax_dev && !direct)
                    e = scatter_rows(u, c->amax_dev, argmax_out, 1, 4, cudaMemcpyDeviceToDevice, c->stream);
                if (e == cudaSuccess && host_am)
                    e = scatter_rows(u, c->amax_dev, c->amax_host, 1, 4, cudaMemcpyDeviceToHost, c->stream);
            }
            if (e != cudaSuccess) {
                set_err("decode", e);
                return stop(k, LCX_COMPUTE_FAILED);
            }
        }
        c->st.n_ubatch++;
        done = (int)k + 1;
    }
    if (!c->host_only && n_out_total > 0) {
        // one synchronization: the argmax rows (host buffer) and the status words. A logit that is
        // not finite fails its ubatch: its cells and those of the later ubatches are released, the
        // rows of the earlier ubatches stay (step 12: they were copied out before it ran)
        const int32_t bad = read_status(c);
        if (bad != 0) {
            const size_t k = bad > 0 && bad <= (int)ubs.size() ? (size_t)(bad - 1) : 0;
            if (host_am) std::memcpy(argmax_out, c->amax_host, (size_t)rows_kept(c, ubs, k) * 4);
            return stop(k, LCX_COMPUTE_FAILED);
        }
        if (host_am) std::memcpy(argmax_out, c->amax_host, (size_t)n_out_total * 4);
    }
    c->st.n_decode++;
    c->st.n_ubatch_last = done;
    c->st.n_outputs_last = n_out_total;
    c->n_outputs_last = n_out_total;
    return LCX_OK;
}

extern "C" int32_t lcx_ctx_set_kv_unified(lcx_ctx *c, int32_t unified) {
    if (!c || c->cells_used != 0) return LCX_INVALID;
    c->kv_unified = unified != 0;
    return LCX_OK;
}

extern "C" int32_t lcx_decode_greedy(lcx_ctx *c, int32_t seq, int32_t token, int32_t n_steps, int32_t *tokens_out) {
    if (!c || n_steps <= 0 || seq < 0 || (uint32_t)seq >= c->n_seq_max) return LCX_INVALID;
    if (token < 0 || token >= c->hp.n_vocab) return LCX_INVALID;
    if (c->host_only) return LCX_INVALID;
    // plan all steps at once: one token each, positions continuing the sequence
    Plan P;
    P.tok.assign(n_steps, token);
    P.seq.assign(n_steps, seq);
    P.pos.resize(n_steps);
    P.flag.assign(n_steps, 1);
    for (int i = 0; i < n_steps; ++i) P.pos[i] = c->seqs[seq].len + i;
    int32_t rc = reserve_cells(c, P);
    if (rc != LCX_OK) return rc;
    const bool out_dev = tokens_out && is_device_ptr(tokens_out);
    const int cap = std::max<int>((int)c->n_ubatch, 4096);
    cudaError_t e = cudaSuccess;
    // steps run in chunks of at most `cap`, metadata uploaded once per chunk
    for (int c0 = 0; c0 < n_steps && e == cudaSuccess; c0 += cap) {
        const int ns = std::min(cap, n_steps - c0);
        std::vector<int> upd;
        for (size_t k = 0; k < P.pt_tok.size(); ++k)
            if (P.pt_tok[k] >= c0 && P.pt_tok[k] < c0 + ns) upd.push_back((int)k);
        const int need = 3 * ns + 2 + 2 * (int)upd.size();
        if (need > c->meta_cap) { e = cudaErrorInvalidValue; break; }
        const int slot = c->meta_slot;
        c->meta_slot ^= 1;
        e = cudaEventSynchronize(c->meta_ev[slot]);
        if (e != cudaSuccess) break;
        int32_t *h = c->meta_host + (size_t)slot * c->meta_cap;
        int32_t *pos = h, *sq = h + ns, *cell = h + 2 * ns, *tok0 = h + 3 * ns, *zero = h + 3 * ns + 1,
                *pu = h + 3 * ns + 2;
        for (int i = 0; i < ns; ++i) {
            pos[i] = P.pos[c0 + i];
            sq[i] = seq;
            cell[i] = P.cell[c0 + i];
        }
        tok0[0] = token;
        zero[0] = 0;   // out_rows of a 1-token ubatch: row 0
        for (size_t k = 0; k < upd.size(); ++k) {
            pu[2 * k] = P.pt_idx[upd[k]];
            pu[2 * k + 1] = P.pt_page[upd[k]];
        }
        e = cudaMemcpyAsync(c->meta_dev, h, (size_t)need * 4, cudaMemcpyHostToDevice, c->stream);
        if (e == cudaSuccess) e = cudaEventRecord(c->meta_ev[slot], c->stream);
        const int32_t *d = c->meta_dev;
        for (int i = 0; i < ns && e == cudaSuccess; ++i) {
            const int step = c0 + i;
            FwdArgs a = c->base;
            a.T = 1;
            a.n_out = 1;
            a.tag = step + 1;
            a.ub.pos = d + i;
            a.ub.seq = d + ns + i;
            a.ub.cell = d + 2 * ns + i;
            a.ub.tok = d + 3 * ns;
            a.ub.out_rows = d + 3 * ns + 1;   // a zero
            a.ub.pt_upd = d + 3 * ns + 2;
            a.ub.n_upd = i == 0 ? (int)upd.size() : 0;
            // step 0 of the call reads `token`; later steps read the previous step's argmax
            a.tok_src = step == 0 ? d + 3 * ns : (i == 0 ? c->amax_dev + cap - 1 : c->amax_dev + i - 1);
            e = run_forward(c, a, P.pos[step] + 1, P.pos[step] + 1.0, c->amax_dev + i);
        }
        if (e == cudaSuccess && tokens_out) {
            if (out_dev)
                e = cudaMemcpyAsync(tokens_out + c0, c->amax_dev, (size_t)ns * 4, cudaMemcpyDeviceToDevice, c->stream);
            else
                e = cudaMemcpyAsync(c->amax_host, c->amax_dev, (size_t)ns * 4, cudaMemcpyDeviceToHost, c->stream);
        }
        if (e == cudaSuccess) {
            // the chunk's status: a step whose logits are not all finite fails it and every later
            // step (their cells are released); the earlier steps stay
            const int32_t bad = read_status(c);
            const int first_bad = bad > 0 && bad - 1 >= c0 && bad - 1 < c0 + ns ? bad - 1 : bad != 0 ? c0 : -1;
            if (tokens_out && !out_dev)
                std::memcpy(tokens_out + c0, c->amax_host, (size_t)((first_bad >= 0 ? first_bad : c0 + ns) - c0) * 4);
            if (first_bad >= 0) {
                release_cells(c, P, first_bad);
                c->st.n_decode++;
                c->st.n_ubatch += first_bad;
                c->st.n_ubatch_last = first_bad;
                c->st.n_outputs_last = first_bad;
                c->n_outputs_last = first_bad;
                return LCX_COMPUTE_FAILED;
            }
        }
        if (e == cudaSuccess && c0 + ns < n_steps) {
            // the next chunk's first step reads slot cap-1
            e = cudaMemcpyAsync(c->amax_dev + cap - 1, c->amax_dev + ns - 1, 4, cudaMemcpyDeviceToDevice, c->stream);
        }
    }
    if (e != cudaSuccess) {
        set_err("greedy decode", e);
        release_cells(c, P, 0);
        return LCX_COMPUTE_FAILED;
    }
    c->st.n_decode++;
    c->st.n_ubatch += n_steps;
    c->st.n_ubatch_last = n_steps;
    c->st.n_outputs_last = n_steps;
    c->n_outputs_last = n_steps;
    return LCX_OK;
}

static void prof_resolve(lcx_ctx *c) {
    if (c->prof_rec.empty()) return;
    cudaStreamSynchronize(c->stream);
    for (size_t i = 0; i < c->prof_rec.size(); ++i) {
        float ms = 0.f;
        cudaEventElapsedTime(&ms, c->prof_ev[2 * i], c->prof_ev[2 * i + 1]);
        lcx_kernel_profile *k = c->prof_rec[i].cls == PC_GEMV ? &c->prof.gemv
                              : c->prof_rec[i].cls == PC_GEMM ? &c->prof.gemm
                              : c->prof_rec[i].cls == PC_ATTN ? &c->prof.attention : &c->prof.other;
        k->launches++;
        k->ms += ms;
        k->bytes += c->prof_rec[i].bytes;
        k->flops += c->prof_rec[i].flops;
    }
    c->prof_rec.clear();
}

extern "C" int32_t lcx_set_profiling(lcx_ctx *c, int32_t on) {
    if (!c || c->host_only) return LCX_INVALID;
    prof_resolve(c);
    c->prof = lcx_profile{};
    if (on == 2) {
        c->prof_on = false;
        return trace_on(c);
    }
    if (c->trace) {   // leaving trace mode
        cudaStreamSynchronize(c->stream);
        cudaFree(c->trace);
        c->trace = nullptr;
    }
    c->prof_on = on != 0;
    if (c->prof_on && c->prof_ev.empty()) {
        c->prof_ev.resize(2 * 4096);
        for (auto &e : c->prof_ev)
            if (cudaEventCreate(&e) != cudaSuccess) return LCX_ALLOC_FAILED;
    }
    return LCX_OK;
}

// mode 2: record the in-kernel timeline of the next launches (up to 8192) instead of events
static int32_t trace_on(lcx_ctx *c) {
    if (!c->trace) {
        c->trace_cap = 8192;
        if (cudaMalloc(&c->trace, (size_t)c->trace_cap * 4 * 8) != cudaSuccess) return LCX_ALLOC_FAILED;
    }
    std::vector<unsigned long long> init((size_t)c->trace_cap * 4);
    for (size_t i = 0; i < init.size(); ++i) init[i] = i % 4 >= 2 ? 0ull : ~0ull;
    cudaMemcpy(c->trace, init.data(), init.size() * 8, cudaMemcpyHostToDevice);
    c->trace_used = 0;
    return LCX_OK;
}

extern "C" int32_t lcx_get_trace(lcx_ctx *c, unsigned long long *out, int32_t max_slots) {
    if (!c || c->host_only || !c->trace) return -1;
    cudaStreamSynchronize(c->stream);
    const int n = std::min(max_slots, c->trace_used);
    if (out && n > 0) cudaMemcpy(out, c->trace, (size_t)n * 4 * 8, cudaMemcpyDeviceToHost);
    return c->trace_used;
}

extern "C" int32_t lcx_get_profile(lcx_ctx *c, lcx_profile *out) {
    if (!c || !out) return LCX_INVALID;
    if (!c->host_only) prof_resolve(c);
    *out = c->prof;
    return LCX_OK;
}

extern "C" int32_t lcx_get_rows(int32_t type, const void *table, int64_t n_rows, int64_t n_cols, const int32_t *ids,
                                int32_t n, float *out, void *cuda_stream) {
    if (!table || !ids || !out || n < 0 || n_rows <= 0 || n_cols <= 0) return LCX_INVALID;
    if (type != LCX_F16 && type != LCX_Q8_0 && type != LCX_Q4_0) return LCX_INVALID;
    cudaError_t e = launch_get_rows(type, table, n_cols, ids, n, out, (cudaStream_t)cuda_stream);
    if (e != cudaSuccess) {
        set_err("get_rows", e);
        return LCX_COMPUTE_FAILED;
    }
    return LCX_OK;
}
