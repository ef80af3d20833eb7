// Internal declarations shared by the lcx library's translation units (host runtime and
// kernels). Not part of the public ABI (include/lcx.h).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace lcx {

constexpr int kPage = 64;            // KV cells per page (all of one sequence)
constexpr int kRowTile = 128;        // internal row padding of every matrix (tensor-core M tile)
constexpr int kGemvMaxT = 8;         // largest ubatch the weight-streaming GEMV serves
constexpr int kGemvSmemX = 96 * 1024;   // bytes of staged activations a GEMV CTA may hold
constexpr int kGemvSmemTotal = 212 * 1024;  // dynamic shared memory of a GEMV CTA (static use < 12 KB)

enum QType { QF16 = 1, Q4 = 2, Q8 = 8 };

// A weight matrix re-laid out for the kernels: N_pad rows (a multiple of 128) of nb 32-element
// blocks (nb even), stored by row quads so that any run of consecutive quads -- quants and scales
// together -- is one contiguous range (one bulk copy per decode stage, one tensor-map box per
// prefill tile). Quad q (rows 4q..4q+3) takes quad_bytes() at q * quad_bytes(), as nb / 2 block
// pairs of pair_bytes() each; pair p (blocks 2p, 2p+1) holds
//   [row 0: block 2p quants, block 2p+1 quants] ... [row 3: ...]   (4 x 2 x QB bytes)
//   [block 2p: f16 scales of rows 0..3] [block 2p+1: scales of rows 0..3]   (16 bytes)
// with QB = 16 (Q4_0 nibbles, GGUF order kept) or 32 (Q8_0 int8). Rows >= N and blocks past the
// stored ones are zero (scale 0).
struct QMat {
    int type = 0;
    int N = 0, N_pad = 0;   // logical and padded rows
    int K = 0, nb = 0;      // padded input width (nb * 32) and blocks per row
    uint8_t *w = nullptr;   // the quad-interleaved storage
    // TMA descriptors (CUtensorMap) of the storage for the tensor-core GEMM: boxes of 64 quads
    // (two 128-row tiles) and of 32 quads (one tile)
    alignas(64) unsigned char tm_w[128] = {};
    alignas(64) unsigned char tm_w1[128] = {};
    bool tm_ready = false;
    int qb() const { return type == Q4 ? 16 : 32; }
    int pair_bytes() const { return 8 * qb() + 16; }
    size_t quad_bytes() const { return (size_t)(nb / 2) * pair_bytes(); }
    size_t bytes() const { return (size_t)(N_pad / 4) * quad_bytes(); }
};

// Byte offsets inside the quad-interleaved storage (host and device).
__host__ __device__ inline int pair_bytes_of(int qb) { return 8 * qb + 16; }
// quants of row rr (0..3) of a quad, block b, relative to the quad
__host__ __device__ inline int quad_q_off(int qb, int rr, int b) { return (b >> 1) * pair_bytes_of(qb) + rr * 2 * qb + (b & 1) * qb; }
// the 4 f16 scales (rows 0..3) of block b, relative to the quad
__host__ __device__ inline int quad_s_off(int qb, int b) { return (b >> 1) * pair_bytes_of(qb) + 8 * qb + (b & 1) * 8; }

struct DevLayer {
    const float *attn_norm, *ffn_norm;
    QMat qkv;      // rows [Wq; Wk; Wv]
    QMat wo;
    QMat gateup;   // row quads alternate: gate rows 4f..4f+3 at quad 2f, up rows 4f..4f+3 at quad 2f+1
    QMat down;     // K = F padded to 128
};

// Epilogue kinds shared by the GEMV and the GEMM.
enum Epi { EPI_QKV = 0, EPI_RESID = 1, EPI_SWIGLU = 2, EPI_LOGITS = 3 };

// Per-ubatch device metadata (one contiguous block, uploaded with one copy).
struct UbDev {
    const int32_t *tok;      // [T] token ids (or NULL: take the previous step's argmax)
    const int32_t *pos;      // [T]
    const int32_t *seq;      // [T]
    const int32_t *cell;     // [T] flat cell = page * kPage + slot
    const int32_t *out_rows; // [n_out] indices of flagged tokens within the ubatch
    const int32_t *pt_upd;   // [n_upd][2] (flat page-table index, page)
    int32_t n_upd;
    const int4 *qtiles;      // [n_qtiles] query tiles: (first token, tokens <= 64, sequence, first position)
    int32_t n_qtiles;
};

// Everything a forward launch needs (device pointers).
struct FwdArgs {
    // shape
    int d, H, KV, hd, F, F_pad, V, L;
    float eps;
    // metadata
    int T, n_out;
    UbDev ub;
    const int32_t *tok_src;      // where the embed kernel reads token ids
    // activations
    float *x;          // [T][d] residual stream
    __half *xh;        // [T][d] normed activations (GEMM path), f16 high part ...
    __half *xh_lo;     // ... and low part: x = hi + lo to about 22 bits
    float *q;          // [T][H*hd]
    float *o32;        // [T][H*hd]
    __half *o16;       // [T][H*hd] (high part)
    __half *o16_lo;    // [T][H*hd] (low part)
    float *h32;        // [T][F_pad]
    __half *h16;       // [T][F_pad] (high part)
    __half *h16_lo;    // [T][F_pad] (low part)
    float *logits;     // [n_out][V]
    unsigned long long *amax_key;  // [n_out]
    int32_t *amax_out; // [n_out] device
    // attention scratch
    float *att_part;   // partial (m, l, acc[hd]) per (token, q head, split)
    int32_t *att_cnt;  // [T][KV] arrival counters, zero between launches
    float *gemm_part;  // split-K partial sums of the tensor-core GEMM (NULL: no splits)
    size_t gemm_part_bytes;
    int32_t *gemm_cnt; // [kGemmMaxTiles] its per-tile arrival counters, zero between launches
    int att_max_split;
    int att_max_chunk; // > 0: cells per attention CTA at most (inside the forward; 0 for the stand-alone call)
    int att_rows_cap;  // > 0: partial rows the attention scratch holds (T * KV * splits at most)
    int32_t *err;      // device error word: set by a kernel whose bounded wait timed out
    int32_t *nonfinite;// 0, or the tag of the first ubatch of the call whose logits held a value
                       // that is not finite (written once, by compare-and-swap)
    int32_t tag;       // this ubatch's (or greedy step's) index in the call + 1
    unsigned long long *trace;   // NULL, or [slots][4] timestamps (first start, first past wait, last staged, last end)
    bool pdl;                    // launched inside the forward's chain of dependent launches
    int trace_slot;              // this launch's slot
    // KV cache
    __half *kc, *vc;   // [L][n_pages][KV][kPage][hd]
    int n_pages;
    int32_t *pt;       // [n_seq_max][max_pages_per_seq]
    int max_pages_per_seq;
    const float2 *rope; // [n_ctx][hd/2] (cos, sin)
};

// ---------------------------------------------------------------- launchers (kernels *.cu)
// All return cudaGetLastError() after the launch(es); `launches` counts kernels issued.
cudaError_t launch_repack(const void *src, int type, int N_src, int nb_src, QMat &dst, int row_offset,
                          int gateup, cudaStream_t s);
cudaError_t launch_rope_table(float2 *tab, int n_pos, int hd, double theta, cudaStream_t s);
cudaError_t launch_embed(const FwdArgs &a, int t_embd, const void *tok_embd, cudaStream_t s, int64_t &launches);
cudaError_t launch_get_rows(int type, const void *table, int64_t n_cols, const int32_t *ids, int n, float *out,
                            cudaStream_t s);
cudaError_t launch_rmsnorm_h(const float *x, const int32_t *rows, int T, int d, const float *g, float eps,
                             __half *out, __half *out_lo, cudaStream_t s, int64_t &launches);
cudaError_t launch_argmax_final(const FwdArgs &a, int32_t *dst, cudaStream_t s, int64_t &launches);

// y = W x for T <= kGemvMaxT tokens with the given epilogue; x rows are read from `x`
// (rows `x_rows` if not NULL), normalised with gains `g` when g != NULL.
struct GemvIn {
    const float *x;
    const int32_t *x_rows;
    const float *g;
};
cudaError_t launch_gemv(const QMat &W, Epi epi, int T, const GemvIn &in, const FwdArgs &a, int layer,
                        cudaStream_t s, int64_t &launches);
bool gemv_fits(const QMat &W, int T);

// GEMM for larger T: A = A_hi + A_lo, f16 activations [T][K] split in two parts
cudaError_t launch_gemm(const QMat &W, Epi epi, int T, const __half *A, const __half *A_lo, const FwdArgs &a,
                        int layer, cudaStream_t s, int64_t &launches, int64_t *wide = nullptr);

// tcgen05 GEMM (k_gemm_tc.cu) and the TMA descriptors of a weight matrix it needs. A launch's tile
// shape: bn tokens x mt 128-row weight tiles per CTA, K steps split over ks CTAs (partial sums in
// FwdArgs::gemm_part, at most kGemmMaxTiles output tiles per split launch).
struct GemmShape {
    int bn, mt, ks;
};
constexpr int kGemmMaxTiles = 4096;
constexpr size_t kGemmPartBytes = (size_t)32 << 20;   // split-K partial sums per context
GemmShape gemm_shape(int type, int N_pad, int T, int nk, int n_sm, size_t part_bytes, int max_tiles);
// (*wide, if given, counts the launches that took tiles of 128 or more tokens)
cudaError_t launch_gemm_tc(const QMat &W, Epi epi, int T, const __half *A, const __half *A_lo, const FwdArgs &a,
                           int layer, cudaStream_t s, int64_t &launches, int64_t *wide = nullptr);
bool make_weight_maps(QMat &W);

// attention over the cache for every token of the ubatch; writes o32 (f32) or o16
cudaError_t launch_attention(const FwdArgs &a, int layer, int max_natt, bool out_f16, cudaStream_t s,
                             int64_t &launches);
int attention_splits(const FwdArgs &a, int max_natt, int *chunk);
// tensor-core attention over the ubatch's query tiles (k_attn_prefill.cu); writes o16 / o16_lo
cudaError_t launch_attention_prefill(const FwdArgs &a, int layer, cudaStream_t s, int64_t &launches);
// the tensor-core (tcgen05) prefill attention: 4 query heads per KV head, head_dim 64 or 128
bool attention_prefill_tc_fits(const FwdArgs &a);
cudaError_t launch_attention_prefill_tc(const FwdArgs &a, int layer, cudaStream_t s, int64_t &launches);
// Scratch bytes one attention launch needs (partials, then arrival counters at
// *counter_offset); 0 when every token fits in a single split.
size_t attention_scratch_bytes(const FwdArgs &a, int max_natt, size_t *counter_offset);

// Persistent one-token decode step (k_decode_step.cu): one cooperative launch runs the whole
// forward of a 1-token ubatch. Prepared once per context; `ok` is false where it does not apply
// (block types or shapes without an instantiation, too little shared memory), and the forward
// then runs as separate launches.
struct DecodeStep {
    bool ok = false;
    bool tried = false;
    void *ph = nullptr;          // device array of the phases
    unsigned int *sync = nullptr;// 2 counters, zero between launches
    const void *kern = nullptr;
    int slot_bytes = 0, slots = 0, x_bytes = 0;
    size_t smem = 0;
    int grid = 0;
    int n_ph = 0;
    double weight_bytes = 0;     // stored weight bytes one step streams (without the head)
    double head_bytes = 0;
};
cudaError_t decode_step_prepare(DecodeStep &ds, const DevLayer *layers, int n_layer, const QMat &head,
                                const float *output_norm, const FwdArgs &a);
void decode_step_release(DecodeStep &ds);
// resets the step's counters (after a launch that reported an error)
cudaError_t decode_step_reset(const DecodeStep &ds, const FwdArgs &a, cudaStream_t s);
cudaError_t launch_decode_step(const DecodeStep &ds, const FwdArgs &a, const void *tok_embd, int t_embd,
                               int32_t *amax_dst, int n_att, cudaStream_t s, int64_t &launches);

// Sets a kernel attribute once per (kernel, device): the first launch on each device does it,
// under a lock, so several host threads and several devices are safe. value must not change
// between calls for the same kernel and attribute.
cudaError_t func_attr_once(const void *kern, cudaFuncAttribute attr, int value);
// SMs of the current device (looked up once per device).
int device_sm_count();

// Launch with programmatic dependent launch allowed: the kernel may start while the previous
// kernel on the stream finishes; it must execute griddepcontrol.wait before reading anything
// the previous kernels wrote (and before writing anything they read).
// Every kernel of the forward asks for the largest shared-memory carveout, so consecutive kernels
// never make an SM re-split its L1 and shared memory between launches.
template <typename F>
inline void prefer_max_shared(F *kern) {
    func_attr_once((const void *)kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args &&...args) {
    prefer_max_shared(kern);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace lcx

// f16 high / low split of an f32 value: hi = f16(v), lo = f16(v - hi); hi + lo carries about
// 22 significant bits of v.
__device__ __forceinline__ void store_split(__half *hi, __half *lo, size_t i, float v) {
    const __half h = __float2half_rn(v);
    hi[i] = h;
    lo[i] = __float2half_rn(v - __half2float(h));
}

__device__ __forceinline__ unsigned long long lcx_gtime() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Launch timeline for measurement (off when a.trace == NULL): thread 0 of every CTA records.
#define LCX_TRACE(a, which)                                                                     \
    do {                                                                                        \
        if ((a).trace && threadIdx.x == 0) {                                                    \
            unsigned long long *t_ = (a).trace + 4 * (a).trace_slot + (which);                  \
            if ((which) >= 2) atomicMax(t_, lcx_gtime()); else atomicMin(t_, lcx_gtime());      \
        }                                                                                       \
    } while (0)

#define LCX_PDL_WAIT() asm volatile("griddepcontrol.wait;" ::: "memory")
#define LCX_PDL_TRIGGER() asm volatile("griddepcontrol.launch_dependents;")
