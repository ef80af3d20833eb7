/*
 * lcx.h -- C ABI of the GB300 Llama ubatch forward.
 *
 * One forward pass of a Llama-architecture decoder over one ubatch (a slice of a batch of
 * tokens), in prefill (many tokens of a sequence) and decode (one new token per sequence),
 * as the article "How inference works in llama.cpp" (romankryvolapov.com, llama-cpp) walks
 * through it: token-embedding gather, then per layer RMSNorm, Q/K/V projections with
 * block-quantized weights, RoPE, KV-cache append, causal grouped-query attention over the
 * cache, output projection, RMSNorm and a SwiGLU feed-forward; then the final norm, the
 * vocabulary logits and a greedy argmax.
 *
 * Every step runs in this library's CUDA kernels on one GPU. Pointers are plain host or
 * device pointers; no call takes a framework type. All device work of a context is ordered on
 * the CUDA stream given to lcx_ctx_create.
 *
 * Threading: a model may be shared by several contexts; a context is used by one host thread
 * at a time.
 */
#ifndef LCX_H
#define LCX_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Stored element types of weight tensors (step 4, GGUF tensor types: quantized types keep
 * elements in fixed-size blocks that share one scale).
 *   LCX_F16:  IEEE binary16, 2 bytes per element.
 *   LCX_Q8_0: 34-byte blocks over 32 consecutive elements of a row: fp16 scale d (little
 *             endian), then int8 q[32]; element value d * q.
 *   LCX_Q4_0: 18-byte blocks over 32 elements: fp16 d, then 16 bytes; byte j holds element j
 *             in its low nibble and element j + 16 in its high nibble; value d * (q - 8).
 * Rows of a block-typed matrix hold ceil(K / 32) blocks; elements past K in the last block
 * are ignored (their input is zero). */
typedef enum { LCX_F16 = 1, LCX_Q4_0 = 2, LCX_Q8_0 = 8 } lcx_type;

/* Model shape (step 5, load_hparams: n_embd, n_layer, n_ff, n_head, n_head_kv (GQA),
 * rope_freq_base). head_dim is the per-head width (n_embd / n_head for these shapes).
 * rms_eps is the RMSNorm epsilon; rope_theta the RoPE frequency base (frequency scale 1,
 * no context extension). t_linear is the type of every layer matrix, t_embd of tok_embd,
 * t_out of the output head. */
typedef struct {
    int32_t n_vocab, n_embd, n_layer, n_head, n_head_kv, head_dim, n_ff;
    float rms_eps, rope_theta;
    int32_t t_linear, t_embd, t_out;
} lcx_hparams;

/* One layer's weights as DEVICE pointers (step 5, load_arch_tensors for llama).
 * Matrices are row-major [N][K] in stored form: row n holds the K inputs of output n.
 *   wq [n_head*head_dim][n_embd], wk, wv [n_head_kv*head_dim][n_embd],
 *   wo [n_embd][n_head*head_dim], w_gate, w_up [n_ff][n_embd],
 *   w_down [n_embd][n_ff] (rows of ceil(n_ff/32) blocks).
 * attn_norm, ffn_norm: float32 [n_embd] gains. */
typedef struct {
    const void *attn_norm, *wq, *wk, *wv, *wo, *ffn_norm, *w_gate, *w_up, *w_down;
} lcx_layer_w;

/* Model weights. tok_embd [n_vocab][n_embd] (t_embd), output_norm float32 [n_embd],
 * output [n_vocab][n_embd] (t_out) or NULL: tied to tok_embd, as llama.cpp does when the file
 * has no output matrix (step 5). layers: HOST array [n_layer] of device-pointer sets. */
typedef struct {
    const void *tok_embd, *output_norm, *output;
    const lcx_layer_w *layers;
} lcx_weights;

/* A batch (step 11, llama_batch): HOST arrays of n_tokens entries.
 *   token:  ids in [0, n_vocab).
 *   pos:    NULL -> each token gets its sequence's last position + 1, + 2, ... in batch order.
 *           Otherwise the positions of each sequence must continue from its last position by
 *           +1 in batch order (a new sequence starts at 0).
 *   seq_id: NULL -> every token belongs to sequence 0. One sequence per token.
 *   logits: NULL -> only the last token is an output row; otherwise nonzero flags mark the
 *           tokens whose logits are computed (step 13c, output rows). */
typedef struct {
    int32_t n_tokens;
    const int32_t *token;
    const int32_t *pos;
    const int32_t *seq_id;
    const int8_t *logits;
} lcx_batch;

typedef struct lcx_model lcx_model;
typedef struct lcx_ctx lcx_ctx;

/* Return codes (step 12, the return value of llama_decode). */
enum {
    LCX_OK = 0,
    LCX_NO_KV_SLOT = 1,      /* the cache cannot hold the whole batch; nothing was committed */
    LCX_ABORTED = 2,         /* the abort callback stopped the batch between ubatches */
    LCX_INVALID = -1,        /* invalid batch or argument */
    LCX_ALLOC_FAILED = -2,   /* device or host allocation failed */
    LCX_COMPUTE_FAILED = -3  /* a computation failed (a CUDA launch or copy, a kernel's timed-out wait, or a
                                logits row holding a value that is not finite): the failed ubatch's cells
                                and those of later ubatches are rolled back (step 12) */
};

/* Builds a model over the caller's weights. The model keeps its own device copy of every layer
 * matrix and of `output`, re-laid out for the kernels (scale planes split from the quantized
 * planes, Q/K/V and gate/up fused): the caller may free or reuse those after this call
 * returns. tok_embd, output_norm and the per-layer norm gains are BORROWED (read in place):
 * they must stay valid and unchanged until lcx_model_free.
 * Requirements: n_embd % 64 == 0, head_dim even and <= 256, (n_head * head_dim) % 64 == 0,
 * n_head % n_head_kv == 0, t_linear in {Q4_0, Q8_0}, t_out in {Q4_0, Q8_0} (t_embd when
 * output is NULL), t_embd in {F16, Q8_0, Q4_0}.
 * Returns NULL on failure with *err (if err != NULL) set to LCX_INVALID or LCX_ALLOC_FAILED.
 * The current CUDA device at this call is the model's device. */
lcx_model *lcx_model_create(const lcx_hparams *hp, const lcx_weights *w, int32_t *err);
void lcx_model_free(lcx_model *model);

/* Creates a context (step 10, llama_context): n_ctx cells of f16 K/V per layer shared by up
 * to n_seq_max sequences (n_ctx is rounded up to a multiple of 256, as the context constructor
 * does), and a workspace sized for n_ubatch tokens, reserved here so that decoding allocates
 * nothing (the worst-case graph reservation). cuda_stream is a cudaStream_t or NULL for the
 * default stream. Returns NULL on failure (invalid sizes, or allocation failure). */
lcx_ctx *lcx_ctx_create(lcx_model *model, uint32_t n_ctx, uint32_t n_seq_max, uint32_t n_ubatch,
                        void *cuda_stream);
void lcx_ctx_free(lcx_ctx *ctx);

/* Decodes a batch (step 12, llama_context::decode): validates and fills it, reserves cells
 * for all of it (or returns LCX_NO_KV_SLOT with nothing committed), cuts it into ubatches of
 * at most n_ubatch consecutive tokens and runs the forward over each in order. Tokens of the
 * same ubatch see each other causally: a token attends every cell of its sequence with
 * position <= its own, its own K/V included.
 *   logits_out: DEVICE float32 [n_out][n_vocab] or NULL; rows are the flagged tokens in
 *               batch order (step 14, the logits buffer).
 *   argmax_out: host or device int32 [n_out] or NULL: the index of each row's largest logit
 *               (lowest index on ties).
 * When the batch has output rows the call synchronizes the stream before it returns (to copy a
 * host argmax_out and to check the logits); otherwise it returns as soon as the work is queued.
 * A logits row holding a value that is not finite (NaN or infinity) fails its ubatch as a failed
 * computation does (step 12, return -3): LCX_COMPUTE_FAILED, the cells of that ubatch and of the
 * later ones released, the earlier ubatches kept in the cache with their rows (which the decode
 * loop copied out before the failed ubatch ran) -- lcx_n_outputs tells how many rows are valid.
 * Returns an LCX_* code. */
int32_t lcx_decode(lcx_ctx *ctx, lcx_batch batch, float *logits_out, int32_t *argmax_out);

/* Greedy generation on the device (the article's generation loop, step 15, with the sampler
 * replaced by argmax): decodes `token` for sequence `seq` at its next position, then n_steps-1
 * further single-token steps, each fed the argmax of the previous one without a host round
 * trip. tokens_out (host or device int32 [n_steps]) receives the argmax of every step.
 * Reserves all n_steps cells first (LCX_NO_KV_SLOT if they do not fit). Synchronizes the stream
 * before it returns. A step whose logits hold a value that is not finite fails with
 * LCX_COMPUTE_FAILED: its cell and those of the later steps are released, the earlier steps stay
 * and lcx_n_outputs gives their number (their tokens are in tokens_out). */
int32_t lcx_decode_greedy(lcx_ctx *ctx, int32_t seq, int32_t token, int32_t n_steps, int32_t *tokens_out);

/* KV layout of a context (step 10 and step 12, init_batch). unified != 0 (the default): one cell
 * store of n_ctx cells shared by all sequences, batches cut into consecutive chunks of n_ubatch
 * tokens (split_simple). unified == 0: a stream per sequence -- each sequence may hold at most
 * n_ctx_seq = n_ctx / n_seq_max cells (a batch that would exceed it returns LCX_NO_KV_SLOT with
 * nothing committed) -- and batches are cut by split_equal: each ubatch takes the same number of
 * next tokens from every sequence that has tokens left (the lowest sequence ids first, at most
 * n_ubatch sequences), as many as the shortest of them has left and at most n_ubatch divided by
 * their number, sequence by sequence in position order. Logits rows stay in batch order either
 * way. When a batch of a context with a stream per sequence stops (LCX_ABORTED or
 * LCX_COMPUTE_FAILED), its completed ubatches stay in the cache but no rows are reported (they
 * are not the batch's first rows). Only while the context holds no cell (after creation or
 * lcx_kv_clear): LCX_INVALID otherwise. */
int32_t lcx_ctx_set_kv_unified(lcx_ctx *ctx, int32_t unified);

/* Frees every cell (the memory clear of the KV-cache section): every sequence becomes empty. */
void lcx_kv_clear(lcx_ctx *ctx);

/* The last position stored for `seq`, or -1 if it has none or seq is out of range. */
int32_t lcx_seq_pos_max(const lcx_ctx *ctx, int32_t seq);

/* Output rows written by the last lcx_decode (or steps of the last lcx_decode_greedy). After a
 * call that stopped (LCX_ABORTED, LCX_COMPUTE_FAILED), the rows of the ubatches that completed
 * before it; 0 after LCX_INVALID or LCX_NO_KV_SLOT. */
int32_t lcx_n_outputs(const lcx_ctx *ctx);

/* Abort callback (step 12, abort -> 2): called on the host before every ubatch after the
 * first; a nonzero return stops the batch with LCX_ABORTED. Earlier ubatches stay in the cache;
 * the cells of the stopped and later ubatches are released. cb NULL removes it. */
void lcx_set_abort(lcx_ctx *ctx, int (*cb)(void *), void *user_data);

/* Copies the stored K and V of one cell to HOST memory: k_out, v_out receive n_head_kv *
 * head_dim f16 values each (the RoPE'd key and the value of layer `layer` at position `pos` of
 * sequence `seq`, as appended by the forward; KV-cache section: keys and values are kept per
 * layer and cell). Synchronizes the context's stream. Returns LCX_OK, or LCX_INVALID when the
 * cell does not exist. */
int32_t lcx_kv_read(lcx_ctx *ctx, int32_t layer, int32_t seq, int32_t pos, uint16_t *k_out, uint16_t *v_out);

/* Counters of a context, for tests and measurement. */
typedef struct {
    int64_t n_decode;          /* lcx_decode / lcx_decode_greedy calls that ran */
    int64_t n_ubatch;          /* ubatches run in total */
    int32_t n_ubatch_last;     /* ubatches of the last call */
    int32_t n_outputs_last;    /* output rows of the last call */
    int64_t n_kernels;         /* kernel launches issued by this context */
    int64_t n_cells_used;      /* cells currently holding K/V */
    uint32_t n_ctx;            /* cells in the cache (after rounding) */
    uint32_t n_pages;          /* KV pages allocated (page = 64 cells of one sequence) */
    int64_t n_gemm_wide;       /* tensor-core matmul launches that took 128-token tiles (large ubatches) */
} lcx_stats;
void lcx_get_stats(const lcx_ctx *ctx, lcx_stats *out);

/* Per-kernel-class timing, for measurement. With profiling on, every kernel the context
 * launches is bracketed by CUDA events on its stream and credited to a class with the
 * algorithmic bytes and flops of that launch (weight and activation bytes as stored, KV bytes
 * of the attended cells, 2 flops per multiply-add). Classes: gemv = weight-streaming matmuls
 * of small ubatches, gemm = matmuls of large ubatches, attention, other (gather, norms, argmax).
 * lcx_set_profiling(ctx, 1) clears the counters; lcx_get_profile synchronizes the stream and
 * returns the totals since then. Profiling adds event records between launches. */
typedef struct {
    int64_t launches;
    double ms, bytes, flops;
} lcx_kernel_profile;
typedef struct {
    lcx_kernel_profile gemv, gemm, attention, other;
} lcx_profile;
int32_t lcx_set_profiling(lcx_ctx *ctx, int32_t on);
int32_t lcx_get_profile(lcx_ctx *ctx, lcx_profile *out);
/* lcx_set_profiling(ctx, 2) instead records an in-kernel timeline of the next matmul-vector and
 * attention launches (up to 8192): per launch the earliest CTA start, the earliest CTA past the
 * wait for the previous kernel, the latest CTA done with its set-up (activations staged, or
 * attention partials computed), and the latest CTA end, as %globaltimer nanoseconds, with no
 * event between launches. lcx_get_trace synchronizes and copies min(max_slots, recorded) slots
 * of 4 values to host `out`; it returns the number recorded (-1 when trace mode is off). */
int32_t lcx_get_trace(lcx_ctx *ctx, unsigned long long *out, int32_t max_slots);

/* A context with no device: every host-side rule of lcx_decode (validation, position and
 * flag filling, cell reservation, ubatch split, abort, return codes) runs, and no kernel is
 * launched; logits_out must be NULL and argmax_out is left untouched. For testing the host
 * runtime on machines without a GPU. */
lcx_ctx *lcx_ctx_create_host_only(const lcx_hparams *hp, uint32_t n_ctx, uint32_t n_seq_max, uint32_t n_ubatch);

/* Host-only contexts: ubatch `ubatch` (0-based, in split order) of the next lcx_decode fails the
 * way a failed launch does -- LCX_COMPUTE_FAILED, the cells of that ubatch and of the later ones
 * released, earlier ubatches kept (step 13: the positions of a failed computation are removed
 * from the cache again) -- so the rollback can be tested without making a GPU fail. -1 cancels.
 * Returns LCX_INVALID for a context with a device. */
int32_t lcx_ctx_inject_failure(lcx_ctx *ctx, int32_t ubatch);

/* Testing aid for the prefill matmuls (the tensor-core GEMM of every ubatch of more than 8
 * tokens): every later launch, in every context of the process, takes the tile shape bn tokens x
 * mt 128-row weight tiles with its K steps split over ks CTAs, instead of the shape its cost
 * model picks -- so each compiled shape can be checked against the oracle on small models. bn
 * is 64, 128 or 256; mt is 1 or 2 (1 with bn 256); ks is 1 to 8. A launch where the forced split
 * does not fit (fewer than 4 K steps a split, or no room in the partial-sum scratch) runs with
 * ks = 1. bn = 0 restores the cost model. Results differ from the default only by summation
 * order. Returns LCX_OK, or LCX_INVALID for a shape that is not compiled. Not thread-safe
 * against decodes running at the same time. */
int32_t lcx_set_gemm_tile(int32_t bn, int32_t mt, int32_t ks);

/* Row gather with dequantisation to float32 (step 13b, ggml_get_rows on the token
 * embeddings): out[i][:] = the n_cols values of row ids[i] of `table` (stored type `type`).
 * ids and out are DEVICE pointers; runs on cuda_stream. Returns LCX_OK or LCX_INVALID /
 * LCX_COMPUTE_FAILED. */
int32_t lcx_get_rows(int32_t type, const void *table, int64_t n_rows, int64_t n_cols, const int32_t *ids, int32_t n,
                     float *out, void *cuda_stream);

/* The attention step of the forward (step 13c: scores of Q against the cached keys, causal
 * mask, softmax, weighted sum of the cached values; KV-cache section: a token attends the
 * cells of its sequence up to and including its own position) over caller-owned buffers of
 * ONE layer, with the split-K kernel lcx_decode uses.
 *   q:          DEVICE float32 [T][n_head * head_dim], RoPE already applied.
 *   k_cache,
 *   v_cache:    DEVICE f16 [n_pages][n_head_kv][64][head_dim]: page p holds 64 consecutive
 *               positions of one sequence.
 *   page_table: DEVICE int32 [n_seq][max_pages]: page ids of each sequence in position order.
 *   pos, seq:   DEVICE int32 [T]: token t attends positions 0..pos[t] of sequence seq[t].
 *   max_pos:    host upper bound of pos[] (sizes the split of the cell range).
 *   out:        DEVICE float32 [T][n_head * head_dim].
 *   workspace:  DEVICE scratch of at least lcx_attention_workspace_size(T, n_head, n_head_kv,
 *               head_dim, max_pos) bytes (may be NULL when that size is 0); it is cleared by
 *               the call as needed, and two calls sharing one workspace must not overlap.
 * head_dim 64 or 128; n_head / n_head_kv in {1, 2, 4, 8}. Stream-ordered on cuda_stream.
 * Returns LCX_OK, LCX_INVALID (bad sizes or a small workspace) or LCX_COMPUTE_FAILED. */
size_t lcx_attention_workspace_size(int32_t T, int32_t n_head, int32_t n_head_kv, int32_t head_dim, int32_t max_pos);
int32_t lcx_attention(int32_t T, int32_t n_head, int32_t n_head_kv, int32_t head_dim, const float *q,
                      const void *k_cache, const void *v_cache, int32_t n_pages, const int32_t *page_table,
                      int32_t max_pages, const int32_t *pos, const int32_t *seq, int32_t max_pos, float *out,
                      void *workspace, size_t workspace_bytes, void *cuda_stream);

/* lcx_attention for callers that cannot allocate device memory (the article has no
 * counterpart: this is an interface addition of this library). Examples of such callers: a
 * plugin whose host application owns every device allocation, a process whose device memory
 * is fully reserved by a framework's caching allocator, a latency-critical path that cannot
 * take cudaMalloc's implicit synchronisation. Same arguments and result as lcx_attention,
 * without the workspace: the scratch is a fixed device array of
 * LCX_ATTENTION_NOALLOC_SCRATCH_BYTES inside the library, present on every GPU that loads the
 * library until the process exits. The call allocates nothing.
 *   - The first call on a device looks up that array's device address (once per device, with
 *     the device current); make that first call before any stream capture. The address is kept
 *     for the life of the process: after a cudaDeviceReset of a device, do not call this entry
 *     point on that device again.
 *   - Calls whose scratch need (lcx_attention_workspace_size) exceeds the array are rejected
 *     with LCX_INVALID and a message in lcx_last_error().
 *   - Every call on a device shares the one array: calls that overlap on the GPU (on different
 *     streams, or from several host threads) race and must not be issued. */
#define LCX_ATTENTION_NOALLOC_SCRATCH_BYTES (8u * 1024u * 1024u)
int32_t lcx_attention_noalloc(int32_t T, int32_t n_head, int32_t n_head_kv, int32_t head_dim, const float *q,
                              const void *k_cache, const void *v_cache, int32_t n_pages, const int32_t *page_table,
                              int32_t max_pages, const int32_t *pos, const int32_t *seq, int32_t max_pos, float *out,
                              void *cuda_stream);

/* Parameters of the sampler chain (article, "Sampler chain", after step 14: a repeat penalty,
 * then the cut-offs top-k, top-p and min-p, then temperature, then one token is chosen).
 *   penalty_repeat: > 0; 1 = off. Each distinct history token's logit is divided by it when
 *                   positive and multiplied by it otherwise (both lower it for a value > 1).
 *   top_k:          keep the k largest logits; <= 0 or >= n_vocab = off.
 *   top_p:          keep the shortest run of candidates, largest logit first, whose softmax
 *                   probability over the candidates left by top-k reaches top_p (at least
 *                   one); >= 1 = off.
 *   min_p:          keep the candidates whose probability is >= min_p times the leader's, i.e.
 *                   logit >= max + ln(min_p); <= 0 = off.
 *   temp:           <= 0: greedy (the largest logit, lowest id on ties). Otherwise the token is
 *                   drawn from the remaining candidates with weights exp((logit - max) / temp). */
typedef struct {
    float penalty_repeat;
    int32_t top_k;
    float top_p;
    float min_p;
    float temp;
} lcx_sampler;

/* Runs the sampler chain on the device over n_rows logits rows and writes one token per row
 * (the sampler running on the backend: only the token leaves the kernel).
 *   logits:     DEVICE float32 [n_rows][n_vocab] (as lcx_decode writes them); finite values.
 *   history:    DEVICE int32 [n_rows][n_history] tokens for the repeat penalty (entries outside
 *               [0, n_vocab) are ignored), or NULL with n_history == 0.
 *   u:          DEVICE float32 [n_rows], the random numbers of the draws, in [0, 1); may be NULL
 *               when temp <= 0. The draw walks the remaining candidates in increasing token id
 *               and returns the first whose running weight exceeds u times the total weight.
 *   tokens_out: DEVICE int32 [n_rows].
 * Candidates are ordered by logit, lower token id first among equal logits. Decisions are
 * taken in float32: a token within float32 rounding of a top-p, min-p or draw boundary may
 * fall on either side of it. n_vocab <= 262144; n_rows == 0 is a no-op. Stream-ordered on cuda_stream; allocates
 * nothing. Returns LCX_OK, LCX_INVALID or LCX_COMPUTE_FAILED. */
int32_t lcx_sample(const lcx_sampler *params, const float *logits, int32_t n_rows, int32_t n_vocab,
                   const int32_t *history, int32_t n_history, const float *u, int32_t *tokens_out,
                   void *cuda_stream);

/* Last CUDA error string seen by the library in this process ("" if none). */
const char *lcx_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* LCX_H */
