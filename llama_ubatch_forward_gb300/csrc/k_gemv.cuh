// Weight-streaming GEMV for decode ubatches (T <= 8 tokens): y = W x with W in Q4_0 / Q8_0.
//
// Decode is bound by reading the weights once (KV-cache section of the article: decode loads
// memory, prefill loads the compute units), so the kernel is built to keep HBM busy with as
// few instructions per weight as possible:
//   * each warp owns a task of 4 rows and its lanes take the rows' 32-element blocks, 32 at a
//     time in an order that makes every quarter-warp's 16-byte loads hit 8 distinct bank groups
//     of the quad-interleaved layout (QMat); a row quad's 4 block scales arrive in one 8-byte load;
//   * the activations are staged once per CTA in shared memory with the RMSNorm fused in, and
//     each 32-element block of them is split into two int8 parts, x ~= s (hi + lo / 128) with
//     s = max|x| / 127 (hi = round(x / s), lo = round(128 (x / s - hi))): about 14 bits of
//     the block's range, finer than an f16 rounding of x;
//   * a block's dot product with the stored integers q is then exact integer arithmetic,
//     four elements per dp4a: P = 128 sum(q hi) + sum(q lo) (minus 8 (128 sum hi + sum lo) for
//     Q4_0's offset), and the row accumulates d * s / 128 * P in f32 -- one I2F and one FMA
//     per block instead of one float FMA per weight;
//   * row sums are reduced with warp shuffles; epilogues (RoPE + KV append, residual add,
//     SwiGLU, logits + argmax) are fused.
// The weight rows stream through a shared-memory ring filled by TMA bulk copies, one copy per
// stage: a stage is a run of consecutive row quads, contiguous in the quad-interleaved layout.
// (The copy engine's cost is per copy much more than per byte: copies of about 32 KB keep HBM
// near its peak, copies of a few KB cap a CTA far below it.)
#pragma once
#include <math_constants.h>
#include "epilogue.cuh"

namespace lcx {
namespace gemv_detail {

// ---------------------------------------------------------------- staged activations
// Per token: hi plane [nb][32 B], lo plane [nb][32 B], then meta [nb] (s / 128, C) with
// C = 8 (128 sum hi + sum lo) for Q4_0 and 0 for Q8_0. Block b sits at position xpos(b): even
// blocks first, then odd ones, matching the lanes' block order (block_of_lane); 16-byte chunk c
// of position i is stored at chunk c ^ ((i >> 2) & 1), so 8 lanes reading 8 consecutive
// positions hit 8 distinct bank groups.
__host__ __device__ constexpr size_t stage_bytes_per_token(int nb) { return (size_t)nb * 72; }

__device__ __forceinline__ int xpos(int nb, int b) { return (b & 1) * (nb >> 1) + (b >> 1); }
__device__ __forceinline__ int plane_chunk_off(int i, int c) { return i * 32 + ((c ^ ((i >> 2) & 1)) << 4); }
// block a lane takes in a run of 32 blocks starting at an even block: lanes 0-7 the even blocks
// 0, 2, .., 14, lanes 8-15 the odd blocks 1, .., 15, lanes 16-31 the same for blocks 16..31
__device__ __forceinline__ int block_of_lane(int lane) { return 2 * ((lane & 7) + 8 * (lane >> 4)) + ((lane >> 3) & 1); }

struct XQ {          // one block of one token, in registers
    int4 h0, h1;     // hi words 0..3, 4..7
    int4 l0, l1;     // lo words
    float s;         // s / 128
    int C;
};

__device__ __forceinline__ void load_xq(const uint8_t *stage_t, int nb, int b, XQ &x) {
    const uint8_t *hp = stage_t, *lp = stage_t + (size_t)nb * 32;
    const float2 *mp = reinterpret_cast<const float2 *>(stage_t + (size_t)nb * 64);
    const int i = xpos(nb, b);
    x.h0 = *reinterpret_cast<const int4 *>(hp + plane_chunk_off(i, 0));
    x.h1 = *reinterpret_cast<const int4 *>(hp + plane_chunk_off(i, 1));
    x.l0 = *reinterpret_cast<const int4 *>(lp + plane_chunk_off(i, 0));
    x.l1 = *reinterpret_cast<const int4 *>(lp + plane_chunk_off(i, 1));
    const float2 m = mp[i];
    x.s = m.x;
    x.C = __float_as_int(m.y);
}

__device__ __forceinline__ int xw(const int4 &a, const int4 &b, int i) {   // word i of the 8
    return i == 0 ? a.x : i == 1 ? a.y : i == 2 ? a.z : i == 3 ? a.w : i == 4 ? b.x : i == 5 ? b.y : i == 6 ? b.z : b.w;
}

// Integer dot of one Q4_0 block (16 bytes of nibbles) with a staged block: 128 sum(q hi) +
// sum(q lo) - C, i.e. 128 / s times sum((q - 8) x) up to the staging rounding.
__device__ __forceinline__ int q4_idot(const uint4 w, const XQ &x) {
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
    int ph = 0, pl = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int lo_n = (int)(ws[i] & 0x0F0F0F0Fu);          // elements 4i .. 4i+3
        const int hi_n = (int)((ws[i] >> 4) & 0x0F0F0F0Fu);   // elements 16+4i .. 16+4i+3
        ph = __dp4a(lo_n, xw(x.h0, x.h1, i), ph);
        ph = __dp4a(hi_n, xw(x.h0, x.h1, 4 + i), ph);
        pl = __dp4a(lo_n, xw(x.l0, x.l1, i), pl);
        pl = __dp4a(hi_n, xw(x.l0, x.l1, 4 + i), pl);
    }
    return ph * 128 + pl - x.C;
}

// Integer dot of one Q8_0 block (32 int8 in two uint4): 128 sum(q hi) + sum(q lo).
__device__ __forceinline__ int q8_idot(const uint4 w0, const uint4 w1, const XQ &x) {
    const uint32_t ws[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
    int ph = 0, pl = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        ph = __dp4a((int)ws[i], xw(x.h0, x.h1, i), ph);
        pl = __dp4a((int)ws[i], xw(x.l0, x.l1, i), pl);
    }
    return ph * 128 + pl;
}

struct GemvParams {
    const uint8_t *w;   // quad-interleaved storage (QMat)
    int N, nb, K;
    int n_tasks;
    int T;
    GemvIn in;
};

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// Stage token t: split every 32-element block of x * g (g = the RMSNorm gains, or 1) into
// hi / lo int8 parts, and leave this thread's share of sum(x^2) in red[t][warp]. The RMS factor
// is a positive scalar, so the block split does not depend on it: it multiplies each row's dot
// product in the epilogue instead, and the sum of squares is reduced while the blocks are being
// split. Two adjacent lanes share a block (16 elements each). Run by the 256 consumer threads.
// x is read through L2 only (it may have been written by other CTAs of the same launch); the
// loads of up to 4 iterations are issued together. gpre, if given, holds this thread's gains of
// the first iteration, loaded earlier by the caller (stage_gains).
constexpr int kStageThreads = 256;

__device__ __forceinline__ void stage_gains(const float *g, int nb, float4 (&gpre)[4]) {
    const int hb = threadIdx.x, b = hb >> 1, half = hb & 1;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        gpre[j] = g && hb < 2 * nb ? *reinterpret_cast<const float4 *>(g + b * 32 + half * 16 + 4 * j)
                                   : make_float4(1.f, 1.f, 1.f, 1.f);
}

template <int QT>
__device__ void stage_token(const GemvParams &p, int t, uint8_t *stage_t, float (*red)[8],
                            const float4 (*gpre)[4] = nullptr) {
    constexpr int NTHR = kStageThreads, U = 4;
    const int nb = p.nb, K = p.K;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float *xr = p.in.x + (size_t)(p.in.x_rows ? p.in.x_rows[t] : t) * K;
    uint8_t *hp = stage_t, *lp = stage_t + (size_t)nb * 32;
    float2 *mp = reinterpret_cast<float2 *>(stage_t + (size_t)nb * 64);
    float ss = 0.f;
    const int n_half = 2 * nb, iters = (n_half + NTHR - 1) / NTHR;   // same trip count in every lane
    for (int it0 = 0; it0 < iters; it0 += U) {
        float4 xv[U][4];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int hb = (it0 + u) * NTHR + threadIdx.x;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                xv[u][j] = it0 + u < iters && hb < n_half
                               ? __ldcg(reinterpret_cast<const float4 *>(xr + (hb >> 1) * 32 + (hb & 1) * 16 + 4 * j))
                               : make_float4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (it0 + u >= iters) break;   // uniform over the CTA
            const int hb = (it0 + u) * NTHR + threadIdx.x, b = hb >> 1, half = hb & 1;
            const bool active = hb < n_half;
            float v[16];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float4 q = xv[u][j];
                ss += q.x * q.x + q.y * q.y + q.z * q.z + q.w * q.w;
                if (p.in.g && active) {
                    const float4 gg = gpre && it0 + u == 0
                                          ? (*gpre)[j]
                                          : *reinterpret_cast<const float4 *>(p.in.g + b * 32 + half * 16 + 4 * j);
                    q.x *= gg.x; q.y *= gg.y; q.z *= gg.z; q.w *= gg.w;
                }
                v[4 * j] = q.x; v[4 * j + 1] = q.y; v[4 * j + 2] = q.z; v[4 * j + 3] = q.w;
            }
            float amax = 0.f;
#pragma unroll
            for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(v[j]));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));   // the partner holds the other half
            const float inv = amax > 0.f ? 127.0f / amax : 0.f;
            uint32_t hw[4], lw[4];
            int sh = 0, sl = 0;
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                uint32_t hbits = 0, lbits = 0;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float y = v[4 * w + e] * inv;
                    const float h = fminf(fmaxf(rintf(y), -127.f), 127.f);
                    const float l = fminf(fmaxf(rintf((y - h) * 128.f), -127.f), 127.f);
                    sh += (int)h;
                    sl += (int)l;
                    hbits |= ((uint32_t)(int)h & 0xffu) << (8 * e);
                    lbits |= ((uint32_t)(int)l & 0xffu) << (8 * e);
                }
                hw[w] = hbits;
                lw[w] = lbits;
            }
            sh += __shfl_xor_sync(0xffffffffu, sh, 1);
            sl += __shfl_xor_sync(0xffffffffu, sl, 1);
            if (active) {
                const int i = xpos(nb, b);
                *reinterpret_cast<uint4 *>(hp + plane_chunk_off(i, half)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                *reinterpret_cast<uint4 *>(lp + plane_chunk_off(i, half)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                if (half == 0) {
                    const int C = QT == Q4 ? 8 * (128 * sh + sl) : 0;
                    mp[i] = make_float2(amax * (1.0f / (127.0f * 128.0f)), __int_as_float(C));
                }
            }
        }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) red[t][warp] = ss;
}

// Output scale of token t from the partial sums left by stage_token: the RMS factor with norm
// gains, else 1. A non-finite sum of squares (a NaN or an infinity in x) makes it NaN: the int8
// split clamps such values to finite codes, so the scale is what carries them to the output.
__device__ __forceinline__ float finite_or_nan(float tot, float rs) { return tot < CUDART_INF_F ? rs : CUDART_NAN_F; }
__device__ __forceinline__ float token_rs(const GemvParams &p, const FwdArgs &a, float (*red)[8], int t) {
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) tot += red[t][w];
    return finite_or_nan(tot, p.in.g ? 1.0f / sqrtf(tot / (float)p.K + a.eps) : 1.f);
}

// ---------------------------------------------------------------- TMA-bulk streaming kernel
// Warp 8 (one elected lane) streams the weight rows of consecutive "stages" -- TPS tasks of 4
// rows each, contiguous in the quant and scale planes -- into a ring of S shared-memory slots
// with cp.async.bulk (mbarrier completion); it starts before the previous kernel's results
// are needed, since the weights do not depend on them. Warps 0..7 stage the activations, then
// consume the ring: warp w takes task w / KS of the stage and the w % KS-th slice of its
// blocks (KS = 8 / TPS), the slices are summed through shared memory and TPS * NT threads
// apply the epilogue. Every wait is bounded: on a timeout the kernel records an error and
// returns instead of spinning.
constexpr int kConsumerWarps = 8;
constexpr int kMaxStages = 8;
constexpr uint32_t kSpinLimit = 1u << 22;

struct StagePlan {
    int tps;            // tasks per stage (4, 2 or 1): row quads per stage
    int slots;          // ring depth
    int quad_bytes;     // bytes of one row quad (quants and scales)
    int stage_bytes;    // tps row quads, rounded to 128
    size_t x_bytes;     // staged activations
    size_t smem;        // total dynamic shared memory
};

// Stages of about 32-40 KB (one bulk copy each); a SwiGLU stage keeps at least 2 tasks (the gate
// and up halves of one feature quad). Ring depth: at most 4 slots -- deeper rings add queueing
// in front of the CTA's own loads without adding bandwidth.
__host__ __device__ inline StagePlan stage_plan(int nb, int qb, int nt, bool swiglu, size_t budget) {
    StagePlan pl{};
    pl.quad_bytes = (nb / 2) * (8 * qb + 16);
    pl.tps = 4;
    while (pl.tps > (swiglu ? 2 : 1) && pl.tps * pl.quad_bytes > 40 * 1024) pl.tps /= 2;
    pl.stage_bytes = (pl.tps * pl.quad_bytes + 127) / 128 * 128;
    pl.x_bytes = ((size_t)nt * stage_bytes_per_token(nb) + 127) / 128 * 128;
    const size_t room = budget > pl.x_bytes + 1024 ? budget - pl.x_bytes - 1024 : 0;
    pl.slots = (int)(room / pl.stage_bytes);
    if (pl.slots > 4) pl.slots = 4;
    pl.smem = pl.x_bytes + (size_t)pl.slots * pl.stage_bytes + 2 * kMaxStages * 8;
    return pl;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// true when the phase with the given parity has completed; false after kSpinLimit polls
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
    const uint32_t a = smem_u32(bar);
    for (uint32_t i = 0; i < kSpinLimit; ++i) {
        uint32_t done;
        // each poll suspends for at most ~1 us (time hint), so a wait gives up after a few seconds
        asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, 1000;\n\tselp.u32 %0, 1, 0, p;\n\t}"
                     : "=r"(done) : "r"(a), "r"(parity) : "memory");
        if (done) return true;
    }
    return false;
}
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}
// Producer side: one bulk copy of stage `st` of matrix p -- its row quads st * tps.. (a SwiGLU
// stage's tasks cover half feature quads, so its quad count is rounded up to even) -- into the
// ring slot at dst, completing on `bar` (one elected thread).
template <int EPI>
__device__ __forceinline__ void issue_stage(const GemvParams &p, const StagePlan &pl, int st, uint8_t *dst,
                                            uint64_t *bar) {
    const int tasks = min(pl.tps, p.n_tasks - st * pl.tps);   // the last stage may be short
    const int quads = EPI == EPI_SWIGLU ? tasks + (tasks & 1) : tasks;
    const uint32_t bytes = (uint32_t)quads * (uint32_t)pl.quad_bytes;
    mbar_expect_tx(bar, bytes);
    bulk_g2s(dst, p.w + (size_t)st * pl.tps * pl.quad_bytes, bytes, bar);
}

template <int NT>
using PartBuf = float[2][16][kConsumerWarps][NT];   // [parity][stage row][k-slice][token]

// Consumer side of one landed stage (the 256 consumer threads): warp w takes task w / KS of the
// stage and the w % KS-th slice of its blocks, releases the slot to the producer, and after the
// slices are summed in part[k & 1], tps * NT threads apply the epilogue. `dead` skips the work
// (after a timed-out wait) but keeps every barrier. best[t] collects the logits argmax keys.
template <int QT, int NT, int EPI, bool OUT16>
__device__ __forceinline__ void consume_stage(const GemvParams &p, const FwdArgs &a, int layer, const StagePlan &pl,
                                              const uint8_t *sq, const uint8_t *xstage, int st, int k, bool dead,
                                              uint64_t *empty_bar, PartBuf<NT> &part, float (*red)[8],
                                              unsigned long long (&best)[NT]) {
    constexpr int QB = QT == Q8 ? 32 : 16;
    const int nb = p.nb, tps = pl.tps, QBY = pl.quad_bytes;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KS = kConsumerWarps / tps;
    const int tg = warp / KS, ks = warp % KS;
    const int nbs = ((nb + KS - 1) / KS + 1) & ~1;   // even, so runs of 32 start on block pairs
    const int b_lo = min(nb, ks * nbs), b_hi = min(nb, b_lo + nbs);
    // quad (within the stage) and row within it of this warp's 4 rows: a plain task is one quad;
    // a SwiGLU task is rows 2h, 2h+1 of a gate quad and of the up quad after it (h = tg & 1)
    int qd[4], rr[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        if (EPI != EPI_SWIGLU) {
            qd[r] = tg;
            rr[r] = r;
        } else {
            qd[r] = 2 * (tg >> 1) + (r >> 1);
            rr[r] = 2 * (tg & 1) + (r & 1);
        }
    }
    // the epilogue threads' memory operands, loaded while the dot products run
    const int e = threadIdx.x;
    const int tasks = min(tps, p.n_tasks - st * tps);
    const bool epi_thread = !dead && e < tasks * NT && e % NT < p.T;
    EpiIn ein{};
    if ((EPI == EPI_RESID || EPI == EPI_QKV) && epi_thread) ein = epi_load<EPI>(a, e % NT, (st * tps + e / NT) * 4, p.N);
    float acc[4][NT];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int t = 0; t < NT; ++t) acc[r][t] = 0.f;
    const int lb = block_of_lane(lane);
    for (int b0 = b_lo; b0 < (dead ? b_lo : b_hi); b0 += 32) {
        const int b = b0 + lb;
        if (b >= b_hi) continue;
        XQ xq[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) load_xq(xstage + t * stage_bytes_per_token(nb), nb, b, xq[t]);
        float d[4];
        if (EPI != EPI_SWIGLU) {
            const uint2 s4 = *reinterpret_cast<const uint2 *>(sq + qd[0] * QBY + quad_s_off(QB, b));
            const float2 d01 = __half22float2(*reinterpret_cast<const __half2 *>(&s4.x));
            const float2 d23 = __half22float2(*reinterpret_cast<const __half2 *>(&s4.y));
            d[0] = d01.x; d[1] = d01.y; d[2] = d23.x; d[3] = d23.y;
        } else {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t s2 = *reinterpret_cast<const uint32_t *>(sq + qd[2 * h] * QBY + quad_s_off(QB, b) + 2 * rr[2 * h]);
                const float2 dd = __half22float2(*reinterpret_cast<const __half2 *>(&s2));
                d[2 * h] = dd.x;
                d[2 * h + 1] = dd.y;
            }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const uint4 *wp = reinterpret_cast<const uint4 *>(sq + qd[r] * QBY + quad_q_off(QB, rr[r], b));
            const uint4 w0 = wp[0];
            const uint4 w1 = QT == Q8 ? wp[1] : w0;
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                const int P = QT == Q4 ? q4_idot(w0, xq[t]) : q8_idot(w0, w1, xq[t]);
                acc[r][t] = fmaf(d[r] * xq[t].s, (float)P, acc[r][t]);
            }
        }
    }
    // the slot's bytes are no longer read by this warp: hand it back to the producer (a NULL
    // barrier: the slot is refilled after the CTA-wide barrier below instead)
    __syncwarp();
    if (lane == 0 && empty_bar) mbar_arrive(empty_bar);
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            float v = acc[r][t];
#pragma unroll
            for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane == 0) part[k & 1][tg * 4 + r][ks][t] = v;
        }
    consumer_sync();
    // epilogue: one thread per (task, token)
    if (epi_thread) {
        const int et = e / NT, t = e % NT;
        {
            float v[4];
            const float rs = token_rs(p, a, red, t);
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                float sum = 0.f;
                for (int q = 0; q < KS; ++q) sum += part[k & 1][et * 4 + r][q][t];
                v[r] = sum * rs;
            }
            const int task = st * tps + et;
            if (EPI == EPI_SWIGLU) {   // features 4 (task / 2) + 2 (task & 1) + {0, 1}
                const float g2[2] = {v[0], v[1]}, u2[2] = {v[2], v[3]};
                epi_swiglu2<OUT16>(a, t, 4 * (task >> 1) + 2 * (task & 1), g2, u2);
            } else {
                unsigned long long bk = 0ull;
                epi_quad_in<EPI>(a, layer, t, task * 4, p.N, v, ein, bk);
#pragma unroll
                for (int tt = 0; tt < NT; ++tt)
                    if (tt == t) best[tt] = bk > best[tt] ? bk : best[tt];
            }
        }
    }
    // part[k & 1] is rewritten two stages later, after the next consumer_sync
}

// The CTA's largest logits keys, one atomicMax per token into a.amax_key (consumer threads).
template <int NT>
__device__ __forceinline__ void logits_cta_reduce(const FwdArgs &a, int T, const unsigned long long (&best)[NT]) {
    __shared__ unsigned long long cbest[NT];
    consumer_sync();
    if (threadIdx.x < NT) cbest[threadIdx.x] = 0ull;
    consumer_sync();
#pragma unroll
    for (int tt = 0; tt < NT; ++tt)
        if (best[tt]) atomicMax(&cbest[tt], best[tt]);
    consumer_sync();
    if (threadIdx.x < NT && threadIdx.x < T && cbest[threadIdx.x]) atomicMax(&a.amax_key[threadIdx.x], cbest[threadIdx.x]);
}

template <int QT, int NT, int EPI, bool OUT16>
__global__ void __launch_bounds__(288, 1) k_gemv(const GemvParams p, const FwdArgs a, const int layer) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int QB = QT == Q8 ? 32 : 16;
    const int nb = p.nb;
    const StagePlan pl = stage_plan(nb, QB, NT, EPI == EPI_SWIGLU, (size_t)kGemvSmemTotal);
    uint8_t *xstage = smem;
    uint8_t *ring = smem + pl.x_bytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(ring + (size_t)pl.slots * pl.stage_bytes);
    uint64_t *empty = full + kMaxStages;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = pl.slots;
    const int n_stages = (p.n_tasks + pl.tps - 1) / pl.tps;
    LCX_TRACE(a, 0);

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kConsumerWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ---------------- producer: the weights do not depend on earlier kernels, so streaming
        // starts before the dependency wait
        if (lane == 0) {
            int k = 0;
            bool ok = true;
            for (int st = blockIdx.x; st < n_stages; st += gridDim.x, ++k) {
                const int slot = k % S;
                if (k >= S && !(ok = mbar_wait(&empty[slot], ((k / S) - 1) & 1))) break;
                issue_stage<EPI>(p, pl, st, ring + (size_t)slot * pl.stage_bytes, &full[slot]);
            }
            if (!ok) atomicExch(a.err, 1);
            // drain: every copy this CTA issued must land before the CTA exits
            const int issued = k;
            for (int j = (issued > S ? issued - S : 0); j < issued; ++j) mbar_wait(&full[j % S], (j / S) & 1);
        }
        return;
    }

    // ---------------- consumers (256 threads)
    if (p.in.g) {   // the norm gains are weights: bring them close before waiting
        for (int l = threadIdx.x; l < p.K / 32; l += 256)
            asm volatile("prefetch.global.L1 [%0];" ::"l"(p.in.g + 32 * l));
    }
    LCX_PDL_WAIT();
    LCX_PDL_TRIGGER();
    LCX_TRACE(a, 1);
    __shared__ float red[NT][8];
    for (int t = 0; t < NT; ++t) {
        if (t < p.T) {
            stage_token<QT>(p, t, xstage + t * stage_bytes_per_token(nb), red);
        } else {
            for (size_t i = threadIdx.x * 16; i < stage_bytes_per_token(nb); i += 256 * 16)
                *reinterpret_cast<uint4 *>(xstage + t * stage_bytes_per_token(nb) + i) = make_uint4(0, 0, 0, 0);
        }
    }
    consumer_sync();
    LCX_TRACE(a, 2);

    __shared__ PartBuf<NT> part;
    unsigned long long best[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) best[t] = 0ull;

    // After a timed-out wait a consumer keeps walking the stage loop (so every named barrier
    // still sees all 256 threads) but skips the waits and the work.
    bool dead = false;
    int k = 0;
    for (int st = blockIdx.x; st < n_stages; st += gridDim.x, ++k) {
        const int slot = k % S;
        if (!dead && !mbar_wait(&full[slot], (k / S) & 1)) {
            dead = true;
            atomicExch(a.err, 1);
        }
        consume_stage<QT, NT, EPI, OUT16>(p, a, layer, pl, ring + (size_t)slot * pl.stage_bytes, xstage, st, k, dead,
                                          &empty[slot], part, red, best);
    }
    LCX_TRACE(a, 3);
    if (EPI == EPI_LOGITS) logits_cta_reduce<NT>(a, p.T, best);
}

template <int QT, int NT, int EPI, bool OUT16>
cudaError_t run(const GemvParams &p, const FwdArgs &a, int layer, cudaStream_t s) {
    auto kern = k_gemv<QT, NT, EPI, OUT16>;
    constexpr int QB = QT == Q8 ? 32 : 16;
    const StagePlan pl = stage_plan(p.nb, QB, NT, EPI == EPI_SWIGLU, (size_t)kGemvSmemTotal);
    if (pl.slots < 2) return cudaErrorInvalidConfiguration;
    cudaError_t e = func_attr_once((const void *)kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGemvSmemTotal);
    if (e != cudaSuccess) return e;
    const int n_sm = device_sm_count();
    const int n_stages = (p.n_tasks + pl.tps - 1) / pl.tps;
    int grid = n_stages < n_sm ? n_stages : n_sm;
    if (grid < 1) grid = 1;
    return launch_pdl(kern, dim3(grid), dim3(288), pl.smem, s, p, a, layer);
}

}  // namespace gemv_detail
}  // namespace lcx
