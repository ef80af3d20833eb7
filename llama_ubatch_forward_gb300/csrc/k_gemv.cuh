// Weight-streaming GEMV for decode ubatches (T <= 8 tokens): y = W x with W in Q4_0 / Q8_0.
//
// Decode is bound by reading the weights once (KV-cache section of the article: decode loads
// memory, prefill loads the compute units), so the kernel is built to keep HBM busy with as
// few instructions per weight as possible:
//   * each warp owns a task of 4 rows and its lanes stride over the rows' 32-element blocks,
//     so every load instruction of a warp reads 512 contiguous bytes (16 B of nibbles or
//     2 x 16 B of int8 per lane); a row quad's 4 block scales arrive in one 8-byte load;
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
// The weight rows stream through a shared-memory ring filled by TMA bulk copies (see k_gemv).
#pragma once
#include "epilogue.cuh"

namespace lcx {
namespace gemv_detail {

// ---------------------------------------------------------------- staged activations
// Per token: hi plane [nb][32 B], lo plane [nb][32 B] (16-byte chunk c of block b stored at
// chunk c ^ ((b >> 2) & 1): 8 lanes reading 8 consecutive blocks hit 8 distinct bank groups),
// then meta [nb] (s / 128, C) with C = 8 (128 sum hi + sum lo) for Q4_0 and 0 for Q8_0.
__host__ __device__ constexpr size_t stage_bytes_per_token(int nb) { return (size_t)nb * 72; }

__device__ __forceinline__ int plane_chunk_off(int b, int c) { return b * 32 + ((c ^ ((b >> 2) & 1)) << 4); }

struct XQ {          // one block of one token, in registers
    int4 h0, h1;     // hi words 0..3, 4..7
    int4 l0, l1;     // lo words
    float s;         // s / 128
    int C;
};

__device__ __forceinline__ void load_xq(const uint8_t *stage_t, int nb, int b, XQ &x) {
    const uint8_t *hp = stage_t, *lp = stage_t + (size_t)nb * 32;
    const float2 *mp = reinterpret_cast<const float2 *>(stage_t + (size_t)nb * 64);
    x.h0 = *reinterpret_cast<const int4 *>(hp + plane_chunk_off(b, 0));
    x.h1 = *reinterpret_cast<const int4 *>(hp + plane_chunk_off(b, 1));
    x.l0 = *reinterpret_cast<const int4 *>(lp + plane_chunk_off(b, 0));
    x.l1 = *reinterpret_cast<const int4 *>(lp + plane_chunk_off(b, 1));
    const float2 m = mp[b];
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
    const uint8_t *qs;
    const __half *sc;
    int N, nb, K;
    int n_tasks;
    int T;
    GemvIn in;
};

// The 4 internal rows of a task. SwiGLU tasks take a gate row pair and the matching up pair
// (128 rows further, in the 128-row chunk layout of the fused gate/up matrix).
template <int EPI>
__device__ __forceinline__ int task_row(int task, int r) {
    if (EPI != EPI_SWIGLU) return task * 4 + r;
    const int c = task / (kRowTile / 2), qq = task % (kRowTile / 2);
    return c * 2 * kRowTile + 2 * qq + (r >= 2 ? kRowTile : 0) + (r & 1);
}

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// Stage token t: split every 32-element block of x * g (g = the RMSNorm gains, or 1) into
// hi / lo int8 parts, and leave this thread's share of sum(x^2) in red[t][warp]. The RMS factor
// is a positive scalar, so the block split does not depend on it: it multiplies each row's dot
// product in the epilogue instead, and the sum of squares is reduced while the blocks are being
// split. Two adjacent lanes share a block (16 elements each). Run by the 256 consumer threads.
template <int QT>
__device__ void stage_token(const GemvParams &p, int t, uint8_t *stage_t, float (*red)[8]) {
    constexpr int NTHR = 256;
    const int nb = p.nb, K = p.K;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float *xr = p.in.x + (size_t)(p.in.x_rows ? p.in.x_rows[t] : t) * K;
    uint8_t *hp = stage_t, *lp = stage_t + (size_t)nb * 32;
    float2 *mp = reinterpret_cast<float2 *>(stage_t + (size_t)nb * 64);
    float ss = 0.f;
    const int n_half = 2 * nb, iters = (n_half + NTHR - 1) / NTHR;   // same trip count in every lane
    for (int it = 0; it < iters; ++it) {
        const int hb = it * NTHR + threadIdx.x, b = hb >> 1, half = hb & 1;
        const bool active = hb < n_half;
        float v[16];
#pragma unroll
        for (int j = 0; j < 16; j += 4) {
            float4 q = active ? *reinterpret_cast<const float4 *>(xr + b * 32 + half * 16 + j) : make_float4(0, 0, 0, 0);
            ss += q.x * q.x + q.y * q.y + q.z * q.z + q.w * q.w;
            if (p.in.g && active) {
                const float4 gg = *reinterpret_cast<const float4 *>(p.in.g + b * 32 + half * 16 + j);
                q.x *= gg.x; q.y *= gg.y; q.z *= gg.z; q.w *= gg.w;
            }
            v[j] = q.x; v[j + 1] = q.y; v[j + 2] = q.z; v[j + 3] = q.w;
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
            *reinterpret_cast<uint4 *>(hp + plane_chunk_off(b, half)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4 *>(lp + plane_chunk_off(b, half)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
            if (half == 0) {
                const int C = QT == Q4 ? 8 * (128 * sh + sl) : 0;
                mp[b] = make_float2(amax * (1.0f / (127.0f * 128.0f)), __int_as_float(C));
            }
        }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) red[t][warp] = ss;
}

// RMS factor of token t from the partial sums left by stage_token (1 without norm gains).
__device__ __forceinline__ float token_rs(const GemvParams &p, const FwdArgs &a, float (*red)[8], int t) {
    if (!p.in.g) return 1.f;
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) tot += red[t][w];
    return 1.0f / sqrtf(tot / (float)p.K + a.eps);
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
    int tps;            // tasks per stage (4, 2 or 1)
    int slots;          // ring depth
    int qs_bytes;       // quant bytes of one stage
    int sc_bytes;       // scale bytes of one stage
    int stage_bytes;    // qs + sc, rounded to 128
    size_t x_bytes;     // staged activations
    size_t smem;        // total dynamic shared memory
};

__host__ __device__ inline StagePlan stage_plan(int nb, int qb, int nt, bool swiglu, size_t budget) {
    StagePlan pl{};
    const int row = nb * qb;
    pl.tps = 4;
    while (pl.tps > (swiglu ? 2 : 1) && pl.tps * 4 * (row + nb * 2) > 40 * 1024) pl.tps /= 2;
    pl.qs_bytes = pl.tps * 4 * row;
    pl.sc_bytes = pl.tps * nb * 8;
    pl.stage_bytes = (pl.qs_bytes + pl.sc_bytes + 127) / 128 * 128;
    pl.x_bytes = ((size_t)nt * stage_bytes_per_token(nb) + 127) / 128 * 128;
    const size_t room = budget > pl.x_bytes + 1024 ? budget - pl.x_bytes - 1024 : 0;
    pl.slots = (int)(room / pl.stage_bytes);
    if (pl.slots > kMaxStages) pl.slots = kMaxStages;
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
// First task of stage `st`, and the global rows / scale quads a stage copies.
template <int EPI>
__device__ __forceinline__ void stage_rows(int st, int tps, int &row_a, int &row_b) {
    const int t0 = st * tps;
    if (EPI != EPI_SWIGLU) {
        row_a = t0 * 4;
        row_b = -1;
    } else {
        const int c = t0 / (kRowTile / 2), qq = t0 % (kRowTile / 2);
        row_a = c * 2 * kRowTile + 2 * qq;   // 2 * tps gate rows
        row_b = row_a + kRowTile;            // 2 * tps up rows
    }
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
    const int tps = pl.tps, S = pl.slots;
    const int n_stages = (p.n_tasks + tps - 1) / tps;
    const int row_bytes = nb * QB;
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
        // ---------------- producer
        if (lane == 0) {
            int k = 0;
            bool ok = true;
            for (int st = blockIdx.x; st < n_stages; st += gridDim.x, ++k) {
                const int slot = k % S;
                if (k >= S && !(ok = mbar_wait(&empty[slot], ((k / S) - 1) & 1))) break;
                uint8_t *dst = ring + (size_t)slot * pl.stage_bytes;
                int ra, rb;
                stage_rows<EPI>(st, tps, ra, rb);
                const int tasks = min(tps, p.n_tasks - st * tps);   // the last stage may be short
                const int rows = EPI == EPI_SWIGLU ? 2 * tasks : 4 * tasks;
                const int quads = EPI == EPI_SWIGLU ? (2 * tasks + 3) / 4 : tasks;
                const uint32_t qbytes = (uint32_t)rows * row_bytes, sbytes = (uint32_t)quads * nb * 8;
                const uint32_t tx = (EPI == EPI_SWIGLU ? 2u : 1u) * (qbytes + sbytes);
                mbar_expect_tx(&full[slot], tx);
                bulk_g2s(dst, p.qs + (size_t)ra * row_bytes, qbytes, &full[slot]);
                bulk_g2s(dst + pl.qs_bytes, p.sc + (size_t)(ra >> 2) * nb * 4, sbytes, &full[slot]);
                if (EPI == EPI_SWIGLU) {
                    bulk_g2s(dst + pl.qs_bytes / 2, p.qs + (size_t)rb * row_bytes, qbytes, &full[slot]);
                    bulk_g2s(dst + pl.qs_bytes + pl.sc_bytes / 2, p.sc + (size_t)(rb >> 2) * nb * 4, sbytes, &full[slot]);
                }
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

    const int KS = kConsumerWarps / tps;
    const int tg = warp / KS, ks = warp % KS;
    const int nbs = (nb + KS - 1) / KS, b_lo = ks * nbs, b_hi = min(nb, b_lo + nbs);
    __shared__ float part[2][16][kConsumerWarps][NT];   // [parity][stage row][k-slice][token]
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
        const uint8_t *sq = ring + (size_t)slot * pl.stage_bytes;
        const __half *ss = reinterpret_cast<const __half *>(sq + pl.qs_bytes);
        // local rows of this warp's task inside the stage, and where their scales sit
        int lrow[4], sidx[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            if (EPI != EPI_SWIGLU) {
                lrow[r] = tg * 4 + r;
                sidx[r] = tg * nb * 4 + r;                              // + b * 4
            } else {
                const int gl = 2 * tg + (r & 1);                        // row within the gate / up half
                lrow[r] = (r < 2 ? 0 : 2 * tps) + gl;
                sidx[r] = (r < 2 ? 0 : (tps / 2) * nb * 4) + (gl >> 2) * nb * 4 + (gl & 3);
            }
        }
        float acc[4][NT];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int t = 0; t < NT; ++t) acc[r][t] = 0.f;
        for (int b = b_lo + lane; b < (dead ? b_lo : b_hi); b += 32) {
            XQ xq[NT];
#pragma unroll
            for (int t = 0; t < NT; ++t) load_xq(xstage + t * stage_bytes_per_token(nb), nb, b, xq[t]);
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const uint4 *wp = reinterpret_cast<const uint4 *>(sq + ((size_t)lrow[r] * nb + b) * QB);
                const uint4 w0 = wp[0];
                const uint4 w1 = QT == Q8 ? wp[1] : w0;
                const float d = __half2float(ss[sidx[r] + b * 4]);
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    const int P = QT == Q4 ? q4_idot(w0, xq[t]) : q8_idot(w0, w1, xq[t]);
                    acc[r][t] = fmaf(d * xq[t].s, (float)P, acc[r][t]);
                }
            }
        }
        // the slot's bytes are no longer read by this warp: hand it back to the producer
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
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
        const int e = threadIdx.x;
        const int tasks = min(tps, p.n_tasks - st * tps);
        if (!dead && e < tasks * NT) {
            const int et = e / NT, t = e % NT;
            if (t < p.T) {
                float v[4];
#pragma unroll
                const float rs = token_rs(p, a, red, t);
                for (int r = 0; r < 4; ++r) {
                    float sum = 0.f;
                    for (int q = 0; q < KS; ++q) sum += part[k & 1][et * 4 + r][q][t];
                    v[r] = sum * rs;
                }
                const int task = st * tps + et;
                if (EPI == EPI_SWIGLU) {
                    const int c = task / (kRowTile / 2), qq = task % (kRowTile / 2);
                    const float g2[2] = {v[0], v[1]}, u2[2] = {v[2], v[3]};
                    epi_swiglu2<OUT16>(a, t, c * kRowTile + 2 * qq, g2, u2);
                } else {
                    unsigned long long bk = 0ull;
                    epi_quad<EPI>(a, layer, t, task * 4, p.N, v, bk);
#pragma unroll
                    for (int tt = 0; tt < NT; ++tt)
                        if (tt == t) best[tt] = bk > best[tt] ? bk : best[tt];
                }
            }
        }
        // part[k & 1] is rewritten two stages later, after the next consumer_sync
    }
    LCX_TRACE(a, 3);
    if (EPI == EPI_LOGITS) {
        __shared__ unsigned long long cbest[NT];
        consumer_sync();
        if (threadIdx.x < NT) cbest[threadIdx.x] = 0ull;
        consumer_sync();
#pragma unroll
        for (int tt = 0; tt < NT; ++tt)
            if (best[tt]) atomicMax(&cbest[tt], best[tt]);
        consumer_sync();
        if (threadIdx.x < NT && threadIdx.x < p.T && cbest[threadIdx.x]) atomicMax(&a.amax_key[threadIdx.x], cbest[threadIdx.x]);
    }
}

template <int QT, int NT, int EPI, bool OUT16>
cudaError_t run(const GemvParams &p, const FwdArgs &a, int layer, cudaStream_t s) {
    auto kern = k_gemv<QT, NT, EPI, OUT16>;
    constexpr int QB = QT == Q8 ? 32 : 16;
    const StagePlan pl = stage_plan(p.nb, QB, NT, EPI == EPI_SWIGLU, (size_t)kGemvSmemTotal);
    if (pl.slots < 2) return cudaErrorInvalidConfiguration;
    static int n_sm = 0;
    if (!n_sm) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGemvSmemTotal);
        if (e != cudaSuccess) return e;
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
    }
    const int n_stages = (p.n_tasks + pl.tps - 1) / pl.tps;
    int grid = n_stages < n_sm ? n_stages : n_sm;
    if (grid < 1) grid = 1;
    return launch_pdl(kern, dim3(grid), dim3(288), pl.smem, s, p, a, layer);
}

}  // namespace gemv_detail
}  // namespace lcx
