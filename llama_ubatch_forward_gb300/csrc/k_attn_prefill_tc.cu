// Causal GQA flash attention for prefill ubatches on the 5th-generation tensor cores (tcgen05 +
// TMEM + TMA): scores, online softmax and the P.V product per key tile, never materialising the
// score matrix (KV-cache section of the article: the tokens of a prefill attend the cached cells
// of their sequence and each other causally, their own K/V included).
//
// One CTA takes 128 query rows -- the 4 query heads that share one KV head x 32 consecutive
// tokens of one sequence -- so every K/V tile it loads serves all four heads (grouped-query
// attention), and walks the key tiles of that KV head, 128 cells (two pages) each:
//   warp 0      TMA producer: K and V of a tile (one box per page and 64-dim half, 128-byte
//               swizzle) into a ring of two stages;
//   warp 1      allocates TMEM and issues tcgen05.mma from one lane: S_j = Q_hi K_j^T + Q_lo K_j^T
//               into one of two score buffers (M 128 rows, N 128 cells), then O += P_hi V_j +
//               P_lo V_j with P read from tensor memory (written over S_j by the softmax) and V
//               read in the cache's own [cell][dim] layout (an MN-major B operand);
//   warps 2..5  one row each (TMEM lane = row): load Q and split it into f16 high + low parts,
//               then per tile the causal mask, the running maximum and sum, P = 2^(s - m) as f16
//               high + low parts stored over the scores, and the rescaling of O by 2^(m_old -
//               m_new); finally O / l, stored as f16 high + low parts for the output projection.
// S_{j+1} is issued before P_j V_j, so the scores of the next tile are computed while the softmax
// of this one runs. q and P each keep about 22 bits (two MMAs per product), K and V are the f16
// values of the cache, accumulation is f32 in tensor memory. All mbarrier waits are bounded; a
// timeout sets the context's error word and the CTA finishes without further work.
#include <math_constants.h>

#include "epilogue.cuh"
#include "tc_common.cuh"

namespace lcx {
namespace tc {
namespace fa {

constexpr int G = 4;          // query heads per KV head
constexpr int TQ = 32;        // tokens per CTA (G x TQ = 128 rows)
constexpr int BC = 128;       // cells per key tile: two pages
constexpr int NTHREADS = 192;

template <int HD>
struct Cfg {
    static constexpr int NH = HD / 64;                 // 64-dim halves: one 128-byte swizzle row each
    static constexpr int Q_BYTES = 128 * HD * 2;       // Q_hi or Q_lo: [half][128 rows][64]
    static constexpr int KV_BYTES = BC * HD * 2;       // a K or V tile: [half][128 cells][64]
    static constexpr int HALF = BC * 128;              // bytes of one half of a K or V tile
    static constexpr int STAGES = 2;
    // at least 116 KB, so that one CTA holds an SM: each allocates all 512 TMEM columns
    static constexpr int SMEM_NEED = 2 * Q_BYTES + STAGES * 2 * KV_BYTES + 1024 /* align */ + 256 /* barriers */;
    static constexpr int SMEM = SMEM_NEED > 116 * 1024 ? SMEM_NEED : 116 * 1024;
    static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
};

// TMEM columns: score buffers b = 0, 1 at 128 b (P written over them as packed f16 pairs: the 32
// scores of cells 32c.. become 16 columns of high parts and 16 of low parts), O at 256.
constexpr uint32_t O_COL = 256;

// Instruction descriptor of kind::f16 with B MN-major (transpose bit): f16 A and B, f32 D.
__host__ __device__ constexpr uint32_t idesc_f16_bmn(int m, int n) { return idesc_f16(m, n) | (1u << 16); }

// Shared-memory descriptor of an MN-major operand in the 128-byte swizzle layout: rows of 128
// bytes hold 64 consecutive MN elements of one K index, 8-row groups 1024 bytes apart along K,
// the next 64 MN elements `lbo` bytes further.
__device__ __forceinline__ uint64_t sw128_desc_mn(uint32_t addr, uint32_t lbo) {
    return (sw128_desc(addr) & ~((uint64_t)0x3FFF << 16)) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16);
}

// O += P V with A (P) in tensor memory
__device__ __forceinline__ void mma_f16_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
                 ::"r"(tmem_d), "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
                 "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
                 ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]),
                   "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
                   "r"(v[15])
                 : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
                 "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
                 "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
                 ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]),
                   "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
                   "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
                   "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
                   "r"(v[29]), "r"(v[30]), "r"(v[31])
                 : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// f16 high part of x and the f16 rounding of the rest, packed for two elements (x0 in the low half)
__device__ __forceinline__ void split_pack(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    const __half2 h = __floats2half2_rn(x0, x1);
    const float2 hf = __half22float2(h);
    const __half2 l = __floats2half2_rn(x0 - hf.x, x1 - hf.y);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

// 2^x by the hardware approximation (relative error about 2^-22; results below 2^-126 flush to 0)
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <int HD>
__global__ void __launch_bounds__(NTHREADS, 1)
    k_attn_prefill_tc(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                      const FwdArgs a, const int layer) {
    using C = Cfg<HD>;
    extern __shared__ uint8_t smem_raw[];
    // this CTA's 32 tokens: half of a 64-token query tile of the ubatch
    // the ubatch's last tiles (the most key tiles under the causal mask) are scheduled first
    const int4 tile = a.ub.qtiles[a.ub.n_qtiles - 1 - (int)(blockIdx.x >> 1)];
    const int half = 1 - (int)(blockIdx.x & 1);
    const int tok0 = tile.x + TQ * half, ntok = min(TQ, tile.y - TQ * half), seq = tile.z, p0 = tile.w + TQ * half;
    if (ntok <= 0) return;   // the whole CTA, before any barrier or allocation
    const int kvh = blockIdx.y;
    const int last_pos = p0 + ntok - 1;
    const int n_kt = last_pos / BC + 1;           // key tiles
    const int last_page = last_pos / kPage;
    const int32_t *ptrow = a.pt + (size_t)seq * a.max_pages_per_seq;

    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t *q_hi = smem, *q_lo = smem + C::Q_BYTES;
    uint8_t *kv = smem + 2 * C::Q_BYTES;
    auto k_tile = [&](int s) { return kv + s * 2 * C::KV_BYTES; };
    auto v_tile = [&](int s) { return kv + s * 2 * C::KV_BYTES + C::KV_BYTES; };
    uint64_t *bars = reinterpret_cast<uint64_t *>(kv + C::STAGES * 2 * C::KV_BYTES);
    // full_kv / empty_kv: a stage's K and V landed / read by the MMAs; s_full: a score buffer
    // computed; p_full: P written over it (and O rescaled); p_free: its P read; o_done: one P.V
    // product complete; q_full: Q staged
    uint64_t *full_kv = bars, *empty_kv = bars + 2, *s_full = bars + 4, *p_full = bars + 6, *p_free = bars + 8,
             *o_done = bars + 10, *q_full = bars + 11;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 12);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&full_kv[i], 1);
            mbar_init(&empty_kv[i], 1);
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 4);   // one arrival per softmax warp
            mbar_init(&p_free[i], 1);
        }
        mbar_init(o_done, 1);
        mbar_init(q_full, 4);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(tmem_slot)), "r"(512u));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------------------------------------------------------- K/V producer
        if (lane == 0) {
            bool ok = true;
            LCX_PDL_WAIT();   // this ubatch's own K/V come from the previous kernel
            int issued = 0;
            for (int j = 0; j < n_kt && ok; ++j) {
                const int s = j & 1;
                if (j >= 2 && !(ok = mbar_wait(&empty_kv[s], ((j >> 1) - 1) & 1))) break;
                mbar_expect_tx(&full_kv[s], 2u * C::KV_BYTES);
                for (int pg = 0; pg < 2; ++pg) {
                    // a page past the sequence's last one repeats the last (finite values; every
                    // cell of it is masked)
                    const int page = __ldg(ptrow + min(2 * j + pg, last_page));
                    const int row = ((layer * a.n_pages + page) * a.KV + kvh) * kPage;
                    for (int h = 0; h < C::NH; ++h) {
                        tma_2d(k_tile(s) + h * C::HALF + pg * kPage * 128, &tm_k, h * 64, row, &full_kv[s]);
                        tma_2d(v_tile(s) + h * C::HALF + pg * kPage * 128, &tm_v, h * 64, row, &full_kv[s]);
                    }
                }
                issued = j + 1;
            }
            if (!ok) atomicExch(a.err, 1);
            // every copy issued lands before the CTA exits
            for (int j = (issued > 2 ? issued - 2 : 0); j < issued; ++j) mbar_wait(&full_kv[j & 1], (j >> 1) & 1);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_f16(128, BC);
            constexpr uint32_t idesc_o = idesc_f16_bmn(128, HD);
            bool ok = mbar_wait(q_full, 0);
            // t: S_t (if t < n_kt), then P_{t-1} V_{t-1} (if t >= 1)
            for (int t = 0; t <= n_kt && ok; ++t) {
                if (t < n_kt) {
                    const int s = t & 1, b = t & 1;
                    ok = mbar_wait(&full_kv[s], (t >> 1) & 1);
                    if (ok && t >= 2) ok = mbar_wait(&p_free[b], ((t >> 1) - 1) & 1);
                    if (!ok) break;
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const uint32_t kb = saddr(k_tile(s));
#pragma unroll
                    for (int kk = 0; kk < HD / 16; ++kk) {
                        const uint32_t off = (kk >> 2) * C::HALF + (kk & 3) * 32;
                        const uint32_t qoff = (kk >> 2) * (128 * 128) + (kk & 3) * 32;
                        mma_f16(tmem + b * BC, sw128_desc(saddr(q_hi) + qoff), sw128_desc(kb + off), idesc_s, kk > 0);
                        mma_f16(tmem + b * BC, sw128_desc(saddr(q_lo) + qoff), sw128_desc(kb + off), idesc_s, 1u);
                    }
                    mma_commit(&s_full[b]);
                }
                if (t >= 1) {
                    const int u = t - 1, s = u & 1, b = u & 1;
                    if (!(ok = mbar_wait(&p_full[b], (u >> 1) & 1))) break;
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const uint32_t vb = saddr(v_tile(s));
#pragma unroll
                    for (int kk = 0; kk < BC / 16; ++kk) {
                        // 16 cells: two 8-row groups of the V tile; the 64-dim halves HALF apart
                        const uint64_t bdesc = sw128_desc_mn(vb + kk * 2048, C::HALF);
                        // P of cells 16kk..16kk+15: high parts at 32 (kk / 2) + 8 (kk % 2), low 16 further
                        const uint32_t pcol = b * BC + 32 * (kk >> 1) + 8 * (kk & 1);
                        mma_f16_ts(tmem + O_COL, tmem + pcol, bdesc, idesc_o, (u > 0 || kk > 0) ? 1u : 0u);
                        mma_f16_ts(tmem + O_COL, tmem + pcol + 16, bdesc, idesc_o, 1u);
                    }
                    mma_commit(&empty_kv[s]);
                    mma_commit(&p_free[b]);
                    mma_commit(o_done);
                }
            }
            if (!ok) atomicExch(a.err, 1);
        }
    } else {
        // ---------------------------------------------------------------- softmax warps
        const int qtr = warp & 3;                     // TMEM lane quarter = query head in the group
        const int row = qtr * 32 + lane;              // TMEM lane
        const int head = kvh * G + qtr;
        const int qw = a.H * HD;
        const bool valid = lane < ntok;
        const int qpos = valid ? p0 + lane : p0;      // rows past the tile's tokens see cell p0 only
        const uint32_t tl = tmem + ((uint32_t)(qtr * 32) << 16);
        LCX_PDL_WAIT();   // q comes from the previous kernel
        LCX_PDL_TRIGGER();
        {
            // Q row -> f16 high + low parts in the K-major 128-byte swizzle layout
            const float *qrow = a.q + (size_t)(tok0 + (valid ? lane : 0)) * qw + head * HD;
#pragma unroll
            for (int c = 0; c < HD / 8; ++c) {        // 16-byte chunks of 8 dims
                float x[8];
                const float4 u0 = valid ? *reinterpret_cast<const float4 *>(qrow + c * 8) : make_float4(0.f, 0.f, 0.f, 0.f);
                const float4 u1 = valid ? *reinterpret_cast<const float4 *>(qrow + c * 8 + 4) : make_float4(0.f, 0.f, 0.f, 0.f);
                x[0] = u0.x; x[1] = u0.y; x[2] = u0.z; x[3] = u0.w;
                x[4] = u1.x; x[5] = u1.y; x[6] = u1.z; x[7] = u1.w;
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) split_pack(x[2 * e], x[2 * e + 1], hi[e], lo[e]);
                const uint32_t off = (c >> 3) * (128 * 128) + row * 128 + (((c & 7) ^ (row & 7)) << 4);
                *reinterpret_cast<uint4 *>(q_hi + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4 *>(q_lo + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // generic writes -> tensor-core reads
            __syncwarp();
            if (lane == 0) mbar_arrive(q_full);
        }
        const float scale = rsqrtf((float)HD) * 1.4426950408889634f;
        float m = -CUDART_INF_F, l = 0.f;
        bool ok = true;
        for (int j = 0; j < n_kt; ++j) {
            const int b = j & 1;
            ok = __all_sync(0xffffffffu, mbar_wait(&s_full[b], (j >> 1) & 1));
            if (!ok) break;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            uint32_t sv[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld32_issue(tl + b * BC + c * 32, sv[c]);
            tmem_ld_wait(sv[0]);
            regs_ready(sv[1]);
            regs_ready(sv[2]);
            regs_ready(sv[3]);
            // the causal mask, on the tiles that hold a cell after the CTA's first position (the
            // same answer for every row of the CTA)
            const int cpos0 = j * BC;
            if (cpos0 + BC - 1 > p0) {
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (cpos0 + c * 32 + i > qpos) sv[c][i] = __float_as_uint(-CUDART_INF_F);
            }
            float mx = -CUDART_INF_F;
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int i = 0; i < 32; ++i) mx = fmaxf(mx, __uint_as_float(sv[c][i]));
            // The reference maximum m moves only when the tile's maximum exceeds it by more than
            // 8 (so P <= 2^8, exact enough in the f16 high + low pair); O and l are rescaled
            // only then, and the final O / l uses the same m throughout. Tile 0 holds cell 0 for
            // every row, so m is finite from the first tile on.
            const float mxs = mx * scale;
            const float m_new = mxs > m + 8.f ? mxs : m;
            const float alpha = ex2_approx(m - m_new);
            // P = 2^(s scale - m) as f16 high + low parts, written over the chunk's own 32 columns:
            // cells 32c..32c+31 -> high parts in columns 32c..32c+15, low parts in 32c+16..32c+31
            float psum = 0.f;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t ph[16], pl[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float e0 = ex2_approx(fmaf(__uint_as_float(sv[c][2 * i]), scale, -m_new));
                    const float e1 = ex2_approx(fmaf(__uint_as_float(sv[c][2 * i + 1]), scale, -m_new));
                    psum += e0 + e1;
                    split_pack(e0, e1, ph[i], pl[i]);
                }
                tmem_st16(tl + b * BC + c * 32, ph);
                tmem_st16(tl + b * BC + c * 32 + 16, pl);
            }
            l = l * alpha + psum;
            m = m_new;
            // O from the previous tiles, rescaled to the new maximum once its last product is done
            if (j > 0) {
                ok = __all_sync(0xffffffffu, mbar_wait(o_done, (j - 1) & 1));
                if (!ok) break;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                if (!__all_sync(0xffffffffu, alpha == 1.f)) {
#pragma unroll
                    for (int c = 0; c < HD / 32; ++c) {
                        uint32_t ov[32];
                        tmem_ld32_issue(tl + O_COL + c * 32, ov);
                        tmem_ld_wait(ov);
#pragma unroll
                        for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
                        tmem_st32(tl + O_COL + c * 32, ov);
                    }
                }
            }
            tmem_st_wait();
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[b]);
        }
        // the last product, then O / l as f16 high + low parts
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(o_done, (n_kt - 1) & 1));
        if (!ok) {
            atomicExch(a.err, 1);
        } else {
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const float inv = 1.f / l;
#pragma unroll
            for (int c = 0; c < HD / 32; ++c) {
                uint32_t ov[32];
                tmem_ld32_issue(tl + O_COL + c * 32, ov);
                tmem_ld_wait(ov);
                if (valid) {
                    // the row's 32 dims as f16 high + low parts, 16-byte stores (8 dims each)
                    const size_t oi = (size_t)(tok0 + lane) * qw + head * HD + c * 32;
#pragma unroll
                    for (int v8 = 0; v8 < 4; ++v8) {
                        uint32_t hi[4], lo[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            split_pack(__uint_as_float(ov[8 * v8 + 2 * e]) * inv, __uint_as_float(ov[8 * v8 + 2 * e + 1]) * inv,
                                       hi[e], lo[e]);
                        *reinterpret_cast<uint4 *>(a.o16 + oi + 8 * v8) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                        *reinterpret_cast<uint4 *>(a.o16_lo + oi + 8 * v8) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                    }
                }
            }
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512u));
    }
}

template <int HD>
cudaError_t run(const FwdArgs &a, int layer, cudaStream_t s) {
    using C = Cfg<HD>;
    auto kern = k_attn_prefill_tc<HD>;
    cudaError_t e = func_attr_once((const void *)kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    // the cache as [rows = L x n_pages x KV x kPage][HD] f16; a box is 64 cells x 64 dims
    const uint64_t rows = (uint64_t)a.L * a.n_pages * a.KV * kPage;
    alignas(64) CUtensorMap tk, tv;
    if (!make_map_2d(&tk, a.kc, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, HD, rows, (uint64_t)HD * 2, 64, kPage,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map_2d(&tv, a.vc, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, HD, rows, (uint64_t)HD * 2, 64, kPage,
                     CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * a.ub.n_qtiles, a.KV);
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = (size_t)C::SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tk, tv, a, layer);
}

}  // namespace fa
}  // namespace tc

bool attention_prefill_tc_fits(const FwdArgs &a) {
    // the cache's rows (layer, page, KV head, cell) are TMA coordinates: signed 32-bit
    const long long rows = (long long)a.L * a.n_pages * a.KV * kPage;
    return a.H == tc::fa::G * a.KV && (a.hd == 64 || a.hd == 128) && rows <= 0x7fffffffLL;
}

cudaError_t launch_attention_prefill_tc(const FwdArgs &a, int layer, cudaStream_t s, int64_t &launches) {
    ++launches;
    if (a.hd == 128) return tc::fa::run<128>(a, layer, s);
    if (a.hd == 64) return tc::fa::run<64>(a, layer, s);
    return cudaErrorInvalidValue;
}

}  // namespace lcx
