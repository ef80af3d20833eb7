// Causal GQA attention for prefill ubatches on the tensor cores (mma.sync m16n8k16, f16 in, f32
// accumulate), flash-style: scores, online softmax and the P.V product per key tile, never
// materialising the score matrix.
//
// A query tile is up to 64 consecutive positions of one sequence inside the ubatch; a CTA
// (4 warps, 16 query rows each) takes one query tile and one query head, and walks the key tiles
// of that head's KV head -- one 64-cell page each, contiguous in the paged cache -- double
// buffered with cp.async into XOR-swizzled shared memory read by ldmatrix. A row attends the cells
// of its sequence with position <= its own (KV-cache section of the article: the tokens of a
// prefill see each other causally, their own K/V included). q and the softmax weights P are each
// carried as f16 high + low parts (two MMAs per product) so the products keep about 22 bits; K and
// V are the f16 values of the cache.
#include <math_constants.h>

#include "epilogue.cuh"

namespace lcx {

namespace {

constexpr int FA_BQ = 64;   // query rows per CTA
constexpr int FA_BK = 64;   // key cells per tile (= one page)

__device__ __forceinline__ uint32_t pack_half2(float lo_elem, float hi_elem) {
    const __half2 h = __floats2half2_rn(lo_elem, hi_elem);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// split (x0, x1) into f16 pairs hi = f16(x), lo = f16(x - hi)
__device__ __forceinline__ void split2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    const __half2 h = __floats2half2_rn(x0, x1);
    const float2 hf = __half22float2(h);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = pack_half2(x0 - hf.x, x1 - hf.y);
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// byte offset of 16-byte chunk c of row r in a [64][HD] f16 tile, chunks XOR-swizzled by row
template <int HD>
__device__ __forceinline__ uint32_t tile_off(int r, int c) {
    return (uint32_t)(r * HD * 2 + ((c ^ (r & 7)) << 4));
}

template <int HD>
__global__ void __launch_bounds__(128) k_attn_prefill(const FwdArgs a, const int layer) {
    constexpr int KSTEPS = HD / 16;   // k-steps of Q.K (head dims)
    constexpr int DT = HD / 8;        // n-tiles of P.V (head dims)
    constexpr int CH = HD / 8;        // 16-byte chunks per row
    extern __shared__ __align__(128) uint8_t sm[];   // [2][K tile, V tile]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, tq = lane & 3;
    const int4 tile = a.ub.qtiles[blockIdx.x];       // (first token, tokens, sequence, first position)
    const int h = blockIdx.y, G = a.H / a.KV, kvh = h / G;
    const int tok0 = tile.x, ntok = tile.y, seq = tile.z, p0 = tile.w;
    const int qw = a.H * HD;
    const float scale_log2 = rsqrtf((float)HD) * 1.4426950408889634f;

    LCX_PDL_WAIT();
    LCX_PDL_TRIGGER();

    // ---- Q fragments (this warp's 16 rows), f16 high + low
    uint32_t qa_hi[KSTEPS][4], qa_lo[KSTEPS][4];
    {
        const int r0 = warp * 16 + g, r1 = r0 + 8;
        const float *q0 = a.q + (size_t)(tok0 + r0) * qw + h * HD;
        const float *q1 = a.q + (size_t)(tok0 + r1) * qw + h * HD;
        const bool v0 = r0 < ntok, v1 = r1 < ntok;
#pragma unroll
        for (int kk = 0; kk < KSTEPS; ++kk) {
            const int c0 = kk * 16 + 2 * tq, c1 = c0 + 8;
            float2 x00 = v0 ? *reinterpret_cast<const float2 *>(q0 + c0) : make_float2(0.f, 0.f);
            float2 x10 = v1 ? *reinterpret_cast<const float2 *>(q1 + c0) : make_float2(0.f, 0.f);
            float2 x01 = v0 ? *reinterpret_cast<const float2 *>(q0 + c1) : make_float2(0.f, 0.f);
            float2 x11 = v1 ? *reinterpret_cast<const float2 *>(q1 + c1) : make_float2(0.f, 0.f);
            split2(x00.x, x00.y, qa_hi[kk][0], qa_lo[kk][0]);
            split2(x10.x, x10.y, qa_hi[kk][1], qa_lo[kk][1]);
            split2(x01.x, x01.y, qa_hi[kk][2], qa_lo[kk][2]);
            split2(x11.x, x11.y, qa_hi[kk][3], qa_lo[kk][3]);
        }
    }

    const int last_pos = p0 + ntok - 1;
    const int n_tiles = last_pos / FA_BK + 1;
    const int32_t *ptrow = a.pt + (size_t)seq * a.max_pages_per_seq;
    const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(sm);
    constexpr uint32_t TILE_BYTES = FA_BK * HD * 2;

    auto load_tile = [&](int kt, int buf) {
        const size_t row = (((size_t)layer * a.n_pages + ptrow[kt]) * a.KV + kvh) * kPage;   // page's first cell
        const __half *ksrc = a.kc + row * HD, *vsrc = a.vc + row * HD;
        const uint32_t kdst = sbase + buf * 2 * TILE_BYTES, vdst = kdst + TILE_BYTES;
        for (int i = threadIdx.x; i < FA_BK * CH; i += 128) {
            const int r = i / CH, c = i % CH;
            cp_async16(kdst + tile_off<HD>(r, c), ksrc + r * HD + c * 8);
            cp_async16(vdst + tile_off<HD>(r, c), vsrc + r * HD + c * 8);
        }
        cp_commit();
    };

    float o[DT][4];
#pragma unroll
    for (int d = 0; d < DT; ++d) o[d][0] = o[d][1] = o[d][2] = o[d][3] = 0.f;
    float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F, l0 = 0.f, l1 = 0.f;
    const int qp0 = p0 + warp * 16 + g, qp1 = qp0 + 8;   // positions of this thread's two rows

    load_tile(0, 0);
    for (int kt = 0; kt < n_tiles; ++kt) {
        const int buf = kt & 1;
        if (kt + 1 < n_tiles) {
            load_tile(kt + 1, buf ^ 1);
            cp_wait<1>();
        } else {
            cp_wait<0>();
        }
        __syncthreads();
        const uint32_t kbase = sbase + buf * 2 * TILE_BYTES, vbase = kbase + TILE_BYTES;

        // ---- S = Q K^T for 64 keys (8 n-tiles of 8)
        float s[8][4];
#pragma unroll
        for (int j = 0; j < 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < KSTEPS; ++kk) {
#pragma unroll
            for (int j = 0; j < 8; j += 2) {
                const int m = lane >> 3, rr = lane & 7;
                const int key = 8 * (j + (m >> 1)) + rr, c = 2 * kk + (m & 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(kbase + tile_off<HD>(key, c), b0, b1, b2, b3);
                mma16816(s[j], qa_hi[kk], b0, b1);
                mma16816(s[j], qa_lo[kk], b0, b1);
                mma16816(s[j + 1], qa_hi[kk], b2, b3);
                mma16816(s[j + 1], qa_lo[kk], b2, b3);
            }
        }
        // ---- scale, causal mask, online softmax (rows g and g + 8 of this warp)
        const bool diag = (kt + 1) * FA_BK - 1 > p0;   // the tile holds positions after the tile's first query
        float mx0 = -CUDART_INF_F, mx1 = -CUDART_INF_F;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int kp = kt * FA_BK + 8 * j + 2 * tq + e;
                float v0 = s[j][e] * scale_log2, v1 = s[j][2 + e] * scale_log2;
                if (diag) {
                    if (kp > qp0) v0 = -CUDART_INF_F;
                    if (kp > qp1) v1 = -CUDART_INF_F;
                }
                s[j][e] = v0;
                s[j][2 + e] = v1;
                mx0 = fmaxf(mx0, v0);
                mx1 = fmaxf(mx1, v1);
            }
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float al0 = exp2f(m0 - mn0), al1 = exp2f(m1 - mn1);   // m = -inf only before the first tile
        m0 = mn0;
        m1 = mn1;
        l0 *= al0;
        l1 *= al1;
#pragma unroll
        for (int d = 0; d < DT; ++d) {
            o[d][0] *= al0;
            o[d][1] *= al0;
            o[d][2] *= al1;
            o[d][3] *= al1;
        }
        // P as A fragments (hi + lo), key k-steps of 16 = n-tiles (2kk, 2kk + 1)
        uint32_t pa_hi[4][4], pa_lo[4][4];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int j = 2 * kk + half;
                const float p00 = exp2f(s[j][0] - mn0), p01 = exp2f(s[j][1] - mn0);
                const float p10 = exp2f(s[j][2] - mn1), p11 = exp2f(s[j][3] - mn1);
                l0 += p00 + p01;
                l1 += p10 + p11;
                split2(p00, p01, pa_hi[kk][2 * half], pa_lo[kk][2 * half]);
                split2(p10, p11, pa_hi[kk][2 * half + 1], pa_lo[kk][2 * half + 1]);
            }
        }
        // ---- O += P V
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
            for (int d = 0; d < DT; d += 2) {
                const int m = lane >> 3, rr = lane & 7;
                const int key = 16 * kk + 8 * (m & 1) + rr, c = d + (m >> 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(vbase + tile_off<HD>(key, c), b0, b1, b2, b3);
                mma16816(o[d], pa_hi[kk], b0, b1);
                mma16816(o[d], pa_lo[kk], b0, b1);
                mma16816(o[d + 1], pa_hi[kk], b2, b3);
                mma16816(o[d + 1], pa_lo[kk], b2, b3);
            }
        }
        __syncthreads();   // the buffer is refilled two tiles later
    }
    // ---- normalise and store (f16 high + low for the output projection)
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const float inv0 = 1.f / l0, inv1 = 1.f / l1;
    const int r0 = warp * 16 + g, r1 = r0 + 8;
#pragma unroll
    for (int d = 0; d < DT; ++d) {
        const int dim = d * 8 + 2 * tq;
        if (r0 < ntok) {
            const size_t oi = (size_t)(tok0 + r0) * qw + h * HD + dim;
            store_split(a.o16, a.o16_lo, oi, o[d][0] * inv0);
            store_split(a.o16, a.o16_lo, oi + 1, o[d][1] * inv0);
        }
        if (r1 < ntok) {
            const size_t oi = (size_t)(tok0 + r1) * qw + h * HD + dim;
            store_split(a.o16, a.o16_lo, oi, o[d][2] * inv1);
            store_split(a.o16, a.o16_lo, oi + 1, o[d][3] * inv1);
        }
    }
}

}  // namespace

cudaError_t launch_attention_prefill(const FwdArgs &a, int layer, cudaStream_t s, int64_t &launches) {
    ++launches;
    const dim3 grid(a.ub.n_qtiles, a.H);
    if (a.hd == 128) {
        cudaError_t e = func_attr_once((const void *)k_attn_prefill<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       4 * FA_BK * 128 * 2);
        if (e != cudaSuccess) return e;
        return launch_pdl(k_attn_prefill<128>, grid, dim3(128), (size_t)4 * FA_BK * 128 * 2, s, a, layer);
    }
    if (a.hd == 64) return launch_pdl(k_attn_prefill<64>, grid, dim3(128), (size_t)4 * FA_BK * 64 * 2, s, a, layer);
    return cudaErrorInvalidValue;
}

}  // namespace lcx
