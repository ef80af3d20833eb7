// Weight-streaming GEMV for decode ubatches (T <= 8 tokens): y = W x with W in Q4_0 / Q8_0.
//
// Decode is bound by reading the weights once (KV-cache section of the article: decode loads
// memory, prefill loads the compute units), so this kernel is built around HBM streaming:
//   * each warp owns a task of 4 rows (a quad) -- 8 rows for the gate/up pair of SwiGLU -- and
//     its lanes stride over the row's 32-element blocks, so every load instruction of a warp
//     reads 512 contiguous bytes (16 B of nibbles or 2 x 16 B of int8 per lane);
//   * the activations are staged once per CTA in shared memory (RMSNorm fused into that
//     prologue), in a 16-byte-chunk XOR swizzle so the lanes' 16-byte reads are conflict free;
//   * nibbles are turned into exact floats in registers with one LOP3 each: OR-ing a nibble
//     at bit s into the mantissa of 2^23 gives 2^23 + q*2^s, and subtracting 2^23 + 8*2^s
//     leaves (q-8)*2^s exactly; the staged activation of that element is pre-multiplied by
//     2^-s, so the packed f32x2 FMA sums exact products (no precision is lost to the trick);
//   * a block's 32 products are summed, scaled once by the block's fp16 scale, accumulated
//     in f32, and the row sums are reduced with warp shuffles.
#pragma once
#include "epilogue.cuh"

namespace lcx {
namespace gemv_detail {

__device__ __forceinline__ float2 f2add(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 f2fma(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float u2f(uint32_t u) { return __uint_as_float(u); }

constexpr uint32_t kMagic = 0x4B000000u;   // 2^23
constexpr float kTwo23 = 8388608.0f;

// shift (bit position) of the nibble holding element e of a Q4_0 block, after the split into
// w (bytes 0..2 low half) and w >> 12 (the rest): lo/hi nibble of byte c
__host__ __device__ constexpr int q4_shift(int c, int hi) {
    return c == 0 ? (hi ? 4 : 0) : c == 1 ? (hi ? 12 : 8) : c == 2 ? (hi ? 8 : 16) : (hi ? 16 : 12);
}

// float offset of element chunk j (elements 4j..4j+3) of block b in the swizzled stage
__device__ __forceinline__ int xs_chunk(int b, int j) { return (b * 8 + (j ^ (b & 7))) * 4; }

// Partial sums of one 32-element Q4_0 block against NT staged token vectors.
template <int NT>
__device__ __forceinline__ void q4_block(const uint4 w, const float *xs_b[NT], int b, float part[NT]) {
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
    float2 acc[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t] = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t lo = ws[i], hi = ws[i] >> 12;
        // (q - 8) * 2^s for the low and high nibble of each byte c
        const float2 d0 = f2add(make_float2(u2f((lo & 0xFu) | kMagic), u2f((lo & 0xF0u) | kMagic)),
                                make_float2(-(kTwo23 + 8.f), -(kTwo23 + 128.f)));
        const float2 d1 = f2add(make_float2(u2f((lo & 0xF00u) | kMagic), u2f((lo & 0xF000u) | kMagic)),
                                make_float2(-(kTwo23 + 2048.f), -(kTwo23 + 32768.f)));
        const float2 d2 = f2add(make_float2(u2f((lo & 0xF0000u) | kMagic), u2f((hi & 0xF00u) | kMagic)),
                                make_float2(-(kTwo23 + 524288.f), -(kTwo23 + 2048.f)));
        const float2 d3 = f2add(make_float2(u2f((hi & 0xF000u) | kMagic), u2f((hi & 0xF0000u) | kMagic)),
                                make_float2(-(kTwo23 + 32768.f), -(kTwo23 + 524288.f)));
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const float4 xl = *reinterpret_cast<const float4 *>(xs_b[t] + xs_chunk(b, i));       // elements 4i..4i+3
            const float4 xh = *reinterpret_cast<const float4 *>(xs_b[t] + xs_chunk(b, i + 4));   // elements 16+4i..
            acc[t] = f2fma(d0, make_float2(xl.x, xh.x), acc[t]);
            acc[t] = f2fma(d1, make_float2(xl.y, xh.y), acc[t]);
            acc[t] = f2fma(d2, make_float2(xl.z, xh.z), acc[t]);
            acc[t] = f2fma(d3, make_float2(xl.w, xh.w), acc[t]);
        }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) part[t] = acc[t].x + acc[t].y;
}

// Partial sums of one Q8_0 block (32 int8 in two uint4).
template <int NT>
__device__ __forceinline__ void q8_block(const uint4 w0, const uint4 w1, const float *xs_b[NT], int b,
                                         float part[NT]) {
    const uint32_t ws[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
    float2 acc[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t] = make_float2(0.f, 0.f);
    const float2 off = make_float2(-(kTwo23 + 128.f), -(kTwo23 + 128.f));
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t u = ws[i] ^ 0x80808080u;   // int8 q -> q + 128 in each byte
        const float2 da = f2add(make_float2(u2f(__byte_perm(u, kMagic, 0x7650u)),
                                            u2f(__byte_perm(u, kMagic, 0x7651u))), off);
        const float2 db = f2add(make_float2(u2f(__byte_perm(u, kMagic, 0x7652u)), u2f(__byte_perm(u, kMagic, 0x7653u))),
                                off);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const float4 x = *reinterpret_cast<const float4 *>(xs_b[t] + xs_chunk(b, i));
            acc[t] = f2fma(da, make_float2(x.x, x.y), acc[t]);
            acc[t] = f2fma(db, make_float2(x.z, x.w), acc[t]);
        }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) part[t] = acc[t].x + acc[t].y;
}

struct GemvParams {
    const uint8_t *qs;
    const __half *sc;
    int N, nb, K;
    int n_tasks;
    int T;
    GemvIn in;
};

// ROWS = 4: a quad of consecutive rows; ROWS = 8: the SwiGLU pair (gate quad, up quad).
template <int QT, int NT, int ROWS, int EPI, bool OUT16>
__global__ void __launch_bounds__(256, (NT > 2 ? 1 : 2)) k_gemv(const GemvParams p, const FwdArgs a, const int layer) {
    extern __shared__ __align__(16) float xs[];   // [NT][nb * 32] swizzled
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nb = p.nb, K = p.K;

    // ---- prologue: stage (normalised, position-scaled) activations
    __shared__ float red[8];
    for (int t = 0; t < NT; ++t) {
        float *xt = xs + (size_t)t * K;
        if (t >= p.T) {
            for (int k = threadIdx.x * 4; k < K; k += blockDim.x * 4) *reinterpret_cast<float4 *>(xt + k) = make_float4(0, 0, 0, 0);
            continue;
        }
        const float *xr = p.in.x + (size_t)(p.in.x_rows ? p.in.x_rows[t] : t) * K;
        float rs = 1.f;
        if (p.in.g) {
            float ss = 0.f;
            for (int k = threadIdx.x * 4; k < K; k += blockDim.x * 4) {
                const float4 v = *reinterpret_cast<const float4 *>(xr + k);
                ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
            }
            for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            __syncthreads();
            if (lane == 0) red[warp] = ss;
            __syncthreads();
            float tot = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) tot += red[w];
            rs = 1.0f / sqrtf(tot / (float)K + a.eps);
        }
        for (int k = threadIdx.x * 4; k < K; k += blockDim.x * 4) {
            float4 v = *reinterpret_cast<const float4 *>(xr + k);
            if (p.in.g) {
                const float4 g = *reinterpret_cast<const float4 *>(p.in.g + k);
                v.x = v.x * rs * g.x; v.y = v.y * rs * g.y; v.z = v.z * rs * g.z; v.w = v.w * rs * g.w;
            }
            const int b = k >> 5, j = (k & 31) >> 2;   // chunk j of block b: elements 4j..4j+3
            if (QT == Q4) {
                // element e = 4j + c: e < 16 -> byte e low nibble; else byte e-16 high nibble
                const int hi = j >= 4;
                v.x *= __int_as_float((127 - q4_shift(0, hi)) << 23);
                v.y *= __int_as_float((127 - q4_shift(1, hi)) << 23);
                v.z *= __int_as_float((127 - q4_shift(2, hi)) << 23);
                v.w *= __int_as_float((127 - q4_shift(3, hi)) << 23);
            }
            *reinterpret_cast<float4 *>(xt + xs_chunk(b, j)) = v;
        }
    }
    __syncthreads();

    const float *xs_b[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) xs_b[t] = xs + (size_t)t * K;

    unsigned long long best[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) best[t] = 0ull;

    const int total_warps = gridDim.x * 8;
    for (int task = blockIdx.x * 8 + warp; task < p.n_tasks; task += total_warps) {
        int rbase[ROWS / 4];
        if (ROWS == 4) {
            rbase[0] = task * 4;
        } else {
            const int c = task / (kRowTile / 4), qq = task % (kRowTile / 4);
            rbase[0] = c * 2 * kRowTile + 4 * qq;
            rbase[ROWS / 4 - 1] = rbase[0] + kRowTile;
        }
        float acc[ROWS][NT];
#pragma unroll
        for (int r = 0; r < ROWS; ++r)
#pragma unroll
            for (int t = 0; t < NT; ++t) acc[r][t] = 0.f;

        // blocks in flight per lane: about 64 registers of weight data
        constexpr int WORDS = ROWS * (QT == Q8 ? 8 : 4) * NT;
        constexpr int U = WORDS <= 16 ? 4 : WORDS <= 32 ? 2 : 1;
        for (int b0 = lane; b0 < nb; b0 += 32 * U) {
            uint4 wq[U][ROWS][QT == Q8 ? 2 : 1];
            uint2 sq[U][ROWS / 4];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int b = b0 + 32 * u;
                if (b < nb) {
#pragma unroll
                    for (int r = 0; r < ROWS; ++r) {
                        const int row = rbase[r / 4] + (r & 3);
                        const uint4 *src = reinterpret_cast<const uint4 *>(p.qs + ((size_t)row * nb + b) * (QT == Q8 ? 32 : 16));
                        wq[u][r][0] = __ldg(src);
                        if (QT == Q8) wq[u][r][QT == Q8 ? 1 : 0] = __ldg(src + 1);
                    }
#pragma unroll
                    for (int g = 0; g < ROWS / 4; ++g)
                        sq[u][g] = __ldg(reinterpret_cast<const uint2 *>(p.sc + ((size_t)(rbase[g] >> 2) * nb + b) * 4));
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int b = b0 + 32 * u;
                if (b < nb) {
#pragma unroll
                    for (int r = 0; r < ROWS; ++r) {
                        float part[NT];
                        if (QT == Q4) q4_block<NT>(wq[u][r][0], xs_b, b, part);
                        else q8_block<NT>(wq[u][r][0], wq[u][r][QT == Q8 ? 1 : 0], xs_b, b, part);
                        const uint32_t sbits = (r & 2) ? sq[u][r / 4].y : sq[u][r / 4].x;
                        const float d = __half2float(__ushort_as_half((unsigned short)((r & 1) ? (sbits >> 16) : (sbits & 0xffffu))));
#pragma unroll
                        for (int t = 0; t < NT; ++t) acc[r][t] = fmaf(d, part[t], acc[r][t]);
                    }
                }
            }
        }
        // reduce across lanes
#pragma unroll
        for (int r = 0; r < ROWS; ++r)
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                float v = acc[r][t];
#pragma unroll
                for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                acc[r][t] = v;
            }
        if (lane < NT && lane < p.T) {
            const int t = lane;
            float v0[4], v1[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                // select acc[.][t] with a static index
                float s0 = 0.f, s1 = 0.f;
#pragma unroll
                for (int tt = 0; tt < NT; ++tt)
                    if (tt == t) { s0 = acc[j][tt]; s1 = acc[(ROWS == 8 ? 4 : 0) + j][tt]; }
                v0[j] = s0;
                v1[j] = s1;
            }
            if (ROWS == 8) {
                const int c = task / (kRowTile / 4), qq = task % (kRowTile / 4);
                epi_swiglu<OUT16>(a, t, c * kRowTile + 4 * qq, v0, v1);
            } else {
                unsigned long long bk = 0ull;
                epi_quad<EPI>(a, layer, t, rbase[0], p.N, v0, bk);
#pragma unroll
                for (int tt = 0; tt < NT; ++tt)
                    if (tt == t) best[tt] = bk > best[tt] ? bk : best[tt];
            }
        }
    }
    if (EPI == EPI_LOGITS) {
        __shared__ unsigned long long cbest[NT];
        __syncthreads();
        if (threadIdx.x < NT) cbest[threadIdx.x] = 0ull;
        __syncthreads();
        if (lane < NT && lane < p.T) {
#pragma unroll
            for (int tt = 0; tt < NT; ++tt)
                if (tt == lane && best[tt]) atomicMax(&cbest[tt], best[tt]);
        }
        __syncthreads();
        if (threadIdx.x < NT && threadIdx.x < p.T && cbest[threadIdx.x]) atomicMax(&a.amax_key[threadIdx.x], cbest[threadIdx.x]);
    }
}

template <int QT, int NT, int ROWS, int EPI, bool OUT16>
cudaError_t run(const GemvParams &p, const FwdArgs &a, int layer, cudaStream_t s) {
    auto kern = k_gemv<QT, NT, ROWS, EPI, OUT16>;
    const size_t smem = (size_t)NT * p.K * sizeof(float);
    static int configured_smem = 0;   // per instantiation
    if ((int)smem > configured_smem) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGemvSmemX + 1024);
        if (e != cudaSuccess) return e;
        configured_smem = kGemvSmemX + 1024;
    }
    static int n_sm = 0;
    if (!n_sm) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
    }
    int occ = 1;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, 256, smem);
    if (occ < 1) occ = 1;
    int grid = (p.n_tasks + 7) / 8;
    grid = grid < n_sm * occ ? grid : n_sm * occ;
    if (grid < 1) grid = 1;
    kern<<<grid, 256, smem, s>>>(p, a, layer);
    return cudaGetLastError();
}

}  // namespace gemv_detail
}  // namespace lcx
