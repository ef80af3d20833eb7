// Small kernels of the forward: weight re-layout, RoPE table, token-embedding gather,
// RMSNorm to f16 (tensor-core path), argmax finalisation, row gather.
#include "lcx_internal.h"

namespace lcx {

// ------------------------------------------------------------------ stored-block reads
__device__ __forceinline__ float half_bits_to_float(uint16_t b) { return __half2float(__ushort_as_half(b)); }

// value of element i of a stored row (F16, Q8_0 or Q4_0); exact in f32 for every type
__device__ __forceinline__ float stored_elem(int type, const uint8_t *row, int64_t i) {
    if (type == QF16) {
        const uint8_t *p = row + 2 * i;
        return half_bits_to_float((uint16_t)(p[0] | (p[1] << 8)));
    }
    int64_t b = i >> 5;
    int e = (int)(i & 31);
    if (type == Q8) {
        const uint8_t *blk = row + b * 34;
        float d = half_bits_to_float((uint16_t)(blk[0] | (blk[1] << 8)));
        return d * (float)(int8_t)blk[2 + e];
    }
    const uint8_t *blk = row + b * 18;
    float d = half_bits_to_float((uint16_t)(blk[0] | (blk[1] << 8)));
    int q = e < 16 ? (blk[2 + e] & 15) : (blk[2 + e - 16] >> 4);
    return d * (float)(q - 8);
}

__host__ __device__ inline int64_t stored_row_bytes(int type, int64_t k) {
    return type == QF16 ? 2 * k : ((k + 31) / 32) * (type == Q8 ? 34 : 18);
}

// ------------------------------------------------------------------ repack
// One thread per (source row, block): copies the block's quant bytes and its scale to the
// destination row's place in the quad-interleaved storage (QMat). With `gateup`, source row r
// of the gate (row_offset 0) or up (row_offset 4) matrix goes to row 8 (r / 4) + row_offset + r % 4:
// the gate and up rows of features 4f..4f+3 form the consecutive quads 2f, 2f+1.
__global__ void k_repack(const uint8_t *__restrict__ src, int type, int N_src, int nb_src, uint8_t *__restrict__ w,
                         int nb_dst, int row_offset, int gateup) {
    int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (int64_t)N_src * nb_src) return;
    int r = (int)(idx / nb_src), b = (int)(idx % nb_src);
    int dr = gateup ? 8 * (r / 4) + row_offset + (r % 4) : r + row_offset;
    const int bb = type == Q8 ? 34 : 18, qb = type == Q8 ? 32 : 16;
    const size_t quad = (size_t)(dr >> 2) * (size_t)(nb_dst / 2) * pair_bytes_of(qb);
    const uint8_t *blk = src + ((int64_t)r * nb_src + b) * bb;
    uint8_t *dq = w + quad + quad_q_off(qb, dr & 3, b);
    for (int i = 0; i < qb; ++i) dq[i] = blk[2 + i];
    uint8_t *ds = w + quad + quad_s_off(qb, b) + 2 * (dr & 3);
    ds[0] = blk[0];
    ds[1] = blk[1];
}

cudaError_t launch_repack(const void *src, int type, int N_src, int nb_src, QMat &dst, int row_offset, int gateup,
                          cudaStream_t s) {
    int64_t n = (int64_t)N_src * nb_src;
    int threads = 256;
    int64_t blocks = (n + threads - 1) / threads;
    k_repack<<<(unsigned)blocks, threads, 0, s>>>((const uint8_t *)src, type, N_src, nb_src, dst.w, dst.nb, row_offset,
                                                 gateup);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ RoPE table
// tab[p][i] = (cos, sin)(p * theta^(-2i/hd)), evaluated in double and rounded to float.
__global__ void k_rope_table(float2 *tab, int n_pos, int hd, double theta) {
    int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    int half_hd = hd / 2;
    if (idx >= (int64_t)n_pos * half_hd) return;
    int p = (int)(idx / half_hd), i = (int)(idx % half_hd);
    double freq = pow(theta, -2.0 * (double)i / (double)hd);
    double sn, cs;
    sincos((double)p * freq, &sn, &cs);
    tab[idx] = make_float2((float)cs, (float)sn);
}

cudaError_t launch_rope_table(float2 *tab, int n_pos, int hd, double theta, cudaStream_t s) {
    int64_t n = (int64_t)n_pos * (hd / 2);
    k_rope_table<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(tab, n_pos, hd, theta);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ embedding gather
// Block t: x[t][:] = dequant(tok_embd[token t]). Block 0 also applies the ubatch's page-table
// updates and clears the argmax keys of its output rows (both are read only by later kernels).
__global__ void k_embed(const uint8_t *__restrict__ table, int type, int d, const int32_t *__restrict__ tok, float *x,
                        const int32_t *__restrict__ pt_upd, int n_upd, int32_t *pt, unsigned long long *keys,
                        int n_out) {
    LCX_PDL_WAIT();
    LCX_PDL_TRIGGER();
    const int t = blockIdx.x;
    const int id = tok[t];
    const uint8_t *row = table + (int64_t)id * stored_row_bytes(type, d);
    for (int i = threadIdx.x; i < d; i += blockDim.x) x[(int64_t)t * d + i] = stored_elem(type, row, i);
    if (t == 0) {
        for (int u = threadIdx.x; u < n_upd; u += blockDim.x) pt[pt_upd[2 * u]] = pt_upd[2 * u + 1];
        for (int r = threadIdx.x; r < n_out; r += blockDim.x) keys[r] = 0ull;
    }
}

cudaError_t launch_embed(const FwdArgs &a, int t_embd, const void *tok_embd, cudaStream_t s, int64_t &launches) {
    ++launches;
    return launch_pdl(k_embed, dim3(a.T), dim3(256), 0, s, (const uint8_t *)tok_embd, t_embd, a.d, a.tok_src, a.x,
                      a.ub.pt_upd, a.ub.n_upd, a.pt, a.amax_key, a.n_out);
}

__global__ void k_get_rows(const uint8_t *__restrict__ table, int type, int64_t n_cols, const int32_t *__restrict__ ids,
                           float *__restrict__ out) {
    const int i = blockIdx.x;
    const uint8_t *row = table + (int64_t)ids[i] * stored_row_bytes(type, n_cols);
    for (int64_t c = threadIdx.x; c < n_cols; c += blockDim.x) out[(int64_t)i * n_cols + c] = stored_elem(type, row, c);
}

cudaError_t launch_get_rows(int type, const void *table, int64_t n_cols, const int32_t *ids, int n, float *out,
                            cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    k_get_rows<<<n, 256, 0, s>>>((const uint8_t *)table, type, n_cols, ids, out);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ RMSNorm -> f16
// out[r][:] = f16(x[row r] / sqrt(mean(x^2) + eps) * g) and out_lo[r][:] the f16 rounding of the
// rest (about 22 bits together); row r of x is rows[r] (or r).
__global__ void k_rmsnorm_h(const float *__restrict__ x, const int32_t *__restrict__ rows, int d,
                            const float *__restrict__ g, float eps, __half *__restrict__ out, __half *__restrict__ out_lo) {
    LCX_PDL_WAIT();
    LCX_PDL_TRIGGER();
    const int r = blockIdx.x;
    const float *xr = x + (int64_t)(rows ? rows[r] : r) * d;
    // the row's first NV x 4 x blockDim values stay in registers between the two passes (the
    // whole row for d <= 4096 with 256 threads); a longer row's rest is read twice
    constexpr int NV = 4;
    float4 v[NV];
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int i = (threadIdx.x + k * blockDim.x) * 4;
        v[k] = i < d ? *reinterpret_cast<const float4 *>(xr + i) : make_float4(0.f, 0.f, 0.f, 0.f);
        ss += v[k].x * v[k].x + v[k].y * v[k].y + v[k].z * v[k].z + v[k].w * v[k].w;
    }
    for (int i = (threadIdx.x + NV * blockDim.x) * 4; i < d; i += blockDim.x * 4) {
        const float4 u = *reinterpret_cast<const float4 *>(xr + i);
        ss += u.x * u.x + u.y * u.y + u.z * u.z + u.w * u.w;
    }
    __shared__ float red[32];
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x < 32) {
        float w = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
        for (int o = 16; o; o >>= 1) w += __shfl_xor_sync(0xffffffffu, w, o);
        if (threadIdx.x == 0) red[0] = w;
    }
    __syncthreads();
    const float rs = 1.0f / sqrtf(red[0] / (float)d + eps);
    // 4 values as f16 high + low parts, one 8-byte store each (a warp writes 256 contiguous bytes)
    auto emit = [&](int i, const float4 u) {
        const float4 gg = *reinterpret_cast<const float4 *>(g + i);
        const float y0 = u.x * rs * gg.x, y1 = u.y * rs * gg.y, y2 = u.z * rs * gg.z, y3 = u.w * rs * gg.w;
        const __half2 h01 = __floats2half2_rn(y0, y1), h23 = __floats2half2_rn(y2, y3);
        const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
        const __half2 l01 = __floats2half2_rn(y0 - f01.x, y1 - f01.y), l23 = __floats2half2_rn(y2 - f23.x, y3 - f23.y);
        const size_t o = (size_t)r * d + i;
        *reinterpret_cast<uint2 *>(out + o) =
            make_uint2(*reinterpret_cast<const uint32_t *>(&h01), *reinterpret_cast<const uint32_t *>(&h23));
        *reinterpret_cast<uint2 *>(out_lo + o) =
            make_uint2(*reinterpret_cast<const uint32_t *>(&l01), *reinterpret_cast<const uint32_t *>(&l23));
    };
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int i = (threadIdx.x + k * blockDim.x) * 4;
        if (i < d) emit(i, v[k]);
    }
    for (int i = (threadIdx.x + NV * blockDim.x) * 4; i < d; i += blockDim.x * 4)
        emit(i, *reinterpret_cast<const float4 *>(xr + i));
}

cudaError_t launch_rmsnorm_h(const float *x, const int32_t *rows, int T, int d, const float *g, float eps,
                             __half *out, __half *out_lo, cudaStream_t s, int64_t &launches) {
    ++launches;
    return launch_pdl(k_rmsnorm_h, dim3(T), dim3(256), 0, s, x, rows, d, g, eps, out, out_lo);
}

// ------------------------------------------------------------------ argmax
// keys hold (ordered float bits << 32) | (0xffffffff - index): the max key is the largest
// logit, ties to the lowest index.
__global__ void k_argmax_final(const unsigned long long *__restrict__ keys, int n, int32_t *__restrict__ dst) {
    LCX_PDL_WAIT();
    LCX_PDL_TRIGGER();
    int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) dst[i] = (int32_t)(0xffffffffu - (uint32_t)(keys[i] & 0xffffffffull));
}

cudaError_t launch_argmax_final(const FwdArgs &a, int32_t *dst, cudaStream_t s, int64_t &launches) {
    if (a.n_out <= 0) return cudaSuccess;
    ++launches;
    return launch_pdl(k_argmax_final, dim3((a.n_out + 127) / 128), dim3(128), 0, s,
                      (const unsigned long long *)a.amax_key, a.n_out, dst);
}

}  // namespace lcx
