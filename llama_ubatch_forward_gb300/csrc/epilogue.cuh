// Epilogues shared by the weight-streaming GEMV and the tensor-core GEMM.
//
// A "quad" is 4 consecutive internal rows (outputs) of one token. The QKV epilogue applies
// RoPE to adjacent pairs (2i, 2i+1) of Q and K -- the rotation of the article's per-layer
// graph, read as the "normal" (adjacent-pair) llama mode -- and appends K and V to the cache
// as f16 (KV-cache section: the new token's K/V are stored before attention reads them).
#pragma once
#include "lcx_internal.h"

namespace lcx {

__device__ __forceinline__ unsigned long long argmax_key(float v, int idx) {
    uint32_t b = __float_as_uint(v);
    b = (b & 0x80000000u) ? ~b : (b | 0x80000000u);   // order-preserving map of float bits
    return ((unsigned long long)b << 32) | (unsigned long long)(0xffffffffu - (uint32_t)idx);
}

// A logit that is not finite fails its ubatch (step 13: a failed compute returns -3 and the
// ubatch's cells are removed again). The first ubatch (or greedy step) of the call to produce one
// leaves its tag (index + 1) in the context's non-finite word; the host reads it after the call.
__device__ __forceinline__ void note_nonfinite(const FwdArgs &a) { atomicCAS(a.nonfinite, 0, a.tag); }

// SiLU with the fast exponential and division (relative error about 1e-6; the exponential
// saturates to inf for very negative g, where the quotient is then 0)
__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// cache address of (layer, cell, kv head, dim) in [L][n_pages][KV][kPage][hd]
__device__ __forceinline__ size_t kv_off(const FwdArgs &a, int layer, int cell, int kvh, int dim) {
    int page = cell / kPage, slot = cell % kPage;
    return ((((size_t)layer * a.n_pages + page) * a.KV + kvh) * kPage + slot) * a.hd + dim;
}

// Operands an epilogue reads from memory, loaded ahead of the dot products that feed it: the
// residual rows (through L2: other CTAs of the same launch may have written them), or the
// token's cache cell and the RoPE (cos, sin) pairs of the quad.
struct EpiIn {
    float4 x;
    float4 cs;     // (cos, sin) of pair r0 / 2 and of pair r0 / 2 + 1 within the head
    int cell;
};

template <int EPI>
__device__ __forceinline__ EpiIn epi_load(const FwdArgs &a, int t, int r0, int N) {
    EpiIn in{};
    if (EPI == EPI_RESID) {
        const float *xr = a.x + (size_t)t * a.d + r0;
        if (r0 + 3 < N) {
            in.x = __ldcg(reinterpret_cast<const float4 *>(xr));
        } else {
            in.x.x = r0 < N ? __ldcg(xr) : 0.f;
            in.x.y = r0 + 1 < N ? __ldcg(xr + 1) : 0.f;
            in.x.z = r0 + 2 < N ? __ldcg(xr + 2) : 0.f;
        }
    } else if (EPI == EPI_QKV) {
        const int qw = a.H * a.hd, kw = a.KV * a.hd;
        in.cell = a.ub.cell[t];
        if (r0 < qw + kw) {   // q or k rows: the quad lies inside one head (hd % 4 == 0)
            const int dim = (r0 < qw ? r0 : r0 - qw) & (a.hd - 1);   // hd is 64 or 128
            in.cs = *reinterpret_cast<const float4 *>(a.rope + (size_t)a.ub.pos[t] * (a.hd / 2) + dim / 2);
        }
    }
    return in;
}

// Epilogue of 4 consecutive rows r0..r0+3 (r0 % 4 == 0) of token t, with its operands loaded.
template <int EPI>
__device__ __forceinline__ void epi_quad_in(const FwdArgs &a, int layer, int t, int r0, int N, const float v[4],
                                            const EpiIn &in, unsigned long long &best) {
    if (EPI == EPI_RESID) {
        float *xr = a.x + (size_t)t * a.d;
        const float xo[4] = {in.x.x, in.x.y, in.x.z, in.x.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (r0 + j < N) xr[r0 + j] = xo[j] + v[j];
    } else if (EPI == EPI_LOGITS) {
        float *lr = a.logits + (size_t)t * a.V;
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (r0 + j < N) {
                lr[r0 + j] = v[j];
                unsigned long long k = argmax_key(v[j], r0 + j);
                best = k > best ? k : best;
                if (!isfinite(v[j])) note_nonfinite(a);
            }
    } else if (EPI == EPI_QKV) {
        const int qw = a.H * a.hd, kw = a.KV * a.hd;
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            const int r = r0 + 2 * p;
            if (r >= qw + 2 * kw) break;
            float y0 = v[2 * p], y1 = v[2 * p + 1];
            if (r < qw + kw) {   // q or k: rotate the pair
                const float c = p ? in.cs.z : in.cs.x, sn = p ? in.cs.w : in.cs.y;
                const float z0 = y0 * c - y1 * sn, z1 = y0 * sn + y1 * c;
                y0 = z0;
                y1 = z1;
            }
            if (r < qw) {
                float *qr = a.q + (size_t)t * qw + r;
                qr[0] = y0;
                qr[1] = y1;
            } else {
                const bool isk = r < qw + kw;
                const int rr = isk ? r - qw : r - qw - kw;
                const int sh = __ffs(a.hd) - 1;   // hd is a power of two
                const int kvh = rr >> sh, dim = rr & (a.hd - 1);
                __half *dst = (isk ? a.kc : a.vc) + kv_off(a, layer, in.cell, kvh, dim);
                *reinterpret_cast<__half2 *>(dst) = __floats2half2_rn(y0, y1);
            }
        }
    }
}

// Epilogue of 4 consecutive rows r0..r0+3 (r0 % 4 == 0) of token t.
template <int EPI>
__device__ __forceinline__ void epi_quad(const FwdArgs &a, int layer, int t, int r0, int N, const float v[4],
                                         unsigned long long &best) {
    epi_quad_in<EPI>(a, layer, t, r0, N, v, epi_load<EPI>(a, t, r0, N), best);
}

// SwiGLU epilogue: features f0..f0+3 of token t from gate g[4] and up u[4].
template <bool OUT16>
__device__ __forceinline__ void epi_swiglu(const FwdArgs &a, int t, int f0, const float g[4], const float u[4]) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int f = f0 + j;
        if (f >= a.F) break;
        const float h = silu_f(g[j]) * u[j];
        if (OUT16) store_split(a.h16, a.h16_lo, (size_t)t * a.F_pad + f, h);
        else a.h32[(size_t)t * a.F_pad + f] = h;
    }
}

// SwiGLU epilogue for two features f0, f0+1.
template <bool OUT16>
__device__ __forceinline__ void epi_swiglu2(const FwdArgs &a, int t, int f0, const float g[2], const float u[2]) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int f = f0 + j;
        if (f >= a.F) break;
        const float h = silu_f(g[j]) * u[j];
        if (OUT16) store_split(a.h16, a.h16_lo, (size_t)t * a.F_pad + f, h);
        else a.h32[(size_t)t * a.F_pad + f] = h;
    }
}

}  // namespace lcx
