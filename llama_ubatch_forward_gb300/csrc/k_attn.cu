// Causal grouped-query attention over the paged f16 KV cache (split-K "flash-decode").
//
// Each query token t (sequence s, position p) attends every cell of s with position <= p, its
// own K/V included (KV-cache section of the article: the new token's K and V are appended to
// the cache first, then Q attends all cached keys). One CTA handles one (token, KV head, split
// of the cell range) and all n_head / n_head_kv query heads that share that KV head, so each K
// and V row is read once for the whole group.
//
// Inside a CTA, 4 warps take interleaved groups of 4 cells; 8 lanes share a cell's K row for
// the Q.K dot products (reduced with shuffles), the scores go through an online softmax, and
// lanes own head_dim/32 output dims for the P.V accumulation. The CTA's 4 warp states are
// merged in shared memory. With several splits, every CTA writes its partial (max, sum, acc)
// and the last CTA of a (token, KV head) to arrive -- an arrival counter, no waiting -- merges
// the partials in split order and writes the output. The counter is reset by that CTA.
#include <math_constants.h>

#include "epilogue.cuh"

namespace lcx {

namespace {

template <int HD, int G, bool OUT16>
__global__ void __launch_bounds__(128) k_attn(const FwdArgs a, const int layer, const int chunk, const int n_split) {
    constexpr int DPL = HD / 8;    // dims per lane in Q.K (8 lanes per cell)
    constexpr int DPV = HD / 32;   // dims per lane in P.V
    const int t = blockIdx.z, kvh = blockIdx.y, sp = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int pos = a.ub.pos[t], seq = a.ub.seq[t];
    const int n_att = pos + 1;
    const int ns_t = (n_att + chunk - 1) / chunk;
    if (sp >= ns_t) return;
    const int c0 = sp * chunk, c1 = min(c0 + chunk, n_att);
    const int qw = a.H * HD;
    const float scale = rsqrtf((float)HD);

    // this lane's Q slice for the QK step: dims (lane % 8) * DPL .. + DPL, pre-scaled
    float qr[G][DPL];
    const int sub = lane & 7, cgrp = lane >> 3;
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const float *qp = a.q + (size_t)t * qw + (size_t)(kvh * G + g) * HD + sub * DPL;
#pragma unroll
        for (int i = 0; i < DPL; i += 4) {
            const float4 v = *reinterpret_cast<const float4 *>(qp + i);
            qr[g][i] = v.x * scale; qr[g][i + 1] = v.y * scale; qr[g][i + 2] = v.z * scale; qr[g][i + 3] = v.w * scale;
        }
    }
    float m[G], l[G], acc[G][DPV];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        m[g] = -CUDART_INF_F;
        l[g] = 0.f;
#pragma unroll
        for (int i = 0; i < DPV; ++i) acc[g][i] = 0.f;
    }
    const int32_t *ptrow = a.pt + (size_t)seq * a.max_pages_per_seq;
    const size_t layer_base = (size_t)layer * a.n_pages;

    for (int j0 = c0 + warp * 4; j0 < c1; j0 += 16) {
        const int j = j0 + cgrp;                 // this lane's cell in the group
        const bool valid = j < c1;
        float s[G];
        int cellrow = 0;
        if (valid) {
            const int page = ptrow[j / kPage];
            cellrow = (int)(((layer_base + page) * a.KV + kvh) * kPage + (j % kPage));
            const __half *kp = a.kc + (size_t)cellrow * HD + sub * DPL;
            float kf[DPL];
#pragma unroll
            for (int i = 0; i < DPL; i += 8) {
                const uint4 raw = *reinterpret_cast<const uint4 *>(kp + i);
                const __half2 *h2 = reinterpret_cast<const __half2 *>(&raw);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = __half22float2(h2[e]);
                    kf[i + 2 * e] = f.x;
                    kf[i + 2 * e + 1] = f.y;
                }
            }
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float d = 0.f;
#pragma unroll
                for (int i = 0; i < DPL; ++i) d = fmaf(qr[g][i], kf[i], d);
                s[g] = d;
            }
        } else {
#pragma unroll
            for (int g = 0; g < G; ++g) s[g] = 0.f;
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float d = s[g];
            d += __shfl_xor_sync(0xffffffffu, d, 1);
            d += __shfl_xor_sync(0xffffffffu, d, 2);
            d += __shfl_xor_sync(0xffffffffu, d, 4);
            s[g] = valid ? d : -CUDART_INF_F;
        }
        // online softmax over the 4 cells of the group
        float p[G], alpha[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float mx = s[g];
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float mn = fmaxf(m[g], mx);
            alpha[g] = expf(m[g] - mn);
            p[g] = expf(s[g] - mn);
            float ps = p[g];
            ps += __shfl_xor_sync(0xffffffffu, ps, 8);
            ps += __shfl_xor_sync(0xffffffffu, ps, 16);
            l[g] = l[g] * alpha[g] + ps;   // lanes l, l^8, l^16, l^24 hold the group's 4 cells
            m[g] = mn;
#pragma unroll
            for (int i = 0; i < DPV; ++i) acc[g][i] *= alpha[g];
        }
        // P.V: lane owns dims lane * DPV .. + DPV
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int cr = __shfl_sync(0xffffffffu, cellrow, 8 * c);
            if (j0 + c >= c1) break;
            float vf[DPV];
            const __half *vp = a.vc + (size_t)cr * HD + lane * DPV;
            if (DPV == 4) {
                const uint2 raw = *reinterpret_cast<const uint2 *>(vp);
                const float2 f0 = __half22float2(*reinterpret_cast<const __half2 *>(&raw.x));
                const float2 f1 = __half22float2(*reinterpret_cast<const __half2 *>(&raw.y));
                vf[0] = f0.x; vf[1 % DPV] = f0.y; vf[2 % DPV] = f1.x; vf[3 % DPV] = f1.y;
            } else {
                const float2 f0 = __half22float2(*reinterpret_cast<const __half2 *>(vp));
                vf[0] = f0.x; vf[1 % DPV] = f0.y;
            }
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float pc = __shfl_sync(0xffffffffu, p[g], 8 * c);
#pragma unroll
                for (int i = 0; i < DPV; ++i) acc[g][i] = fmaf(pc, vf[i], acc[g][i]);
            }
        }
    }

    // ---- merge the 4 warps
    __shared__ float sm_m[4][G], sm_l[4][G];
    __shared__ float sm_acc[4][G][HD];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        if (lane == 0) { sm_m[warp][g] = m[g]; sm_l[warp][g] = l[g]; }
#pragma unroll
        for (int i = 0; i < DPV; ++i) sm_acc[warp][g][lane * DPV + i] = acc[g][i];
    }
    __syncthreads();
    // thread -> (g, dim) pairs
    const bool single = ns_t == 1;
    float *part = a.att_part;
    const size_t prow = (size_t)(t * a.KV + kvh) * n_split;   // partial rows of this (token, kv head)
    for (int idx = threadIdx.x; idx < G * HD; idx += blockDim.x) {
        const int g = idx / HD, dd = idx % HD;
        float M = -CUDART_INF_F;
#pragma unroll
        for (int w = 0; w < 4; ++w) M = fmaxf(M, sm_m[w][g]);
        float L = 0.f, A = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const float f = sm_m[w][g] == -CUDART_INF_F ? 0.f : expf(sm_m[w][g] - M);
            L += sm_l[w][g] * f;
            A += sm_acc[w][g][dd] * f;
        }
        if (single) {
            const float o = A / L;
            const size_t oi = (size_t)t * qw + (size_t)(kvh * G + g) * HD + dd;
            if (OUT16) a.o16[oi] = __float2half_rn(o);
            else a.o32[oi] = o;
        } else {
            float *pr = part + ((prow + sp) * G + g) * (HD + 2);
            pr[2 + dd] = A;
            if (dd == 0) { pr[0] = M; pr[1] = L; }
        }
    }
    if (single) return;

    // ---- split merge by the last CTA to arrive
    __shared__ int last;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const int prev = atomicAdd(&a.att_cnt[t * a.KV + kvh], 1);
        last = prev == ns_t - 1;
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    for (int idx = threadIdx.x; idx < G * HD; idx += blockDim.x) {
        const int g = idx / HD, dd = idx % HD;
        float M = -CUDART_INF_F;
        for (int s2 = 0; s2 < ns_t; ++s2) M = fmaxf(M, __ldcg(part + ((prow + s2) * G + g) * (HD + 2)));
        float L = 0.f, A = 0.f;
        for (int s2 = 0; s2 < ns_t; ++s2) {
            const float *pr = part + ((prow + s2) * G + g) * (HD + 2);
            const float f = expf(__ldcg(pr) - M);
            L += __ldcg(pr + 1) * f;
            A += __ldcg(pr + 2 + dd) * f;
        }
        const float o = A / L;
        const size_t oi = (size_t)t * qw + (size_t)(kvh * G + g) * HD + dd;
        if (OUT16) a.o16[oi] = __float2half_rn(o);
        else a.o32[oi] = o;
    }
    if (threadIdx.x == 0) a.att_cnt[t * a.KV + kvh] = 0;
}

template <int HD, int G>
cudaError_t run(const FwdArgs &a, int layer, int chunk, int ns, bool out16, cudaStream_t s) {
    dim3 grid(ns, a.KV, a.T);
    if (out16) k_attn<HD, G, true><<<grid, 128, 0, s>>>(a, layer, chunk, ns);
    else k_attn<HD, G, false><<<grid, 128, 0, s>>>(a, layer, chunk, ns);
    return cudaGetLastError();
}

template <int HD>
cudaError_t run_g(const FwdArgs &a, int layer, int chunk, int ns, bool out16, cudaStream_t s) {
    switch (a.H / a.KV) {
        case 1: return run<HD, 1>(a, layer, chunk, ns, out16, s);
        case 2: return run<HD, 2>(a, layer, chunk, ns, out16, s);
        case 4: return run<HD, 4>(a, layer, chunk, ns, out16, s);
        case 8: return run<HD, 8>(a, layer, chunk, ns, out16, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

int attention_splits(const FwdArgs &a, int max_natt, int *chunk) {
    static int n_sm = 0;
    if (!n_sm) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
    }
    const int target = 4 * n_sm;
    const int units = a.T * a.KV;
    int ns = units >= target ? 1 : (target + units - 1) / units;
    int by_len = (max_natt + 63) / 64;
    ns = ns < by_len ? ns : by_len;
    ns = ns < a.att_max_split ? ns : a.att_max_split;
    if (ns < 1) ns = 1;
    int ch = (max_natt + ns - 1) / ns;
    ch = (ch + 15) / 16 * 16;
    ns = (max_natt + ch - 1) / ch;
    *chunk = ch;
    return ns;
}

size_t attention_scratch_bytes(const FwdArgs &a, int max_natt, size_t *counter_offset) {
    int chunk = 0;
    const int ns = attention_splits(a, max_natt, &chunk);
    if (ns <= 1) {
        if (counter_offset) *counter_offset = 0;
        return 0;
    }
    const size_t part = (size_t)a.T * a.KV * ns * (a.H / a.KV) * (a.hd + 2) * sizeof(float);
    const size_t off = (part + 255) / 256 * 256;
    if (counter_offset) *counter_offset = off;
    return off + (size_t)a.T * a.KV * sizeof(int32_t);
}

cudaError_t launch_attention(const FwdArgs &a, int layer, int max_natt, bool out_f16, cudaStream_t s,
                             int64_t &launches) {
    int chunk = 0;
    const int ns = attention_splits(a, max_natt, &chunk);
    ++launches;
    if (a.hd == 64) return run_g<64>(a, layer, chunk, ns, out_f16, s);
    if (a.hd == 128) return run_g<128>(a, layer, chunk, ns, out_f16, s);
    return cudaErrorInvalidValue;
}

}  // namespace lcx
