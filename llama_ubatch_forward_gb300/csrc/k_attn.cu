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

// 2^x by the hardware approximation (relative error about 2^-22; results below 2^-126 flush to 0)
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <int HD, int G, bool OUT16>
__global__ void __launch_bounds__(128) k_attn(const FwdArgs a, const int layer, const int chunk, const int n_split) {
    constexpr int DPL = HD / 8;    // dims per lane in Q.K (8 lanes per cell)
    constexpr int DPV = HD / 32;   // dims per lane in P.V
    const int t = blockIdx.z, kvh = blockIdx.y, sp = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    LCX_TRACE(a, 0);
    // The ubatch metadata, the page table and the cells of positions <= pos - T (stored by earlier
    // ubatches) do not depend on the preceding kernel, which writes q and this ubatch's cells: each
    // warp loads its first 16 cells into registers before waiting for that kernel, and re-reads
    // afterwards only the cells this ubatch may have written.
    const int pos = a.ub.pos[t], seq = a.ub.seq[t];
    const int n_att = pos + 1;
    const int ns_t = (n_att + chunk - 1) / chunk;
    const int c0 = sp * chunk, c1 = min(c0 + chunk, n_att);
    const int sub = lane & 7, cgrp = lane >> 3;
    const int32_t *ptrow = a.pt + (size_t)seq * a.max_pages_per_seq;
    const size_t layer_base = (size_t)layer * a.n_pages;
    const int fresh = n_att - a.T;   // cells at positions >= fresh may come from this ubatch
    // two buffers of one super-group's K/V each: the next super-group's loads are in flight while
    // the current one is used
    uint4 kA[4][DPL / 8], kB[4][DPL / 8];
    uint2 vA[16], vB[16];
    // K/V of the super-group of 16 cells at j0 (inside one page) into (kraw, vraw); `only_fresh`
    // re-reads just the cells this ubatch may have written
    auto load_sg = [&](int j0, bool only_fresh, uint4 (&kraw)[4][DPL / 8], uint2 (&vraw)[16]) {
        const int page = ptrow[j0 / kPage];
        const size_t row0 = ((layer_base + page) * a.KV + kvh) * kPage + (j0 % kPage);
#pragma unroll
        for (int g4 = 0; g4 < 4; ++g4) {
            const int j = j0 + 4 * g4 + cgrp;
            if (only_fresh && (j < fresh || j >= c1)) continue;
            if (j < c1) {
                const __half *kp = a.kc + (row0 + 4 * g4 + cgrp) * HD + sub * DPL;
#pragma unroll
                for (int i = 0; i < DPL / 8; ++i) kraw[g4][i] = *reinterpret_cast<const uint4 *>(kp + 8 * i);
            } else {
#pragma unroll
                for (int i = 0; i < DPL / 8; ++i) kraw[g4][i] = make_uint4(0, 0, 0, 0);
            }
        }
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            const int j = j0 + c;
            if (only_fresh && j < fresh) continue;
            if (j < c1) {
                const __half *vp = a.vc + (row0 + c) * HD + lane * DPV;
                if (DPV == 4) vraw[c] = *reinterpret_cast<const uint2 *>(vp);
                else vraw[c] = make_uint2(*reinterpret_cast<const uint32_t *>(vp), 0u);
            }
        }
    };
    const int j_first = c0 + warp * 16;
    if (sp < ns_t && j_first < c1) load_sg(j_first, false, kA, vA);
    LCX_PDL_WAIT();
    LCX_PDL_TRIGGER();
    LCX_TRACE(a, 1);
    if (sp >= ns_t) return;
    if (j_first < c1 && j_first + 16 > fresh) load_sg(j_first, true, kA, vA);
    const int qw = a.H * HD;
    const float scale = rsqrtf((float)HD) * 1.4426950408889634f;   // scores in the log2 domain

    // this lane's Q slice for the QK step: dims (lane % 8) * DPL .. + DPL, pre-scaled
    float qr[G][DPL];
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

    // Each warp takes super-groups of 16 consecutive cells (inside one 64-cell page): all K and
    // V loads of a super-group are issued before any of them is used, one super-group ahead. The
    // 16 cells' scores are computed first and take one online-softmax step together (one
    // maximum, one rescaling of the accumulators), in the log2 domain (q carries log2(e)).
    auto consume = [&](int j0, const uint4 (&kraw)[4][DPL / 8], const uint2 (&vraw)[16]) {
        float s[4][G];   // cell j0 + 4 g4 + cgrp, query head g (every lane of the cell holds it)
#pragma unroll
        for (int g4 = 0; g4 < 4; ++g4) {
            const bool valid = j0 + 4 * g4 + cgrp < c1;
            float kf[DPL];
#pragma unroll
            for (int i = 0; i < DPL / 8; ++i) {
                const __half2 *h2 = reinterpret_cast<const __half2 *>(&kraw[g4][i]);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = __half22float2(h2[e]);
                    kf[8 * i + 2 * e] = f.x;
                    kf[8 * i + 2 * e + 1] = f.y;
                }
            }
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float d = 0.f;
#pragma unroll
                for (int i = 0; i < DPL; ++i) d = fmaf(qr[g][i], kf[i], d);
                d += __shfl_xor_sync(0xffffffffu, d, 1);
                d += __shfl_xor_sync(0xffffffffu, d, 2);
                d += __shfl_xor_sync(0xffffffffu, d, 4);
                s[g4][g] = valid ? d : -CUDART_INF_F;
            }
        }
        // one online-softmax step over the 16 cells (cell j0 is always valid: m stays finite)
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float mx = fmaxf(fmaxf(s[0][g], s[1][g]), fmaxf(s[2][g], s[3][g]));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float mn = fmaxf(m[g], mx);
            const float alpha = ex2_approx(m[g] - mn);
            float ps = 0.f;
#pragma unroll
            for (int g4 = 0; g4 < 4; ++g4) {
                s[g4][g] = ex2_approx(s[g4][g] - mn);   // now the weight p of the cell
                ps += s[g4][g];
            }
            ps += __shfl_xor_sync(0xffffffffu, ps, 8);
            ps += __shfl_xor_sync(0xffffffffu, ps, 16);
            l[g] = l[g] * alpha + ps;   // lanes l, l^8, l^16, l^24 hold the group's 4 cells
            m[g] = mn;
#pragma unroll
            for (int i = 0; i < DPV; ++i) acc[g][i] *= alpha;
        }
        // P.V: lane owns dims lane * DPV .. + DPV
#pragma unroll
        for (int g4 = 0; g4 < 4; ++g4) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if (j0 + 4 * g4 + c >= c1) break;
                const uint2 raw = vraw[4 * g4 + c];
                float vf[DPV];
                const float2 f0 = __half22float2(*reinterpret_cast<const __half2 *>(&raw.x));
                vf[0] = f0.x;
                vf[1 % DPV] = f0.y;
                if (DPV == 4) {
                    const float2 f1 = __half22float2(*reinterpret_cast<const __half2 *>(&raw.y));
                    vf[2 % DPV] = f1.x;
                    vf[3 % DPV] = f1.y;
                }
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float pc = __shfl_sync(0xffffffffu, s[g4][g], 8 * c);
#pragma unroll
                    for (int i = 0; i < DPV; ++i) acc[g][i] = fmaf(pc, vf[i], acc[g][i]);
                }
            }
        }
    };
    for (int j0 = j_first; j0 < c1; j0 += 128) {
        if (j0 + 64 < c1) load_sg(j0 + 64, false, kB, vB);
        consume(j0, kA, vA);
        if (j0 + 64 >= c1) break;
        if (j0 + 128 < c1) load_sg(j0 + 128, false, kA, vA);
        consume(j0 + 64, kB, vB);
    }

    LCX_TRACE(a, 2);
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
            const float f = sm_m[w][g] == -CUDART_INF_F ? 0.f : exp2f(sm_m[w][g] - M);
            L += sm_l[w][g] * f;
            A += sm_acc[w][g][dd] * f;
        }
        if (single) {
            const float o = A / L;
            const size_t oi = (size_t)t * qw + (size_t)(kvh * G + g) * HD + dd;
            if (OUT16) store_split(a.o16, a.o16_lo, oi, o);
            else a.o32[oi] = o;
        } else {
            float *pr = part + ((prow + sp) * G + g) * (HD + 2);
            pr[2 + dd] = A;
            if (dd == 0) { pr[0] = M; pr[1] = L; }
        }
    }
    if (single) {
        LCX_TRACE(a, 3);
        return;
    }

    // ---- split merge by the last CTA to arrive
    __shared__ int last;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const int prev = atomicAdd(&a.att_cnt[t * a.KV + kvh], 1);
        last = prev == ns_t - 1;
    }
    __syncthreads();
    if (!last) {
        LCX_TRACE(a, 3);
        return;
    }
    __threadfence();
    // merge weights of the splits: w_s = 2^(M_s - M*) / L*, one warp per query head
    __shared__ float sw[64][G];
    for (int g = warp; g < G; g += 4) {
        float ms[2], ls[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int s2 = lane + 32 * h;
            const float *pr = part + ((prow + s2) * G + g) * (HD + 2);
            ms[h] = s2 < ns_t ? __ldcg(pr) : -CUDART_INF_F;
            ls[h] = s2 < ns_t ? __ldcg(pr + 1) : 0.f;
        }
        float M = fmaxf(ms[0], ms[1]);
#pragma unroll
        for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        float e[2], L = 0.f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            e[h] = lane + 32 * h < ns_t ? exp2f(ms[h] - M) : 0.f;
            L += e[h] * ls[h];
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
#pragma unroll
        for (int h = 0; h < 2; ++h)
            if (lane + 32 * h < ns_t) sw[lane + 32 * h][g] = e[h] / L;
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < G * HD; idx += blockDim.x) {
        const int g = idx / HD, dd = idx % HD;
        float o = 0.f;
        int s2 = 0;
        for (; s2 + 8 <= ns_t; s2 += 8) {   // 8 independent loads in flight
            float v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = __ldcg(part + ((prow + s2 + u) * G + g) * (HD + 2) + 2 + dd);
#pragma unroll
            for (int u = 0; u < 8; ++u) o = fmaf(sw[s2 + u][g], v[u], o);
        }
        for (; s2 < ns_t; ++s2) o = fmaf(sw[s2][g], __ldcg(part + ((prow + s2) * G + g) * (HD + 2) + 2 + dd), o);
        const size_t oi = (size_t)t * qw + (size_t)(kvh * G + g) * HD + dd;
        if (OUT16) store_split(a.o16, a.o16_lo, oi, o);
        else a.o32[oi] = o;
    }
    if (threadIdx.x == 0) a.att_cnt[t * a.KV + kvh] = 0;
    LCX_TRACE(a, 3);
}

template <int HD, int G>
cudaError_t run(const FwdArgs &a, int layer, int chunk, int ns, bool out16, cudaStream_t s) {
    dim3 grid(ns, a.KV, a.T);
    if (!a.pdl) {   // stand-alone call: fully ordered after the caller's preceding work
        if (out16) k_attn<HD, G, true><<<grid, 128, 0, s>>>(a, layer, chunk, ns);
        else k_attn<HD, G, false><<<grid, 128, 0, s>>>(a, layer, chunk, ns);
        return cudaGetLastError();
    }
    if (out16) return launch_pdl(k_attn<HD, G, true>, grid, dim3(128), 0, s, a, layer, chunk, ns);
    return launch_pdl(k_attn<HD, G, false>, grid, dim3(128), 0, s, a, layer, chunk, ns);
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
    const int n_sm = device_sm_count();
    // one CTA per SM: the next kernel's CTAs (started early, waiting for this one) leave room for
    // about one attention CTA per SM, so a second wave would double the latency
    const int target = n_sm;
    const int units = a.T * a.KV;
    int ns = units >= target ? 1 : (target + units - 1) / units;
    // inside the forward, no CTA walks more than att_max_chunk cells: with many units (a ubatch of
    // one token per sequence over long contexts) one CTA per unit would leave the longest context's
    // CTAs running alone at the end
    if (a.att_max_chunk > 0) ns = max(ns, (max_natt + a.att_max_chunk - 1) / a.att_max_chunk);
    int by_len = (max_natt + 63) / 64;
    ns = ns < by_len ? ns : by_len;
    ns = ns < a.att_max_split ? ns : a.att_max_split;
    if (a.att_rows_cap > 0) ns = min(ns, max(1, a.att_rows_cap / units));   // partial rows available
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
