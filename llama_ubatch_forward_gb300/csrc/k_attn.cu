// Causal grouped-query attention over the paged f16 KV cache (split-K "flash-decode").
//
// Each query token t (sequence s, position p) attends every cell of s with position <= p, its
// own K/V included (KV-cache section of the article: the new token's K and V are appended to
// the cache first, then Q attends all cached keys). One CTA handles one (token, KV head, split
// of the cell range) and all n_head / n_head_kv query heads that share that KV head, so each K
// and V row is read once for the whole group.
//
// Inside a CTA, 4 warps take interleaved key tiles of 16 cells, staged by cp.async into a ring of
// three tiles per warp; the products run on the tensor cores (mma.sync m16n8k16, f16 in, f32
// accumulate) with the query heads as the MMA rows: S = Q K^T (q as f16 high + low parts, pre-
// scaled into the log2 domain), one online-softmax step per tile, O += P V (P as f16 high + low
// parts). The CTA's 4 warp states are merged in shared memory. With several splits, every CTA
// writes its partial (max, sum, acc) and the last CTA of a (token, KV head) to arrive -- an
// arrival counter, no waiting -- merges the partials in split order and writes the output. The
// counter is reset by that CTA.
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

// mma.sync m16n8k16 (f16 in, f32 accumulate) and its operand loads, as in the prefill kernel
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
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
// f16 high part of x and the f16 rounding of the rest, packed for two elements (x0 in the low half)
__device__ __forceinline__ void split2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    const __half2 h = __floats2half2_rn(x0, x1);
    const float2 hf = __half22float2(h);
    const __half2 l = __floats2half2_rn(x0 - hf.x, x1 - hf.y);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

constexpr int AT_CELLS = 16;   // cells of a key tile
constexpr int AT_STAGES = 3;   // key tiles in flight per warp

template <int HD>
constexpr int attn_smem_bytes() { return 4 /* warps */ * AT_STAGES * 2 * AT_CELLS * HD * 2; }

// byte offset of 16-byte chunk c of row r in a [16][HD] f16 tile, chunks XOR-swizzled by row
template <int HD>
__device__ __forceinline__ uint32_t at_off(int r, int c) {
    return (uint32_t)(r * HD * 2 + ((c ^ (r & 7)) << 4));
}

template <int HD, int G, bool OUT16>
__global__ void __launch_bounds__(128) k_attn(const FwdArgs a, const int layer, const int chunk, const int n_split) {
    constexpr int CH = HD / 8;                 // 16-byte chunks of a K or V row
    constexpr int TILE = AT_CELLS * HD * 2;    // bytes of a K or V tile
    const int t = blockIdx.z, kvh = blockIdx.y, sp = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, tq = lane & 3;    // fragment row (query head) and column pair
    LCX_TRACE(a, 0);
    const int pos = a.ub.pos[t], seq = a.ub.seq[t];
    const int n_att = pos + 1;
    const int ns_t = (n_att + chunk - 1) / chunk;
    const int c0 = sp * chunk, c1 = min(c0 + chunk, n_att);
    const int32_t *ptrow = a.pt + (size_t)seq * a.max_pages_per_seq;
    const size_t layer_base = (size_t)layer * a.n_pages;
    const int fresh = n_att - a.T;   // cells at positions >= fresh may come from this ubatch
    extern __shared__ __align__(128) uint8_t at_sm[];
    const uint32_t wbase = (uint32_t)__cvta_generic_to_shared(at_sm) + warp * AT_STAGES * 2 * TILE;

    // Warp w takes the 16-cell key tiles at c0 + 16 w + 64 i (each inside one page), staged by
    // cp.async into a ring of AT_STAGES (K, V) tiles. Cells past c1 repeat cell c1 - 1 (finite
    // values; their scores are masked), so that P = 0 times V is 0.
    const int j_first = c0 + AT_CELLS * warp;
    const int n_mine = j_first < c1 ? (c1 - j_first + 4 * AT_CELLS - 1) / (4 * AT_CELLS) : 0;
    auto load_tile = [&](int i) {   // this warp's i-th tile into stage i % AT_STAGES
        const int j0 = j_first + i * 4 * AT_CELLS;
        const int page = ptrow[j0 / kPage];
        const size_t row0 = ((layer_base + page) * a.KV + kvh) * kPage + (j0 % kPage);
        const uint32_t kd = wbase + (i % AT_STAGES) * 2 * TILE, vd = kd + TILE;
#pragma unroll
        for (int u = 0; u < AT_CELLS * CH / 32; ++u) {
            const int idx = u * 32 + lane, r = idx / CH, c = idx % CH;
            const int rr = min(j0 + r, c1 - 1) - j0;   // a cell past c1 repeats the last one
            cp_async16(kd + at_off<HD>(r, c), a.kc + (row0 + rr) * HD + c * 8);
            cp_async16(vd + at_off<HD>(r, c), a.vc + (row0 + rr) * HD + c * 8);
        }
    };
    // The cells of positions < fresh were stored by earlier ubatches and do not depend on the
    // preceding kernel: the first tile is requested before waiting for it when it holds none of
    // this ubatch's cells.
    const bool early = sp < ns_t && n_mine > 0 && j_first + AT_CELLS <= fresh;
    if (early) load_tile(0);
    LCX_PDL_WAIT();
    LCX_PDL_TRIGGER();
    LCX_TRACE(a, 1);
    if (sp >= ns_t) return;
    if (n_mine > 0 && !early) load_tile(0);
    cp_commit();
#pragma unroll
    for (int i = 1; i < AT_STAGES - 1; ++i) {
        if (i < n_mine) load_tile(i);
        cp_commit();
    }
    const int qw = a.H * HD;

    // Q as the A operand: rows = the G query heads of this KV head (rows >= G zero), pre-scaled
    // by log2(e) / sqrt(hd), f16 high + low parts
    const float scale = rsqrtf((float)HD) * 1.4426950408889634f;   // scores in the log2 domain
    uint32_t qa_hi[HD / 16][4], qa_lo[HD / 16][4];
    {
        const bool row_ok = g < G;
        const float *qp = a.q + (size_t)t * qw + (size_t)(kvh * G + (row_ok ? g : 0)) * HD;
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
            const int c0d = kk * 16 + 2 * tq, c1d = c0d + 8;
            const float2 x0 = row_ok ? *reinterpret_cast<const float2 *>(qp + c0d) : make_float2(0.f, 0.f);
            const float2 x1 = row_ok ? *reinterpret_cast<const float2 *>(qp + c1d) : make_float2(0.f, 0.f);
            split2(x0.x * scale, x0.y * scale, qa_hi[kk][0], qa_lo[kk][0]);
            split2(x1.x * scale, x1.y * scale, qa_hi[kk][2], qa_lo[kk][2]);
            qa_hi[kk][1] = qa_lo[kk][1] = qa_hi[kk][3] = qa_lo[kk][3] = 0u;   // rows g + 8
        }
    }
    float o[HD / 8][4];
#pragma unroll
    for (int d = 0; d < HD / 8; ++d) o[d][0] = o[d][1] = o[d][2] = o[d][3] = 0.f;
    float mrow = -CUDART_INF_F, lrow = 0.f;   // row g's running maximum and (this thread's) sum

    for (int i = 0; i < n_mine; ++i) {
        if (i + AT_STAGES - 1 < n_mine) load_tile(i + AT_STAGES - 1);
        cp_commit();
        cp_wait<AT_STAGES - 1>();
        __syncwarp();
        const int j0 = j_first + i * 4 * AT_CELLS;
        const uint32_t kb = wbase + (i % AT_STAGES) * 2 * TILE, vb = kb + TILE;
        // S = Q K^T for the tile's 16 cells (two n-tiles of 8)
        float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
            const int mm = lane >> 3, rr = lane & 7;
            uint32_t b0, b1, b2, b3;
            ldsm_x4(kb + at_off<HD>(8 * (mm >> 1) + rr, 2 * kk + (mm & 1)), b0, b1, b2, b3);
            mma16816(sc[0], qa_hi[kk], b0, b1);
            mma16816(sc[0], qa_lo[kk], b0, b1);
            mma16816(sc[1], qa_hi[kk], b2, b3);
            mma16816(sc[1], qa_lo[kk], b2, b3);
        }
        // cells past c1 masked; one online-softmax step for the tile (row g: this quad's 4 lanes)
        float mx = -CUDART_INF_F;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                if (j0 + 8 * nt + 2 * tq + e >= c1) sc[nt][e] = -CUDART_INF_F;
                mx = fmaxf(mx, sc[nt][e]);
            }
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float mn = fmaxf(mrow, mx);   // finite: the tile's first cell is valid
        const float alpha = ex2_approx(mrow - mn);
        mrow = mn;
        uint32_t pa_hi[4], pa_lo[4];
        {
            const float p00 = ex2_approx(sc[0][0] - mn), p01 = ex2_approx(sc[0][1] - mn);
            const float p10 = ex2_approx(sc[1][0] - mn), p11 = ex2_approx(sc[1][1] - mn);
            lrow = lrow * alpha + (p00 + p01 + p10 + p11);
            split2(p00, p01, pa_hi[0], pa_lo[0]);   // row g, cells 2tq, 2tq+1
            split2(p10, p11, pa_hi[2], pa_lo[2]);   // row g, cells 8 + 2tq, 8 + 2tq + 1
            pa_hi[1] = pa_lo[1] = pa_hi[3] = pa_lo[3] = 0u;
        }
#pragma unroll
        for (int d = 0; d < HD / 8; ++d) {
            o[d][0] *= alpha;
            o[d][1] *= alpha;
        }
        // O += P V (16 cells: one k-step; n-tiles of 8 dims)
#pragma unroll
        for (int d = 0; d < HD / 8; d += 2) {
            const int mm = lane >> 3, rr = lane & 7;
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(vb + at_off<HD>(8 * (mm & 1) + rr, d + (mm >> 1)), b0, b1, b2, b3);
            mma16816(o[d], pa_hi, b0, b1);
            mma16816(o[d], pa_lo, b0, b1);
            mma16816(o[d + 1], pa_hi, b2, b3);
            mma16816(o[d + 1], pa_lo, b2, b3);
        }
        __syncwarp();   // the stage is refilled AT_STAGES - 1 tiles later
    }
    cp_wait<0>();
    lrow += __shfl_xor_sync(0xffffffffu, lrow, 1);
    lrow += __shfl_xor_sync(0xffffffffu, lrow, 2);

    LCX_TRACE(a, 2);
    // ---- merge the 4 warps
    __shared__ float sm_m[4][G], sm_l[4][G];
    __shared__ float sm_acc[4][G][HD];
    if (g < G) {
        if (tq == 0) {
            sm_m[warp][g] = n_mine > 0 ? mrow : -CUDART_INF_F;
            sm_l[warp][g] = lrow;
        }
#pragma unroll
        for (int d = 0; d < HD / 8; ++d) {
            sm_acc[warp][g][d * 8 + 2 * tq] = o[d][0];
            sm_acc[warp][g][d * 8 + 2 * tq + 1] = o[d][1];
        }
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
    constexpr int smem = attn_smem_bytes<HD>();
    auto k16 = k_attn<HD, G, true>, k32 = k_attn<HD, G, false>;
    cudaError_t e = func_attr_once((const void *)(out16 ? k16 : k32), cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (!a.pdl) {   // stand-alone call: fully ordered after the caller's preceding work
        if (out16) k16<<<grid, 128, smem, s>>>(a, layer, chunk, ns);
        else k32<<<grid, 128, smem, s>>>(a, layer, chunk, ns);
        return cudaGetLastError();
    }
    if (out16) return launch_pdl(k16, grid, dim3(128), (size_t)smem, s, a, layer, chunk, ns);
    return launch_pdl(k32, grid, dim3(128), (size_t)smem, s, a, layer, chunk, ns);
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
