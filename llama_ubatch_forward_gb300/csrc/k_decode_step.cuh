// Persistent decode step: the whole forward of a one-token ubatch in one cooperative launch.
//
// Decode of one token reads every weight once (KV-cache section of the article: decode loads
// memory), and as a chain of separate launches it loses HBM time at every launch boundary: a
// GEMV CTA holds most of an SM's shared memory, so the next matrix's weights only start to
// stream once the previous launch has drained, and each launch re-pays its ramp-up. Here one
// CTA per SM lives for the whole step:
//   * the weight stages of every matrix of the step -- per layer the fused QKV, the output
//     projection, the fused gate/up and the down projection, then the vocabulary head -- stream
//     back to back through one ring of shared-memory slots with TMA bulk copies: the first
//     slots are filled at launch, and each slot is refilled with the stage S ahead in that
//     sequence as soon as its stage has been consumed. The ring thus runs ahead across phase
//     boundaries and is full of the next matrix while the CTA waits on a barrier, stages
//     activations or computes attention. (No separate producer warp: 8 warps per CTA leave
//     each thread up to 255 registers, 9 would cap it at 168.)
//   * the 8 warps run the phases in order: embedding gather; per layer QKV (RMSNorm, RoPE and
//     KV append fused), attention, output projection (+ residual), gate/up (RMSNorm, SwiGLU
//     fused), down (+ residual); then the logits with their argmax. A phase that reads what
//     another CTA wrote starts after a grid barrier (a monotonic arrival counter, bounded
//     polling); data written inside the step is read through L2 (ld.cg), never from L1;
//   * attention over the cache is split into (KV head, cell range) units, one per CTA, each
//     merged in the CTA and across splits by the last CTA of a KV head to arrive; the unit's
//     cached K/V lines are prefetched into L2 at the start of the layer, before QKV runs. A
//     unit does not wait for the whole QKV phase: each QKV epilogue publishes its row quad on a
//     per-KV-head counter (release), and the unit starts once its head's q, k and v rows are in.
// Every wait is bounded: a timed-out wait sets the error word, the CTA stops, and the others
// see the error word and stop at their next barrier.
//
// Code size matters as much as data movement here: with HBM saturated, every instruction-cache
// miss costs a loaded memory round trip (microseconds), so a kernel whose per-layer code does not
// stay cached pays them at every phase of every layer. The GEMV of all layer matrices is one
// non-inlined routine (epilogue chosen at run time), the activation staging and the attention
// loops are rolled, and the phase table lives in shared memory (the 28 KB L1 left next to the
// ring does not keep it).
#pragma once
#include <math_constants.h>

#include "k_gemv.cuh"

namespace lcx {
namespace step_detail {

using namespace gemv_detail;

// One weight-streaming phase: the matrix, its input vector and gains, and its stage plan.
struct alignas(16) StepPhase {
    GemvParams p;
    StagePlan pl;
    int n_stages;
};

struct StepArgs {
    const StepPhase *ph;   // [4 * n_layer + 1]: per layer QKV, O, gate/up, down; then the head
    int n_ph_all;          // 4 * n_layer + 1 (the table copied to shared memory)
    int slot_bytes;        // ring slot size (>= every phase's stage bytes)
    int slots;
    int x_bytes;           // staged activations / attention scratch at the start of shared memory
    unsigned int *sync;    // [0] barrier arrivals, [1] arrivals at the end, [16 + h] QKV quads of KV
                           // head h written so far; zero between launches
    int att_ns, att_chunk; // attention splits of this token: att_ns ranges of att_chunk cells
    int kvh_quads;         // QKV row quads per KV head and layer: (n_head / n_head_kv + 2) head_dim / 4
    const uint8_t *tok_embd;
    int t_embd;
    int32_t *amax_dst;     // argmax of the logits row (n_out == 1)
};

enum { PH_QKV = 0, PH_O = 1, PH_GU = 2, PH_DOWN = 3 };

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ int ld_volatile_i32(const int32_t *p) { return *reinterpret_cast<const volatile int32_t *>(p); }

// OR of a predicate over the 256 consumer threads (also a barrier among them)
__device__ __forceinline__ bool consumer_any(bool v) {
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, 1, 256, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
                 : "=r"(r) : "r"((uint32_t)v) : "memory");
    return r != 0;
}

// this thread's gains of the first staging iteration of a phase (constant inputs of the step)
__device__ __forceinline__ void gains_of(const StepPhase &P, float4 (&g)[4]) {
    const int hb = threadIdx.x, b = hb >> 1, half = hb & 1;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        g[j] = P.p.in.g && hb < 2 * P.p.nb ? *reinterpret_cast<const float4 *>(P.p.in.g + b * 32 + half * 16 + 4 * j)
                                           : make_float4(1.f, 1.f, 1.f, 1.f);
}

// Grid barrier among the consumers of all CTAs: barrier number n (1-based) completes when the
// counter reaches n * gridDim.x. Returns false (and the error word is set) if this CTA or any
// other gave up. With `next`, every thread loads its gains of that phase while the barrier
// completes: after this CTA's arrival (a release orders the loads issued before it too, so
// loading them earlier would delay the arrival by their round trip).
__device__ __forceinline__ bool grid_sync(const FwdArgs &a, unsigned *cnt, unsigned n, bool dead, int *s_ok,
                                          const StepPhase *next = nullptr, float4 (*gpre)[4] = nullptr) {
    const bool any_dead = consumer_any(dead);
    if (next && threadIdx.x != 0) gains_of(*next, *gpre);
    if (threadIdx.x == 0) {
        bool ok = !any_dead;
        if (!ok && next) gains_of(*next, *gpre);
        if (ok) {
            // release: this CTA's writes (ordered before by the barrier above) become visible
            // to the CTAs whose acquire load sees the count
            asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(cnt) : "memory");
            if (next) gains_of(*next, *gpre);
            const unsigned target = n * gridDim.x;
            ok = false;
            for (uint32_t i = 0; i < kSpinLimit; ++i) {
                if (ld_acquire_u32(cnt) >= target) {
                    ok = true;
                    break;
                }
                if ((i & 255u) == 255u && ld_volatile_i32(a.err)) break;
            }
        }
        if (!ok) atomicExch(a.err, 1);
        *s_ok = ok;
    }
    consumer_sync();
    return *s_ok != 0;
}

// producer wait for a free slot; gives up on the error word or after kSpinLimit polls
__device__ __forceinline__ bool producer_wait(uint64_t *bar, uint32_t parity, const int32_t *err) {
    const uint32_t ad = smem_u32(bar);
    for (uint32_t i = 0; i < kSpinLimit; ++i) {
        uint32_t done;
        asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, 1000;\n\tselp.u32 %0, 1, 0, p;\n\t}"
                     : "=r"(done) : "r"(ad), "r"(parity) : "memory");
        if (done) return true;
        if ((i & 1023u) == 1023u && ld_volatile_i32(err)) return false;
    }
    return false;
}

// timeline of the step (trace mode): slot = first slot + phase, 4 values per slot: [0] first
// CTA to enter the phase, [1] first CTA done staging its input (attention: its partial),
// [2] last CTA done staging, [3] last CTA done with the phase
__device__ __forceinline__ void step_trace(const FwdArgs &a, int phase, int which) {
    if (a.trace && threadIdx.x == 0) {
        unsigned long long *t = a.trace + 4 * (a.trace_slot + phase) + which;
        if (which < 2) atomicMin(t, lcx_gtime());
        else atomicMax(t, lcx_gtime());
    }
}

__device__ __forceinline__ float embd_elem(int type, const uint8_t *row, int i) {
    if (type == QF16) return __half2float(__ushort_as_half((uint16_t)(row[2 * i] | (row[2 * i + 1] << 8))));
    const int b = i >> 5, e = i & 31;
    const uint8_t *blk = row + (size_t)b * (type == Q8 ? 34 : 18);
    const float d = __half2float(__ushort_as_half((uint16_t)(blk[0] | (blk[1] << 8))));
    if (type == Q8) return d * (float)(int8_t)blk[2 + e];
    const int q = e < 16 ? (blk[2 + e] & 15) : (blk[2 + e - 16] >> 4);
    return d * (float)(q - 8);
}

// L2 prefetch of the cached K/V lines of this CTA's attention unit (cells [c0, c1) of KV head
// kvh, at most 512 cells); the cell the step itself appends is written later and not fetched.
template <int HD>
__device__ __forceinline__ void attn_prefetch(const FwdArgs &a, int layer, int kvh, int c0, int c1, const int *pages,
                                              int page0) {
    constexpr int LINES = HD * 2 / 128;   // 128-byte lines of one K (or V) row
    const int n_att = a.ub.pos[0] + 1;
    c1 = min(min(c1, n_att - 1), c0 + 512);
    for (int i = threadIdx.x; i < (c1 - c0) * 2 * LINES; i += 256) {
        const int j = c0 + i / (2 * LINES), w = i % (2 * LINES);
        const int page = pages[(j >> 6) - page0];
        const size_t row = (((size_t)layer * a.n_pages + page) * a.KV + kvh) * kPage + (j % kPage);
        const __half *base = (w < LINES ? a.kc : a.vc) + row * HD + (w % LINES) * 64;
        asm volatile("prefetch.global.L2 [%0];" ::"l"(base));
    }
}

// ---------------------------------------------------------------- attention
constexpr int kMaxUnitPages = 64;   // page ids of an attention unit kept in shared memory

// 2^x by the hardware approximation (relative error about 2^-22; results below 2^-126 flush to
// 0): the attention's scores and maxima are kept in the log2 domain
__device__ __forceinline__ float step_ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// K and V of 4 consecutive cells (inside one page), in registers: lanes 8c..8c+7 hold K dims
// (lane & 7) * HD / 8 .. of cell c; lane l holds V dims l * HD / 32 .. of cells 0..3.
template <int HD>
struct KVGroup {
    uint4 k[HD / 64];
    uint2 v[4];
};

// page of cell j of the unit's sequence (ids of the unit's pages in shared memory)
__device__ __forceinline__ int unit_page(const FwdArgs &a, const int *pages, int page0, int j) {
    const int i = (j >> 6) - page0;
    return i < kMaxUnitPages ? pages[i] : __ldcg(a.pt + (size_t)a.ub.seq[0] * a.max_pages_per_seq + (j >> 6));
}

// loads the group of cells j..j+3 (j % 4 == 0) of KV head kvh; cells >= c1 as zeros
template <int HD>
__device__ __forceinline__ void kv_group_load(const FwdArgs &a, int layer, int kvh, int page, int j, int c1,
                                              KVGroup<HD> &g) {
    constexpr int DPL = HD / 8, DPV = HD / 32;
    const int lane = threadIdx.x & 31, sub = lane & 7, cg = lane >> 3;
    const size_t row0 = (((size_t)layer * a.n_pages + page) * a.KV + kvh) * kPage + (j % kPage);
    const __half *kp = a.kc + (row0 + cg) * HD + sub * DPL;
#pragma unroll
    for (int i = 0; i < DPL / 8; ++i)
        g.k[i] = j + cg < c1 ? __ldcg(reinterpret_cast<const uint4 *>(kp + 8 * i)) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const __half *vp = a.vc + (row0 + c) * HD + lane * DPV;
        if (j + c < c1) {
            if (DPV == 4) g.v[c] = __ldcg(reinterpret_cast<const uint2 *>(vp));
            else g.v[c] = make_uint2(__ldcg(reinterpret_cast<const unsigned int *>(vp)), 0u);
        } else {
            g.v[c] = make_uint2(0u, 0u);
        }
    }
}

// One attention unit: query token 0 against cells [c0, c1) of KV head kvh by the 8 warps (the
// math of k_attn): warp w takes the 4-cell groups at c0 + 4 w + 32 i. A queue of 4 groups
// in registers keeps the next groups' K/V in flight while one is used; it was filled before this
// step's K/V were appended (the group holding the appended cell is re-read here). With one split
// the result goes to o32; otherwise the partial (max, sum, acc) is written and the last CTA of
// the KV head to arrive merges the splits in order. scr: attn_scratch_bytes(HD, G) of shared memory.
template <int HD, int G>
__device__ __forceinline__ void step_attention(const FwdArgs &a, int layer, int kvh, int sp, int chunk, int ns,
                                               float *scr, const int *pages, int page0, KVGroup<HD> (&q)[4],
                                               int trace_phase) {
    constexpr int NW = 8, DPL = HD / 8, DPV = HD / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int n_att = a.ub.pos[0] + 1;
    const int c0 = sp * chunk, c1 = min(c0 + chunk, n_att);
    const int sub = lane & 7, cg = lane >> 3;
    const float scale = rsqrtf((float)HD) * 1.4426950408889634f;   // scores in the log2 domain
    const int j_first = c0 + 4 * warp;
    {   // re-read the queued group that holds the appended cell (warp-uniform)
        const int jf = (n_att - 1) & ~3, i = (jf - j_first) >> 5;
        if (jf >= j_first && ((jf - j_first) & 31) == 0 && i < 4) {
            const int pg = unit_page(a, pages, page0, jf);
            if (i == 0) kv_group_load<HD>(a, layer, kvh, pg, jf, c1, q[0]);
            else if (i == 1) kv_group_load<HD>(a, layer, kvh, pg, jf, c1, q[1]);
            else if (i == 2) kv_group_load<HD>(a, layer, kvh, pg, jf, c1, q[2]);
            else kv_group_load<HD>(a, layer, kvh, pg, jf, c1, q[3]);
        }
    }

    float qr[G][DPL];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const float *qp = a.q + (size_t)(kvh * G + g) * HD + sub * DPL;
#pragma unroll
        for (int i = 0; i < DPL; i += 4) {
            const float4 v = __ldcg(reinterpret_cast<const float4 *>(qp + i));
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
#pragma unroll 1
    for (int j = j_first; j < c1; j += 4 * NW) {
        const KVGroup<HD> cur = q[0];
        q[0] = q[1];
        q[1] = q[2];
        q[2] = q[3];
        const int jn = j + 16 * NW;   // 4 groups ahead
        if (jn < c1) kv_group_load<HD>(a, layer, kvh, unit_page(a, pages, page0, jn), jn, c1, q[3]);
        const bool valid = j + cg < c1;
        float s[G];
        {
            float kf[DPL];
#pragma unroll
            for (int i = 0; i < DPL / 8; ++i) {
                const __half2 *h2 = reinterpret_cast<const __half2 *>(&cur.k[i]);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = __half22float2(h2[e]);
                    kf[8 * i + 2 * e] = f.x;
                    kf[8 * i + 2 * e + 1] = f.y;
                }
            }
#pragma unroll
            for (int g = 0; g < G; ++g) {   // two partial sums per head: shorter dependent chains
                float d0 = 0.f, d1 = 0.f;
#pragma unroll
                for (int i = 0; i < DPL; i += 2) {
                    d0 = fmaf(qr[g][i], kf[i], d0);
                    d1 = fmaf(qr[g][i + 1], kf[i + 1], d1);
                }
                float d = d0 + d1;
                d += __shfl_xor_sync(0xffffffffu, d, 1);
                d += __shfl_xor_sync(0xffffffffu, d, 2);
                d += __shfl_xor_sync(0xffffffffu, d, 4);
                s[g] = valid ? d : -CUDART_INF_F;
            }
        }
        float p[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {   // online softmax over the group's 4 cells
            float mx = s[g];
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float mn = fmaxf(m[g], mx);
            const float alpha = step_ex2(m[g] - mn);
            p[g] = step_ex2(s[g] - mn);
            float ps = p[g];
            ps += __shfl_xor_sync(0xffffffffu, ps, 8);
            ps += __shfl_xor_sync(0xffffffffu, ps, 16);
            l[g] = l[g] * alpha + ps;
            m[g] = mn;
#pragma unroll
            for (int i = 0; i < DPV; ++i) acc[g][i] *= alpha;
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {   // P.V; cells past c1 have p = 0 and zero V
            const uint2 raw = cur.v[c];
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
                const float pc = __shfl_sync(0xffffffffu, p[g], 8 * c);
#pragma unroll
                for (int i = 0; i < DPV; ++i) acc[g][i] = fmaf(pc, vf[i], acc[g][i]);
            }
        }
    }

    // ---- merge the 8 warps: per query head the max, the sum and the 8 warps' weights once
    float *sm_m = scr, *sm_l = scr + NW * G, *fac = scr + 2 * NW * G, *sM = scr + 3 * NW * G, *sL = sM + G;
    int *flag = reinterpret_cast<int *>(sL + G);
    float *sm_acc = scr + 3 * NW * G + 2 * G + 4;   // [NW][G][HD]
#pragma unroll
    for (int g = 0; g < G; ++g) {
        if (lane == 0) {
            sm_m[warp * G + g] = m[g];
            sm_l[warp * G + g] = l[g];
        }
#pragma unroll
        for (int i = 0; i < DPV; ++i) sm_acc[(warp * G + g) * HD + lane * DPV + i] = acc[g][i];
    }
    consumer_sync();
    if (threadIdx.x < G) {
        const int g = threadIdx.x;
        float M = -CUDART_INF_F;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, sm_m[w * G + g]);
        float L = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const float mw = sm_m[w * G + g];
            const float f = mw == -CUDART_INF_F ? 0.f : exp2f(mw - M);
            fac[w * G + g] = f;
            L += sm_l[w * G + g] * f;
        }
        sM[g] = M;
        sL[g] = L;
    }
    consumer_sync();
    float *part = a.att_part;
    const size_t prow = (size_t)kvh * ns;   // partial rows of this KV head (token 0)
#pragma unroll 1
    for (int idx = threadIdx.x; idx < G * HD; idx += 256) {
        const int g = idx / HD, dd = idx % HD;
        float A = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) A = fmaf(sm_acc[(w * G + g) * HD + dd], fac[w * G + g], A);
        if (ns == 1) {
            a.o32[(size_t)(kvh * G + g) * HD + dd] = A / sL[g];
        } else {
            float *pr = part + ((prow + sp) * G + g) * (HD + 2);
            pr[2 + dd] = A;
            if (dd == 0) {
                pr[0] = sM[g];
                pr[1] = sL[g];
            }
        }
    }
    step_trace(a, trace_phase, 1);
    step_trace(a, trace_phase, 2);
    if (ns == 1) return;

    // ---- split merge by the last CTA of this KV head to arrive: the barrier orders the CTA's
    // partial stores before thread 0's acq_rel arrival, which publishes them and, for the last
    // CTA, acquires the others'
    consumer_sync();
    if (threadIdx.x == 0) {
        unsigned prev;
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(prev) : "l"(a.att_cnt + kvh) : "memory");
        *flag = prev == (unsigned)(ns - 1);
    }
    consumer_sync();
    if (!*flag) return;
    // the partial sums of this thread's outputs for the first 24 splits are loaded first, so their
    // round trip overlaps the one of the weights w_s = 2^(M_s - M*) / L* (one warp per query
    // head, lanes over splits)
    constexpr int PER = (G * HD + 255) / 256, NB = 24;
    float av[PER][NB];
#pragma unroll
    for (int q = 0; q < PER; ++q) {
        const int idx = threadIdx.x + 256 * q;
        const int g = idx / HD, dd = idx % HD;
#pragma unroll
        for (int u = 0; u < NB; ++u)
            av[q][u] = idx < G * HD && u < ns ? __ldcg(part + ((prow + u) * G + g) * (HD + 2) + 2 + dd) : 0.f;
    }
    float *sw = sm_acc;   // [64][G]
    for (int g = warp; g < G; g += NW) {
        float ms[2], ls[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int s2 = lane + 32 * h;
            const float *pr = part + ((prow + s2) * G + g) * (HD + 2);
            ms[h] = s2 < ns ? __ldcg(pr) : -CUDART_INF_F;
            ls[h] = s2 < ns ? __ldcg(pr + 1) : 0.f;
        }
        float M = fmaxf(ms[0], ms[1]);
#pragma unroll
        for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        float e[2], L = 0.f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            e[h] = lane + 32 * h < ns ? exp2f(ms[h] - M) : 0.f;
            L += e[h] * ls[h];
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
#pragma unroll
        for (int h = 0; h < 2; ++h)
            if (lane + 32 * h < ns) sw[(lane + 32 * h) * G + g] = e[h] / L;
    }
    consumer_sync();
#pragma unroll
    for (int q = 0; q < PER; ++q) {
        const int idx = threadIdx.x + 256 * q;
        if (idx >= G * HD) continue;
        const int g = idx / HD, dd = idx % HD;
        float o = 0.f;
#pragma unroll
        for (int u = 0; u < NB; ++u)
            if (u < ns) o = fmaf(sw[u * G + g], av[q][u], o);
#pragma unroll 1
        for (int s0 = NB; s0 < ns; ++s0)   // splits past the first 24 (long contexts of small models)
            o = fmaf(sw[s0 * G + g], __ldcg(part + ((prow + s0) * G + g) * (HD + 2) + 2 + dd), o);
        a.o32[(size_t)(kvh * G + g) * HD + dd] = o;
    }
    if (threadIdx.x == 0) a.att_cnt[kvh] = 0;
}

__host__ __device__ constexpr int attn_scratch_bytes(int hd, int g) { return (3 * 8 * g + 2 * g + 4 + 8 * g * hd) * 4; }

// ---------------------------------------------------------------- weight streaming
// The ring's refill cursor (used by one thread, kFeedThread): the next stage of the step's
// sequence -- phase `ph`, stage `st` of it -- and the number of stages issued so far.
constexpr int kFeedThread = 255;
struct Feeder {
    int ph, st, issued;
};

// Issues the cursor's stage into ring slot issued % slots and advances the cursor; nothing once
// the sequence is exhausted. tab: the phase table (shared memory).
__device__ __forceinline__ void feed_one(const StepArgs &s, const StepPhase *tab, int n_ph, int L, Feeder &f,
                                         uint8_t *ring, uint64_t *full) {
    while (f.ph < n_ph && f.st >= tab[f.ph].n_stages) {
        ++f.ph;
        f.st = blockIdx.x;
    }
    if (f.ph >= n_ph) return;
    const StepPhase &P = tab[f.ph];
    const int slot = f.issued % s.slots;
    uint8_t *dst = ring + (size_t)slot * s.slot_bytes;
    if (f.ph != 4 * L && f.ph % 4 == PH_GU) issue_stage<EPI_SWIGLU>(P.p, P.pl, f.st, dst, &full[slot]);
    else issue_stage<EPI_RESID>(P.p, P.pl, f.st, dst, &full[slot]);
    f.st += gridDim.x;
    ++f.issued;
}

// Stages x (token 0) for a matrix with nb blocks: as stage_token, in a rolled loop over pairs of
// half-block iterations, the next pair's values loading while the current ones are split (two
// independent chains per thread). gpre: this thread's gains of the first iteration, loaded
// before the barrier (or NULL).
template <int QT>
__device__ __forceinline__ void stage_x(const GemvParams &p, uint8_t *stage_t, float *red, const float4 *gpre) {
    constexpr int NTHR = 256;
    const int nb = p.nb;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float *xr = p.in.x;
    uint8_t *hp = stage_t, *lp = stage_t + (size_t)nb * 32;
    float2 *mp = reinterpret_cast<float2 *>(stage_t + (size_t)nb * 64);
    float ss = 0.f;
    const int n_half = 2 * nb, iters = (n_half + NTHR - 1) / NTHR;
    float4 nx[2][4];
    auto load = [&](int it, float4 (&dst)[4]) {
        const int hb = it * NTHR + threadIdx.x;
#pragma unroll
        for (int j = 0; j < 4; ++j)
            dst[j] = it < iters && hb < n_half
                         ? __ldcg(reinterpret_cast<const float4 *>(xr + (hb >> 1) * 32 + (hb & 1) * 16 + 4 * j))
                         : make_float4(0, 0, 0, 0);
    };
    // split one half block (16 values of iteration it) into the hi / lo planes and the meta
    auto split = [&](int it, const float4 (&xv)[4]) {
        const int hb = it * NTHR + threadIdx.x, b = hb >> 1, half = hb & 1;
        const bool active = hb < n_half;
        float v[16];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float4 q = xv[j];
            ss += q.x * q.x + q.y * q.y + q.z * q.z + q.w * q.w;
            if (p.in.g && active) {
                const float4 gg = gpre && it == 0 ? gpre[j]
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
    };
    load(0, nx[0]);
    load(1, nx[1]);
#pragma unroll 1
    for (int it = 0; it < iters; it += 2) {
        float4 c0[4], c1[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            c0[j] = nx[0][j];
            c1[j] = nx[1][j];
        }
        if (it + 2 < iters) {
            load(it + 2, nx[0]);
            load(it + 3, nx[1]);
        }
        split(it, c0);
        if (it + 1 < iters) split(it + 1, c1);   // uniform over the CTA
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) red[warp] = ss;
}

// How one phase's stages map onto the 256 threads. The R = 4 tps rows of a stage are split into
// G row groups of NR = R / G rows; the 256 / G threads of a group (whole warps) take the nb
// blocks of the row, NBT <= 2 blocks each, fixed for the whole phase: a thread keeps its blocks'
// staged activations in registers and multiplies them with the NR rows of every stage, so the
// shared-memory traffic of a stage is its weights alone.
struct GemvMap {
    int G, NR, NBT;
};
__host__ __device__ inline GemvMap gemv_map(int tps, int nb) {
    const int R = 4 * tps;
    int g = 1;
    while (g * 2 <= R && g * 2 <= 8 && nb * g * 2 <= 256) g *= 2;
    GemvMap m;
    m.G = g;
    m.NR = R / g;
    m.NBT = (nb + 256 / g - 1) / (256 / g);
    return m;
}

// Sums v over the 32 lanes of a warp, scattering the NR row sums: afterwards every lane holds the
// sum of row `row` (the lanes whose bits 16, 8, .. select it), 4 + 2 + 1 + 1 + 1 shuffles for 8 rows.
template <int NR>
__device__ __forceinline__ float warp_reduce_rows(float (&v)[NR], int lane, int &row) {
    int base = 0;
#pragma unroll
    for (int st = 0; st < 5; ++st) {
        const int m = 16 >> st;
        const int n = NR >> st;   // rows still held (a constant once unrolled)
        if (n >= 2) {
            const bool up = lane & m;
#pragma unroll
            for (int i = 0; i < NR / 2; ++i) {
                if (i < n / 2) {
                    const float send = up ? v[i] : v[i + n / 2];
                    const float keep = up ? v[i + n / 2] : v[i];
                    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
                }
            }
            if (up) base += n / 2;
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], m);
        }
    }
    row = base;
    return v[0];
}

// The dot products of one landed stage for this thread's NR rows and NBT blocks, reduced over
// the warp and left in part[stage row * 8 + warp within the row group].
template <int QT, int NR>
__device__ __forceinline__ void stage_dots(const uint8_t *sq, int QBY, int nb, const XQ (&xq)[2], const int (&bk)[2],
                                           int nbt, int grp, int wg, float *pk) {
    constexpr int QB = QT == Q8 ? 32 : 16;
    const int lane = threadIdx.x & 31;
    float acc[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) acc[r] = 0.f;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        if (i >= nbt) break;
        const int b = bk[i];
        if (b >= nb) continue;
        float d[NR];
#pragma unroll
        for (int r = 0; r < NR; r += 4) {   // scales of whole quads (NR >= 4) ...
            if (NR >= 4) {
                const int sr = grp * NR + r;
                const uint2 s4 = *reinterpret_cast<const uint2 *>(sq + (sr >> 2) * QBY + quad_s_off(QB, b));
                const float2 d01 = __half22float2(*reinterpret_cast<const __half2 *>(&s4.x));
                const float2 d23 = __half22float2(*reinterpret_cast<const __half2 *>(&s4.y));
                d[r] = d01.x; d[(r + 1) % NR] = d01.y; d[(r + 2) % NR] = d23.x; d[(r + 3) % NR] = d23.y;
            }
        }
        if (NR < 4) {   // ... or of single rows
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                const int sr = grp * NR + r;
                d[r] = __half2float(*reinterpret_cast<const __half *>(sq + (sr >> 2) * QBY + quad_s_off(QB, b) + 2 * (sr & 3)));
            }
        }
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            const int sr = grp * NR + r;
            const uint4 *wp = reinterpret_cast<const uint4 *>(sq + (sr >> 2) * QBY + quad_q_off(QB, sr & 3, b));
            const uint4 w0 = wp[0];
            const uint4 w1 = QT == Q8 ? wp[1] : w0;
            const int Pd = QT == Q4 ? q4_idot(w0, xq[i]) : q8_idot(w0, w1, xq[i]);
            acc[r] = fmaf(d[r] * xq[i].s, (float)Pd, acc[r]);
        }
    }
    int row;
    const float sum = warp_reduce_rows<NR>(acc, lane, row);
    if ((lane & (32 / NR - 1)) == 0) pk[(grp * NR + row) * 8 + wg] = sum;
}

// The dot products of one landed stage (all 256 threads; one copy of the loop per row count),
// left in pk[stage row * 8 + warp of the row group].
template <int QT>
__device__ __forceinline__ void dots_rt(const StepPhase &P, const GemvMap &mp, const uint8_t *sq, const XQ (&xq)[2],
                                        const int (&bk)[2], float *pk) {
    const int per_grp = 256 / mp.G;   // threads of a row group
    const int grp = threadIdx.x / per_grp, wg = (threadIdx.x % per_grp) >> 5;
    switch (mp.NR) {
        case 8: stage_dots<QT, 8>(sq, P.pl.quad_bytes, P.p.nb, xq, bk, mp.NBT, grp, wg, pk); break;
        case 4: stage_dots<QT, 4>(sq, P.pl.quad_bytes, P.p.nb, xq, bk, mp.NBT, grp, wg, pk); break;
        case 2: stage_dots<QT, 2>(sq, P.pl.quad_bytes, P.p.nb, xq, bk, mp.NBT, grp, wg, pk); break;
        default: stage_dots<QT, 1>(sq, P.pl.quad_bytes, P.p.nb, xq, bk, mp.NBT, grp, wg, pk); break;
    }
}

// Epilogue of task e of stage st (one thread), epilogue kind chosen at run time: a task is a row
// quad, or for SwiGLU the gate and up rows of 2 features.
__device__ __forceinline__ void epilogue_rt(const StepPhase &P, const GemvMap &mp, int epi, const FwdArgs &a,
                                            int layer, int st, int e, const float *pk, float rs, const EpiIn &ein,
                                            unsigned long long &best, unsigned *kvh_cnt) {
    const GemvParams &p = P.p;
    const int n_wg = 8 / mp.G;   // warps of a row group: partial sums per row
    const bool swiglu = epi == EPI_SWIGLU;
    float v[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        // stage row of output r: the task's quad, or gate (r < 2) / up rows of its feature pair
        const int sr = swiglu ? (2 * (e >> 1) + (r >> 1)) * 4 + 2 * (e & 1) + (r & 1) : 4 * e + r;
        const float4 lo = *reinterpret_cast<const float4 *>(pk + sr * 8);
        const float4 hi = *reinterpret_cast<const float4 *>(pk + sr * 8 + 4);
        float sum = lo.x;
        if (n_wg > 1) sum += lo.y;
        if (n_wg > 2) sum += lo.z + lo.w;
        if (n_wg > 4) sum += hi.x + hi.y + hi.z + hi.w;
        v[r] = sum * rs;
    }
    const int task = st * P.pl.tps + e, r0 = 4 * task;
    unsigned long long bkey = 0ull;
    switch (epi) {
        case EPI_SWIGLU: {   // features 4 (task / 2) + 2 (task & 1) + {0, 1}
            const float g2[2] = {v[0], v[1]}, u2[2] = {v[2], v[3]};
            epi_swiglu2<false>(a, 0, 4 * (task >> 1) + 2 * (task & 1), g2, u2);
            break;
        }
        case EPI_QKV: {
            epi_quad_in<EPI_QKV>(a, layer, 0, r0, p.N, v, ein, bkey);
            // count the quad for its KV head (shared memory); the CTA publishes the counts once,
            // after its last QKV stage
            const int qw = a.H * a.hd, kw = a.KV * a.hd;
            if (r0 < qw + 2 * kw) {
                const int sh = __ffs(a.hd) - 1;
                const int kvh = r0 < qw ? (r0 >> sh) / (a.H / a.KV) : ((r0 - qw) >> sh) % a.KV;
                atomicAdd(kvh_cnt + kvh, 1u);
            }
            break;
        }
        case EPI_RESID: epi_quad_in<EPI_RESID>(a, layer, 0, r0, p.N, v, ein, bkey); break;
        default: epi_quad_in<EPI_LOGITS>(a, layer, 0, r0, p.N, v, ein, bkey); break;
    }
    best = bkey > best ? bkey : best;
}

// The token's constants for the whole step, in shared memory from the launch on: its cache cell
// and the RoPE (cos, sin) row of its position. The QKV epilogue reads them there instead of
// a dependent chain of global loads (position, then the row it indexes) at every stage pair.
struct StepConst {
    const float2 *rope;   // [head_dim / 2]
    int cell;
    unsigned *pub;        // [n_head_kv] QKV quads of this CTA per KV head, not yet published
};

__device__ __forceinline__ EpiIn qkv_in(const FwdArgs &a, int r0, const StepConst &sc) {
    EpiIn in{};
    in.cell = sc.cell;
    const int qw = a.H * a.hd, kw = a.KV * a.hd;
    if (r0 < qw + kw) {   // q or k rows: the quad lies inside one head (hd % 4 == 0)
        const int dim = (r0 < qw ? r0 : r0 - qw) & (a.hd - 1);
        in.cs = *reinterpret_cast<const float4 *>(sc.rope + dim / 2);
    }
    return in;
}

// State the GEMV routine carries from phase to phase.
struct GemvState {
    int k;                    // ring uses so far
    Feeder f;                 // refill cursor (kFeedThread)
    bool dead;
    unsigned long long best;  // logits argmax key of this thread
};

// One weight-streaming phase (all 256 threads): stage x, then consume this CTA's stages of the
// phase's matrix from the ring, refilling each slot with the stage S ahead in the sequence.
template <int QT>
__device__ __noinline__ void step_gemv(const StepArgs &s, const StepPhase *tab, int ph, int n_ph, int epi,
                                       const FwdArgs &a, int layer, uint8_t *xs, uint8_t *ring, uint64_t *full,
                                       GemvState &gs, float *part, float *red, const float4 *gpre, int trace_phase,
                                       StepConst sc) {
    const StepPhase &P = tab[ph];
    if (!gs.dead) stage_x<QT>(P.p, xs, red, 2 * P.p.nb <= 256 ? gpre : nullptr);
    consumer_sync();
    float rs;   // RMS factor of the phase's input (1 without norm gains; NaN for a non-finite input)
    {
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) tot += red[w];
        rs = finite_or_nan(tot, P.p.in.g ? 1.0f / sqrtf(tot / (float)P.p.K + a.eps) : 1.f);
    }
    // this thread's blocks and their staged activations, for the whole phase
    const GemvMap mp = gemv_map(P.pl.tps, P.p.nb);
    XQ xq[2];
    int bk[2];
    {
        const int per_grp = 256 / mp.G, wg = (threadIdx.x % per_grp) >> 5;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            bk[i] = 32 * wg + block_of_lane(threadIdx.x & 31) + i * per_grp;
            if (i < mp.NBT && bk[i] < P.p.nb) load_xq(xs, P.p.nb, bk[i], xq[i]);
        }
    }
    step_trace(a, trace_phase, 1);
    step_trace(a, trace_phase, 2);
    int k = gs.k;
    bool dead = gs.dead;
    unsigned long long best = gs.best;
    Feeder f = gs.f;
    const int tps = P.pl.tps, n_tasks = P.p.n_tasks;
    // stages in pairs: both stages' dot products, one barrier, then warp 0 and warp 1 apply the
    // two epilogues side by side, and both slots are refilled
    int bi = 0;   // pair index: the partial sums alternate between two buffers
#pragma unroll 1
    for (int st = blockIdx.x; st < P.n_stages; st += 2 * gridDim.x, ++bi) {
        const int st2 = st + gridDim.x;
        const bool two = st2 < P.n_stages;
        const int slot0 = k % s.slots, slot1 = (k + 1) % s.slots;
        float *pk0 = part + (bi & 1) * 256, *pk1 = pk0 + 128;
        // this thread's epilogue, if any: warp 0 takes the tasks of the first stage, warp 1 the second's
        const int my_st = threadIdx.x < 32 ? st : st2, e = threadIdx.x & 31;
        const bool epi_thread = !dead && threadIdx.x < 64 && (threadIdx.x < 32 || two) &&
                                e < min(tps, n_tasks - my_st * tps);
        EpiIn ein{};
        if (epi_thread && epi == EPI_RESID) ein = epi_load<EPI_RESID>(a, 0, (my_st * tps + e) * 4, P.p.N);
        if (epi_thread && epi == EPI_QKV) ein = qkv_in(a, (my_st * tps + e) * 4, sc);
        // the pair's two stages through one copy of the dot-product code (instruction cache)
#pragma unroll 1
        for (int u = 0; u < (two ? 2 : 1); ++u) {
            const int slot = u ? slot1 : slot0;
            if (!dead && !mbar_wait(&full[slot], ((k + u) / s.slots) & 1)) {
                dead = true;
                atomicExch(a.err, 1);
            }
            if (!dead) dots_rt<QT>(P, mp, ring + (size_t)slot * s.slot_bytes, xq, bk, u ? pk1 : pk0);
        }
        consumer_sync();
        if (epi_thread) epilogue_rt(P, mp, epi, a, layer, my_st, e, threadIdx.x < 32 ? pk0 : pk1, rs, ein, best, sc.pub);
        // every warp is past its reads of the slots (the barrier above): refill them
        if (threadIdx.x == kFeedThread && !dead) {
            feed_one(s, tab, n_ph, a.L, f, ring, full);
            if (two) feed_one(s, tab, n_ph, a.L, f, ring, full);
        }
        k += two ? 2 : 1;
    }
    gs.k = k;
    gs.dead = dead;
    gs.best = best;
    gs.f = f;
    if (epi == EPI_QKV) {
        // publish this CTA's quads, one release reduction per KV head: the barrier orders every
        // epilogue thread's stores before it
        consumer_sync();
        if ((int)threadIdx.x < a.KV) {
            const unsigned n = sc.pub[threadIdx.x];
            if (n && !dead) asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(s.sync + 16 + threadIdx.x), "r"(n) : "memory");
            sc.pub[threadIdx.x] = 0u;
        }
    }
    step_trace(a, trace_phase, 3);
}


template <int QL, int QH, int HD, int G>
__global__ void __launch_bounds__(256, 1) k_decode_step(const __grid_constant__ StepArgs s,
                                                        const __grid_constant__ FwdArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *xs = smem;
    uint8_t *ring = smem + s.x_bytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(ring + (size_t)s.slots * s.slot_bytes);
    StepPhase *tab = reinterpret_cast<StepPhase *>(full + kMaxStages);
    int *pages = reinterpret_cast<int *>(tab + s.n_ph_all);
    const int L = a.L;
    const int n_ph = 4 * L + (a.n_out > 0 ? 1 : 0);

    if (threadIdx.x == 0) {
        for (int i = 0; i < s.slots; ++i) mbar_init(&full[i], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    {   // the phase table, into shared memory
        const uint4 *src = reinterpret_cast<const uint4 *>(s.ph);
        uint4 *dst = reinterpret_cast<uint4 *>(tab);
        const int n16 = (int)(s.n_ph_all * sizeof(StepPhase) / 16);
        for (int i = threadIdx.x; i < n16; i += 256) dst[i] = src[i];
    }
    __shared__ __align__(16) float2 s_rope[128];   // head_dim <= 256
    __shared__ int s_cell;
    __shared__ unsigned s_pub[48];                  // n_head_kv <= 48
    {   // the token's constants (written by the host before the launch)
        const int pos0 = a.ub.pos[0];
        for (int i = threadIdx.x; i < a.hd / 2; i += 256) s_rope[i] = a.rope[(size_t)pos0 * (a.hd / 2) + i];
        if (threadIdx.x == 0) s_cell = a.ub.cell[0];
        if (threadIdx.x < 48) s_pub[threadIdx.x] = 0u;
    }
    __syncthreads();
    const StepConst sc{s_rope, s_cell, s_pub};
    GemvState gs{0, Feeder{0, (int)blockIdx.x, 0}, false, 0ull};
    // fill the ring: the weights do not depend on anything this step computes
    if (threadIdx.x == kFeedThread)
        for (int i = 0; i < s.slots; ++i) feed_one(s, tab, n_ph, L, gs.f, ring, full);

    __shared__ float red[8];
    __shared__ __align__(16) float part[2 * 2 * 16 * 8];   // [batch parity][stage of the pair][16 rows][8]
    __shared__ int s_ok;
    unsigned *bar = s.sync;
    unsigned n_bar = 0;
    const int units = a.KV * s.att_ns;
    const bool has_unit = (int)blockIdx.x < units;
    const int u_kvh = blockIdx.x % a.KV, u_sp = blockIdx.x / a.KV;

    // embedding row of the token, spread over the CTAs; CTA 0 also applies the page-table
    // updates and clears the argmax key
    step_trace(a, 0, 0);
    {
        const int id = a.tok_src[0];
        const uint8_t *row = s.tok_embd + (size_t)id * (s.t_embd == QF16 ? 2 * a.d : (a.d / 32) * (s.t_embd == Q8 ? 34 : 18));
        for (int i = blockIdx.x * 256 + threadIdx.x; i < a.d; i += gridDim.x * 256) a.x[i] = embd_elem(s.t_embd, row, i);
        if (blockIdx.x == 0) {
            for (int u = threadIdx.x; u < a.ub.n_upd; u += 256) a.pt[a.ub.pt_upd[2 * u]] = a.ub.pt_upd[2 * u + 1];
            if (threadIdx.x < a.n_out) a.amax_key[threadIdx.x] = 0ull;
        }
    }
    step_trace(a, 0, 3);

    // this token's attention unit: cells [ac0, ac1) of KV head u_kvh
    const int n_att = a.ub.pos[0] + 1;
    const int ac0 = u_sp * s.att_chunk, ac1 = min(ac0 + s.att_chunk, n_att);
    const int page0 = ac0 >> 6;
    KVGroup<HD> kvq[4];   // this warp's first 4 groups of the unit, loaded before each attention barrier
    float4 gpre[4];
    gs.dead = !grid_sync(a, bar, ++n_bar, gs.dead, &s_ok, &tab[0], &gpre);
    if (has_unit) {   // the unit's page ids (the page table is complete after the barrier)
        const int n_pg = min(kMaxUnitPages, ((max(ac1, ac0 + 1) - 1) >> 6) - page0 + 1);
        const int32_t *ptrow = a.pt + (size_t)a.ub.seq[0] * a.max_pages_per_seq;
        for (int i = threadIdx.x; i < n_pg; i += 256) pages[i] = __ldcg(ptrow + page0 + i);
        consumer_sync();
    }

    for (int l = 0; l < L && !gs.dead; ++l) {
        const int tp = 1 + 5 * l;
        // QKV (the attention unit's cached K/V lines go to L2 meanwhile)
        step_trace(a, tp, 0);
        if (has_unit) attn_prefetch<HD>(a, l, u_kvh, ac0, ac1, pages, page0);
        step_gemv<QL>(s, tab, 4 * l + PH_QKV, n_ph, EPI_QKV, a, l, xs, ring, full, gs, part, red, gpre, tp, sc);
        if (has_unit) {
            const int jf = ac0 + 4 * (threadIdx.x >> 5);
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (jf + 32 * i < ac1)
                    kv_group_load<HD>(a, l, u_kvh, unit_page(a, pages, page0, jf + 32 * i), jf + 32 * i, ac1, kvq[i]);
        }
        if (has_unit) {   // this unit's KV head: all its q, k and v quads of layer l written
            if (threadIdx.x == 0) {
                const unsigned target = (unsigned)(l + 1) * (unsigned)s.kvh_quads;
                bool ok = !gs.dead;
                if (ok) {
                    ok = false;
                    for (uint32_t i = 0; i < kSpinLimit; ++i) {
                        if (ld_acquire_u32(s.sync + 16 + u_kvh) >= target) {
                            ok = true;
                            break;
                        }
                        if ((i & 255u) == 255u && ld_volatile_i32(a.err)) break;
                    }
                    if (!ok) atomicExch(a.err, 1);
                }
                s_ok = ok;
            }
            consumer_sync();
            gs.dead = !s_ok;
        }
        // attention
        step_trace(a, tp + 1, 0);
        if (has_unit)
            step_attention<HD, G>(a, l, u_kvh, u_sp, s.att_chunk, s.att_ns, reinterpret_cast<float *>(xs), pages, page0,
                                  kvq, tp + 1);
        step_trace(a, tp + 1, 3);
        gs.dead = !grid_sync(a, bar, ++n_bar, gs.dead, &s_ok);
        if (gs.dead) break;
        // output projection + residual
        step_trace(a, tp + 2, 0);
        step_gemv<QL>(s, tab, 4 * l + PH_O, n_ph, EPI_RESID, a, l, xs, ring, full, gs, part, red, nullptr, tp + 2, sc);
        gs.dead = !grid_sync(a, bar, ++n_bar, gs.dead, &s_ok, &tab[4 * l + PH_GU], &gpre);
        if (gs.dead) break;
        // gate/up + SwiGLU
        step_trace(a, tp + 3, 0);
        step_gemv<QL>(s, tab, 4 * l + PH_GU, n_ph, EPI_SWIGLU, a, l, xs, ring, full, gs, part, red, gpre, tp + 3, sc);
        gs.dead = !grid_sync(a, bar, ++n_bar, gs.dead, &s_ok);
        if (gs.dead) break;
        // down + residual
        step_trace(a, tp + 4, 0);
        step_gemv<QL>(s, tab, 4 * l + PH_DOWN, n_ph, EPI_RESID, a, l, xs, ring, full, gs, part, red, nullptr, tp + 4, sc);
        // next layer's QKV, or the head
        gs.dead = !grid_sync(a, bar, ++n_bar, gs.dead, &s_ok, &tab[4 * l + 4], &gpre);
    }
    if (gs.dead) {
        // copies still in flight must land before the CTA's shared memory is released
        if (threadIdx.x == kFeedThread)
            for (int j = gs.f.issued > s.slots ? gs.f.issued - s.slots : 0; j < gs.f.issued; ++j)
                mbar_wait(&full[j % s.slots], (j / s.slots) & 1);
        return;
    }
    if (a.n_out > 0) {
        const int tp = 1 + 5 * L;
        step_trace(a, tp, 0);
        step_gemv<QH>(s, tab, 4 * L, n_ph, EPI_LOGITS, a, -1, xs, ring, full, gs, part, red, gpre, tp, sc);
        const unsigned long long bst[1] = {gs.best};
        logits_cta_reduce<1>(a, 1, bst);
    }
    // the last CTA to finish writes the argmax and resets the step's counters: every other CTA
    // is past its last barrier by then
    consumer_sync();
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(&bar[1], 1u) == gridDim.x - 1) {
            __threadfence();
            if (a.n_out > 0 && s.amax_dst) {
                const unsigned long long key = __ldcg(a.amax_key);
                s.amax_dst[0] = (int32_t)(0xffffffffu - (uint32_t)(key & 0xffffffffull));
            }
            bar[0] = 0u;
            bar[1] = 0u;
            for (int h = 0; h < a.KV; ++h) bar[16 + h] = 0u;
        }
    }
}

}  // namespace step_detail
}  // namespace lcx
