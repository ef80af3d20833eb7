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
//     cached K/V lines are prefetched into L2 at the start of the layer, before QKV runs.
// Every wait is bounded: a timed-out wait sets the error word, the CTA stops, and the others
// see the error word and stop at their next barrier.
#pragma once
#include <math_constants.h>

#include "k_gemv.cuh"

namespace lcx {
namespace step_detail {

using namespace gemv_detail;

// One weight-streaming phase: the matrix, its input vector and gains, and its stage plan.
struct StepPhase {
    GemvParams p;
    StagePlan pl;
    int n_stages;
};

struct StepArgs {
    const StepPhase *ph;   // [4 * n_layer + 1]: per layer QKV, O, gate/up, down; then the head
    int slot_bytes;        // ring slot size (>= every phase's stage bytes)
    int slots;
    int x_bytes;           // staged activations / attention scratch at the start of shared memory
    unsigned int *sync;    // [0] barrier arrivals, [1] arrivals at the end; zero between launches
    int att_ns, att_chunk; // attention splits of this token: att_ns ranges of att_chunk cells
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

// Grid barrier among the consumers of all CTAs: barrier number n (1-based) completes when the
// counter reaches n * gridDim.x. Returns false (and the error word is set) if this CTA or any
// other gave up.
__device__ __forceinline__ bool grid_sync(const FwdArgs &a, unsigned *cnt, unsigned n, bool dead, int *s_ok) {
    const bool any_dead = consumer_any(dead);
    if (threadIdx.x == 0) {
        bool ok = !any_dead;
        if (ok) {
            // release: this CTA's writes (ordered before by the barrier above) become visible
            // to the CTAs whose acquire load sees the count
            asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(cnt) : "memory");
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
__device__ __forceinline__ void attn_prefetch(const FwdArgs &a, int layer, int kvh, int c0, int c1) {
    constexpr int LINES = HD * 2 / 128;   // 128-byte lines of one K (or V) row
    const int seq = a.ub.seq[0];
    const int n_att = a.ub.pos[0] + 1;
    c1 = min(min(c1, n_att - 1), c0 + 512);
    const int32_t *ptrow = a.pt + (size_t)seq * a.max_pages_per_seq;
    for (int i = threadIdx.x; i < (c1 - c0) * 2 * LINES; i += 256) {
        const int j = c0 + i / (2 * LINES), w = i % (2 * LINES);
        const int page = __ldcg(ptrow + j / kPage);
        const size_t row = (((size_t)layer * a.n_pages + page) * a.KV + kvh) * kPage + (j % kPage);
        const __half *base = (w < LINES ? a.kc : a.vc) + row * HD + (w % LINES) * 64;
        asm volatile("prefetch.global.L2 [%0];" ::"l"(base));
    }
}

// K/V of one 16-cell super-group of a warp, in registers: lanes 8c..8c+7 hold dims of cell
// 4 g4 + c of K (DPL = HD / 8 per lane), lane l holds dims l * HD / 32.. of every V row.
template <int HD>
struct AttnRegs {
    uint4 kraw[4][HD / 64];
    uint2 vraw[16];
};

// Loads the super-group of 16 cells at j0 (inside one page) of KV head kvh, cells >= c1 as
// zeros; only_fresh re-reads just the cells at positions >= fresh (written by this step).
template <int HD>
__device__ __forceinline__ void attn_load_sg(const FwdArgs &a, int layer, int kvh, int j0, int c1, int fresh,
                                             bool only_fresh, AttnRegs<HD> &R) {
    constexpr int DPL = HD / 8, DPV = HD / 32;
    const int lane = threadIdx.x & 31, sub = lane & 7, cgrp = lane >> 3;
    if (j0 >= c1) return;
    const int32_t *ptrow = a.pt + (size_t)a.ub.seq[0] * a.max_pages_per_seq;
    const int page = __ldcg(ptrow + j0 / kPage);
    const size_t row0 = (((size_t)layer * a.n_pages + page) * a.KV + kvh) * kPage + (j0 % kPage);
#pragma unroll
    for (int g4 = 0; g4 < 4; ++g4) {
        const int j = j0 + 4 * g4 + cgrp;
        if (only_fresh && j < fresh) continue;
        const __half *kp = a.kc + (row0 + 4 * g4 + cgrp) * HD + sub * DPL;
#pragma unroll
        for (int i = 0; i < DPL / 8; ++i)
            R.kraw[g4][i] = j < c1 ? __ldcg(reinterpret_cast<const uint4 *>(kp + 8 * i)) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int c = 0; c < 16; ++c) {
        if (only_fresh && j0 + c < fresh) continue;
        const __half *vp = a.vc + (row0 + c) * HD + lane * DPV;
        if (j0 + c < c1) {
            if (DPV == 4) R.vraw[c] = __ldcg(reinterpret_cast<const uint2 *>(vp));
            else R.vraw[c] = make_uint2(__ldcg(reinterpret_cast<const unsigned int *>(vp)), 0u);
        } else {
            R.vraw[c] = make_uint2(0u, 0u);
        }
    }
}

// One attention unit: query token 0 against cells [c0, c1) of KV head kvh, by the 8 consumer
// warps (the math of k_attn with 8 warps instead of 4): warp w takes the super-groups at
// c0 + 16 w + 128 i, the first of them already in R (loaded before this step's K/V were
// appended; the appended cell is re-read here). With one split the result goes to o32;
// otherwise the partial (max, sum, acc) is written and the last CTA of the KV head to arrive
// merges the splits in order. scr: shared scratch of at least attn_scratch_bytes(HD, G).
template <int HD, int G>
__device__ __forceinline__ void attn_unit(const FwdArgs &a, int layer, int kvh, int sp, int chunk, int ns, float *scr,
                                          AttnRegs<HD> &R, int trace_phase) {
    constexpr int NW = 8, DPL = HD / 8, DPV = HD / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int n_att = a.ub.pos[0] + 1;
    const int c0 = sp * chunk, c1 = min(c0 + chunk, n_att);
    const int sub = lane & 7, cgrp = lane >> 3;
    const float scale = rsqrtf((float)HD);
    const int j_first = c0 + 16 * warp;
    if (j_first < c1 && j_first + 16 > n_att - 1) attn_load_sg<HD>(a, layer, kvh, j_first, c1, n_att - 1, true, R);

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
    for (int j0 = j_first; j0 < c1; j0 += 16 * NW) {
        if (j0 != j_first) attn_load_sg<HD>(a, layer, kvh, j0, c1, 0, false, R);
#pragma unroll
        for (int g4 = 0; g4 < 4; ++g4) {
            if (j0 + 4 * g4 >= c1) break;
            const int j = j0 + 4 * g4 + cgrp;
            const bool valid = j < c1;
            float s[G];
            {
                float kf[DPL];
#pragma unroll
                for (int i = 0; i < DPL / 8; ++i) {
                    const __half2 *h2 = reinterpret_cast<const __half2 *>(&R.kraw[g4][i]);
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
                    s[g] = valid ? d : -CUDART_INF_F;
                }
            }
            float p[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float mx = s[g];
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                const float mn = fmaxf(m[g], mx);
                const float alpha = expf(m[g] - mn);
                p[g] = expf(s[g] - mn);
                float ps = p[g];
                ps += __shfl_xor_sync(0xffffffffu, ps, 8);
                ps += __shfl_xor_sync(0xffffffffu, ps, 16);
                l[g] = l[g] * alpha + ps;
                m[g] = mn;
#pragma unroll
                for (int i = 0; i < DPV; ++i) acc[g][i] *= alpha;
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if (j0 + 4 * g4 + c >= c1) break;
                const uint2 raw = R.vraw[4 * g4 + c];
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
    }

    // ---- merge the 8 warps
    float *sm_m = scr, *sm_l = scr + NW * G, *sm_acc = scr + 2 * NW * G;   // [NW][G], [NW][G], [NW][G][HD]
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
    float *part = a.att_part;
    const size_t prow = (size_t)kvh * ns;   // partial rows of this KV head (token 0)
    for (int idx = threadIdx.x; idx < G * HD; idx += 256) {
        const int g = idx / HD, dd = idx % HD;
        float M = -CUDART_INF_F;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, sm_m[w * G + g]);
        float L = 0.f, A = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const float mw = sm_m[w * G + g];
            const float f = mw == -CUDART_INF_F ? 0.f : expf(mw - M);
            L += sm_l[w * G + g] * f;
            A += sm_acc[(w * G + g) * HD + dd] * f;
        }
        if (ns == 1) {
            a.o32[(size_t)(kvh * G + g) * HD + dd] = A / L;
        } else {
            float *pr = part + ((prow + sp) * G + g) * (HD + 2);
            pr[2 + dd] = A;
            if (dd == 0) {
                pr[0] = M;
                pr[1] = L;
            }
        }
    }
    step_trace(a, trace_phase, 1);
    step_trace(a, trace_phase, 2);
    if (ns == 1) return;

    // ---- split merge by the last CTA of this KV head to arrive: the barrier orders the CTA's
    // partial stores before thread 0's acq_rel arrival, which publishes them and, for the last
    // CTA, acquires the others'
    int *last = reinterpret_cast<int *>(sm_m);   // sm_m is no longer read after the barrier below
    consumer_sync();
    if (threadIdx.x == 0) {
        unsigned prev;
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(prev) : "l"(a.att_cnt + kvh) : "memory");
        *last = prev == (unsigned)(ns - 1);
    }
    consumer_sync();
    if (!*last) return;
    // every thread's partial sums first (up to 32 splits in flight at once), then the weights
    // w_s = exp(M_s - M*) / L* per query head (one warp per head, lanes over splits)
    constexpr int PER = (G * HD + 255) / 256;   // outputs per thread
    float av[PER][32];
    for (int s0 = 0; s0 < ns; s0 += 32) {
#pragma unroll
        for (int q = 0; q < PER; ++q) {
            const int idx = threadIdx.x + 256 * q;
            const int g = idx / HD, dd = idx % HD;
#pragma unroll
            for (int u = 0; u < 32; ++u)
                av[q][u] = idx < G * HD && s0 + u < ns ? __ldcg(part + ((prow + s0 + u) * G + g) * (HD + 2) + 2 + dd) : 0.f;
        }
        if (s0 == 0) {
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
                    e[h] = lane + 32 * h < ns ? expf(ms[h] - M) : 0.f;
                    L += e[h] * ls[h];
                }
#pragma unroll
                for (int o = 16; o; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    if (lane + 32 * h < ns) sw[(lane + 32 * h) * G + g] = e[h] / L;
            }
            consumer_sync();
        }
#pragma unroll
        for (int q = 0; q < PER; ++q) {
            const int idx = threadIdx.x + 256 * q;
            if (idx >= G * HD) continue;
            const int g = idx / HD, dd = idx % HD;
            float *o = a.o32 + (size_t)(kvh * G + g) * HD + dd;
            float acc_o = s0 == 0 ? 0.f : *o;
#pragma unroll
            for (int u = 0; u < 32; ++u)
                if (s0 + u < ns) acc_o = fmaf(sm_acc[(s0 + u) * G + g], av[q][u], acc_o);
            *o = acc_o;
        }
    }
    if (threadIdx.x == 0) a.att_cnt[kvh] = 0;
}

__host__ __device__ constexpr int attn_scratch_bytes(int hd, int g) { return (2 * 8 * g + 8 * g * hd) * 4; }

// The ring's refill cursor (used by one thread, kFeedThread): the next stage of the step's
// sequence -- phase `ph`, stage `st` of it -- and the number of stages issued so far.
constexpr int kFeedThread = 255;
struct Feeder {
    int ph, st, issued;
};

// Issues the cursor's stage into ring slot issued % slots and advances the cursor; nothing once
// the sequence is exhausted.
template <int QL, int QH>
__device__ __forceinline__ void feed_one(const StepArgs &s, int n_ph, int L, Feeder &f, uint8_t *ring, uint64_t *full) {
    while (f.ph < n_ph && f.st >= s.ph[f.ph].n_stages) {
        ++f.ph;
        f.st = blockIdx.x;
    }
    if (f.ph >= n_ph) return;
    const StepPhase &P = s.ph[f.ph];
    const bool head = f.ph == 4 * L;
    const int slot = f.issued % s.slots;
    uint8_t *dst = ring + (size_t)slot * s.slot_bytes;
    if (!head && f.ph % 4 == PH_GU) issue_stage<EPI_SWIGLU>(P.p, P.pl, f.st, dst, &full[slot]);
    else issue_stage<EPI_RESID>(P.p, P.pl, f.st, dst, &full[slot]);
    f.st += gridDim.x;
    ++f.issued;
}

// One weight-streaming phase: stage the input vector, then consume this CTA's stages of the
// matrix from the ring (k counts ring uses over the whole step), refilling each slot.
template <int QL, int QH, int QT, int EPI>
__device__ __forceinline__ void gemv_phase(const StepArgs &s, const StepPhase &P, const FwdArgs &a, int layer,
                                           uint8_t *xs, uint8_t *ring, uint64_t *full, int &k, Feeder &f, int n_ph,
                                           bool &dead, PartBuf<1> &part, float (*red)[8],
                                           unsigned long long (&best)[1], int trace_phase,
                                           const float4 (*gpre)[4] = nullptr) {
    if (!dead) stage_token<QT>(P.p, 0, xs, red, 2 * P.p.nb <= kStageThreads ? gpre : nullptr);
    consumer_sync();
    step_trace(a, trace_phase, 1);
    step_trace(a, trace_phase, 2);
    for (int st = blockIdx.x; st < P.n_stages; st += gridDim.x, ++k) {
        const int slot = k % s.slots;
        if (!dead && !mbar_wait(&full[slot], (k / s.slots) & 1)) {
            dead = true;
            atomicExch(a.err, 1);
        }
        consume_stage<QT, 1, EPI, false>(P.p, a, layer, P.pl, ring + (size_t)slot * s.slot_bytes, xs, st, k, dead,
                                         nullptr, part, red, best);
        // every warp is past its reads of the slot (the barrier inside consume_stage): refill it
        if (threadIdx.x == kFeedThread && !dead) feed_one<QL, QH>(s, n_ph, a.L, f, ring, full);
    }
    step_trace(a, trace_phase, 3);
}

template <int QL, int QH, int HD, int G>
__global__ void __launch_bounds__(256, 1) k_decode_step(const StepArgs s, const FwdArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *xs = smem;
    uint8_t *ring = smem + s.x_bytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(ring + (size_t)s.slots * s.slot_bytes);
    const int L = a.L;
    const int n_ph = 4 * L + (a.n_out > 0 ? 1 : 0);

    if (threadIdx.x == 0) {
        for (int i = 0; i < s.slots; ++i) mbar_init(&full[i], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // fill the ring: the weights do not depend on anything this step computes
    Feeder f{0, (int)blockIdx.x, 0};
    if (threadIdx.x == kFeedThread)
        for (int i = 0; i < s.slots; ++i) feed_one<QL, QH>(s, n_ph, L, f, ring, full);

    __shared__ float red[1][8];
    __shared__ PartBuf<1> part;
    __shared__ int s_ok;
    unsigned long long best[1] = {0ull};
    unsigned *bar = s.sync;
    unsigned n_bar = 0;
    int k = 0;
    bool dead = false;
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
    AttnRegs<HD> R;
    // the norm gains of the next phase that has them, loaded before the barrier it waits on
    float4 gpre[4];
    stage_gains(s.ph[0].p.in.g, s.ph[0].p.nb, gpre);
    dead = !grid_sync(a, bar, ++n_bar, dead, &s_ok);

    for (int l = 0; l < L && !dead; ++l) {
        const int tp = 1 + 5 * l;
        const StepPhase &Pq = s.ph[4 * l + PH_QKV], &Po = s.ph[4 * l + PH_O], &Pg = s.ph[4 * l + PH_GU],
                        &Pd = s.ph[4 * l + PH_DOWN];
        // QKV (the attention unit's cached K/V lines go to L2 meanwhile)
        step_trace(a, tp, 0);
        if (has_unit) attn_prefetch<HD>(a, l, u_kvh, ac0, ac1);
        gemv_phase<QL, QH, QL, EPI_QKV>(s, Pq, a, l, xs, ring, full, k, f, n_ph, dead, part, red, best, tp, &gpre);
        if (has_unit) attn_load_sg<HD>(a, l, u_kvh, ac0 + 16 * (threadIdx.x >> 5), ac1, 0, false, R);
        dead = !grid_sync(a, bar, ++n_bar, dead, &s_ok);
        if (dead) break;
        // attention
        step_trace(a, tp + 1, 0);
        if (has_unit) attn_unit<HD, G>(a, l, u_kvh, u_sp, s.att_chunk, s.att_ns, reinterpret_cast<float *>(xs), R, tp + 1);
        step_trace(a, tp + 1, 3);
        dead = !grid_sync(a, bar, ++n_bar, dead, &s_ok);
        if (dead) break;
        // output projection + residual
        step_trace(a, tp + 2, 0);
        gemv_phase<QL, QH, QL, EPI_RESID>(s, Po, a, l, xs, ring, full, k, f, n_ph, dead, part, red, best, tp + 2);
        stage_gains(Pg.p.in.g, Pg.p.nb, gpre);
        dead = !grid_sync(a, bar, ++n_bar, dead, &s_ok);
        if (dead) break;
        // gate/up + SwiGLU
        step_trace(a, tp + 3, 0);
        gemv_phase<QL, QH, QL, EPI_SWIGLU>(s, Pg, a, l, xs, ring, full, k, f, n_ph, dead, part, red, best, tp + 3, &gpre);
        dead = !grid_sync(a, bar, ++n_bar, dead, &s_ok);
        if (dead) break;
        // down + residual
        step_trace(a, tp + 4, 0);
        gemv_phase<QL, QH, QL, EPI_RESID>(s, Pd, a, l, xs, ring, full, k, f, n_ph, dead, part, red, best, tp + 4);
        const StepPhase &Pn = s.ph[4 * l + 4];   // next layer's QKV, or the head
        stage_gains(Pn.p.in.g, Pn.p.nb, gpre);
        dead = !grid_sync(a, bar, ++n_bar, dead, &s_ok);
    }
    if (dead) {
        // copies still in flight must land before the CTA's shared memory is released
        if (threadIdx.x == kFeedThread)
            for (int j = f.issued > s.slots ? f.issued - s.slots : 0; j < f.issued; ++j)
                mbar_wait(&full[j % s.slots], (j / s.slots) & 1);
        return;
    }
    if (a.n_out > 0) {
        const int tp = 1 + 5 * L;
        step_trace(a, tp, 0);
        gemv_phase<QL, QH, QH, EPI_LOGITS>(s, s.ph[4 * L], a, -1, xs, ring, full, k, f, n_ph, dead, part, red, best, tp, &gpre);
        logits_cta_reduce<1>(a, 1, best);
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
        }
    }
}

}  // namespace step_detail
}  // namespace lcx
