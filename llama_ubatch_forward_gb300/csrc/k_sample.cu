// The sampler chain on the device: one CTA per logits row picks that row's token.
//
// Sampling (article, "Sampler chain", after step 14 on llama_get_logits_ith) is a chain of steps
// over one row of logits: a repeat penalty on the tokens that already appeared; the cut-offs
// top-k (the k largest logits), top-p (the tokens whose accumulated probability reaches p) and
// min-p (drop what lies far below the leader); temperature; then one token -- the leader
// (greedy) or a random draw with the softmax probabilities of what is left. The article notes
// that a backend may run the sampler itself and hand back only the token: this kernel is that,
// the row never leaves the GPU.
//
// Every cut-off keeps a prefix of one order -- larger logit first, lower token id first among
// equal logits -- so the survivors of the whole chain are the tokens whose 64-bit key
//   (order-preserving bits of the penalised logit) << 32 | (0xffffffff - id)
// reaches one threshold: the largest of the thresholds the cut-offs find. Each threshold comes
// from a radix select (8-bit digits of the logit bits, most significant first): by count for
// top-k, by probability mass for top-p; ties on the logit are settled by id with one scan in id
// order. The draw is one scan of the survivors' weights in id order.
//
// With a top-k of at most kCap, the pass that finds the leader also builds a 4096-bin histogram
// of the top 12 key bits; the tokens in the bins at and above the k-th largest -- every top-k
// survivor, usually a few dozen -- are compacted in id order into shared memory, and the rest of
// the chain runs there. Otherwise every step re-reads the row from L2 (a 128k-entry row is
// 513 KB). Row passes keep 8 loads in flight per thread: one CTA streams the row alone, so the
// pass time is the L2 latency divided by the loads in flight.
#include <math.h>

#include "../../include/lcx.h"
#include "lcx_internal.h"

namespace lcx {
void set_error_text(const char *msg);

namespace smp {

constexpr int NT = 1024;
constexpr int NWARP = NT / 32;
constexpr int kMaxVocab = 1 << 18;   // the penalty bitmap takes kMaxVocab / 8 bytes of shared memory
constexpr int kBatch = 8;            // loads in flight per thread in a row pass
constexpr unsigned FULL = 0xffffffffu;

struct Smem {
    uint32_t pen[kMaxVocab / 32];   // tokens of the history (bitmap)
    uint32_t hc[256];               // radix bins: counts
    float hm[256];                  // radix bins: probability mass
    float excl[NT + 1];             // id-order scan: weight before each thread's chunk, then the total
    float wf[NWARP];
    unsigned long long wu[NWARP];
    int first, res, lastid;
    uint32_t digit, cabove, eqc;
    float above;
};

// One row of logits with the repeat penalty applied on the fly: a history token's logit is
// divided by the penalty when positive and multiplied by it otherwise (IEEE round to nearest).
struct Row {
    const float *l;
    int V;
    const uint32_t *pen;   // null: no penalty
    float r;
    __device__ __forceinline__ float apply(int i, float x) const {
        if (pen && ((pen[i >> 5] >> (i & 31)) & 1u)) x = x > 0.f ? __fdiv_rn(x, r) : __fmul_rn(x, r);
        return x;
    }
    // f(i, value) for this thread's share of the row (i = threadIdx.x + k * NT)
    template <class F>
    __device__ __forceinline__ void foreach(F f) const {
        for (int base = threadIdx.x; base < V; base += kBatch * NT) {
            float x[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int i = base + u * NT;
                x[u] = i < V ? __ldg(l + i) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int i = base + u * NT;
                if (i < V) f(i, apply(i, x[u]));
            }
        }
    }
    // f(i, value) for i in [i0, i1) in increasing order
    template <class F>
    __device__ __forceinline__ void run(int i0, int i1, F f) const {
        for (int base = i0; base < i1; base += kBatch) {
            float x[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) x[u] = base + u < i1 ? __ldg(l + base + u) : 0.f;
#pragma unroll
            for (int u = 0; u < kBatch; ++u)
                if (base + u < i1) f(base + u, apply(base + u, x[u]));
        }
    }
};

// order-preserving unsigned image of a float (-0 and +0 map to the same key)
__device__ __forceinline__ uint32_t vkey(float f) {
    const uint32_t b = f == 0.f ? 0u : __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float vkey_val(uint32_t k) { return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k); }
__device__ __forceinline__ uint64_t ckey(uint32_t vk, int id) {
    return ((uint64_t)vk << 32) | (uint64_t)(0xffffffffu - (uint32_t)id);
}
__device__ __forceinline__ int ckey_id(uint64_t c) { return (int)(0xffffffffu - (uint32_t)c); }

// What the selection steps run over: the whole row (position = token id), or the candidate
// list compacted in shared memory in increasing id order. foreach(f) calls f(position, value)
// for this thread's share; run(j0, j1, f) for positions j0..j1-1 in order.
struct RowSrc {
    Row row;
    __device__ __forceinline__ int n() const { return row.V; }
    __device__ __forceinline__ int id(int j) const { return j; }
    template <class F>
    __device__ __forceinline__ void foreach(F f) const { row.foreach(f); }
    template <class F>
    __device__ __forceinline__ void run(int j0, int j1, F f) const { row.run(j0, j1, f); }
};
struct ListSrc {
    const float *v;
    const int *ids;
    int cnt;
    __device__ __forceinline__ int n() const { return cnt; }
    __device__ __forceinline__ int id(int j) const { return ids[j]; }
    template <class F>
    __device__ __forceinline__ void foreach(F f) const {
        for (int j = threadIdx.x; j < cnt; j += NT) f(j, v[j]);
    }
    template <class F>
    __device__ __forceinline__ void run(int j0, int j1, F f) const {
        for (int j = j0; j < j1; ++j) f(j, v[j]);
    }
};

// ------------------------------------------------------------------ block primitives (all 1024 threads)
__device__ __forceinline__ float block_sum(float v, Smem &s) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
    if (lane == 0) s.wf[warp] = v;
    __syncthreads();
    float t = 0.f;
    for (int w = 0; w < NWARP; ++w) t += s.wf[w];   // the same order in every thread
    __syncthreads();
    return t;
}

__device__ __forceinline__ unsigned long long block_max(unsigned long long v, Smem &s) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        const unsigned long long y = __shfl_xor_sync(FULL, v, o);
        v = y > v ? y : v;
    }
    if (lane == 0) s.wu[warp] = v;
    __syncthreads();
    unsigned long long t = 0;
    for (int w = 0; w < NWARP; ++w) t = s.wu[w] > t ? s.wu[w] : t;
    __syncthreads();
    return t;
}

// exclusive scan of one float per thread in thread order; *total = the sum of all
__device__ __forceinline__ float block_excl_scan(float v, Smem &s, float *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float inc = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const float y = __shfl_up_sync(FULL, inc, d);
        if (lane >= d) inc += y;
    }
    float ex = __shfl_up_sync(FULL, inc, 1);
    if (lane == 0) ex = 0.f;
    if (lane == 31) s.wf[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        const float w = s.wf[lane];
        float wi = w;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const float y = __shfl_up_sync(FULL, wi, d);
            if (lane >= d) wi += y;
        }
        float we = __shfl_up_sync(FULL, wi, 1);
        if (lane == 0) we = 0.f;
        s.wf[lane] = we;
        if (lane == 31) s.excl[NT] = wi;
    }
    __syncthreads();
    const float out = s.wf[warp] + ex;
    *total = s.excl[NT];
    __syncthreads();
    return out;
}

// The first position (in increasing id order) at which the running sum of the weights w(j, value)
// reaches the target (`strict`: exceeds it); target = frac * total when `of_total`. Each thread
// takes a contiguous chunk; the chunk holding the crossing is found from the scan of the chunk
// sums and walked again. If rounding leaves no crossing, the last position with a positive
// weight; -1 if there is none.
template <class Src, class W>
__device__ int id_crossing(const Src &src, W w, float target, bool of_total, bool strict, Smem &s) {
    const int n = src.n();
    const int CH = (n + NT - 1) / NT;
    const int j0 = min(n, (int)threadIdx.x * CH), j1 = min(n, j0 + CH);
    float sum = 0.f;
    int last = -1;
    src.run(j0, j1, [&](int j, float v) {
        const float x = w(j, v);
        sum += x;
        if (x > 0.f) last = j;
    });
    float total;
    const float ex = block_excl_scan(sum, s, &total);
    if (of_total) target *= total;
    s.excl[threadIdx.x] = ex;
    if (threadIdx.x == 0) {
        s.first = NT;
        s.lastid = -1;
    }
    __syncthreads();
    auto cross = [&](float x) { return strict ? x > target : x >= target; };
    if (cross(threadIdx.x + 1 < NT ? s.excl[threadIdx.x + 1] : total)) atomicMin(&s.first, (int)threadIdx.x);
    if (last >= 0) atomicMax(&s.lastid, last);
    __syncthreads();
    if ((int)threadIdx.x == s.first) {
        float r = ex;
        int found = -1;
        src.run(j0, j1, [&](int j, float v) {
            const float x = w(j, v);
            r += x;
            if (found < 0 && x > 0.f && cross(r)) found = j;
        });
        s.res = found >= 0 ? found : last;
    }
    __syncthreads();
    const int out = s.first < NT ? s.res : s.lastid;
    __syncthreads();
    return out;
}

// Warp 0: the digit of the radix pass -- scanning the 256 bins from the top, the bin where the
// count reaches krem; its count-above and its own count go to shared memory.
__device__ __forceinline__ void digit_by_count(Smem &s, uint32_t krem) {
    const int lane = threadIdx.x & 31;
    uint32_t c = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) c += s.hc[255 - 8 * lane - j];
    uint32_t inc = c;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t y = __shfl_up_sync(FULL, inc, d);
        if (lane >= d) inc += y;
    }
    const uint32_t ex = inc - c;
    const unsigned bal = __ballot_sync(FULL, ex < krem && krem <= inc);
    const int L = bal ? __ffs(bal) - 1 : 31;   // the source always holds krem matching elements
    if (lane == L) {
        uint32_t acc = ex;
        s.digit = 255 - 8 * lane - 7;
        s.cabove = acc;
        s.eqc = 0;
        for (int j = 0; j < 8; ++j) {
            const int b = 255 - 8 * lane - j;
            if (acc + s.hc[b] >= krem) {
                s.digit = (uint32_t)b;
                s.cabove = acc;
                s.eqc = s.hc[b];
                break;
            }
            acc += s.hc[b];
        }
    }
}

// Warp 0: as digit_by_count over the probability mass, for the target t. Rounding may leave no
// bin where the mass reaches t: then the lowest non-empty bin (the whole remaining mass).
__device__ __forceinline__ void digit_by_mass(Smem &s, float t) {
    const int lane = threadIdx.x & 31;
    float m = 0.f;
    uint32_t c = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        m += s.hm[255 - 8 * lane - j];
        c += s.hc[255 - 8 * lane - j];
    }
    float inc = m;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const float y = __shfl_up_sync(FULL, inc, d);
        if (lane >= d) inc += y;
    }
    float ex = __shfl_up_sync(FULL, inc, 1);
    if (lane == 0) ex = 0.f;
    const unsigned cross = __ballot_sync(FULL, c > 0 && ex < t && t <= inc);
    const unsigned nonempty = __ballot_sync(FULL, c > 0);
    const int L = cross ? __ffs(cross) - 1 : (nonempty ? 31 - __clz(nonempty) : 0);
    if (lane == L) {
        float acc = ex;
        uint32_t lb = 255 - 8 * lane, lc = 0;
        float la = acc;
        bool done = false;
        for (int j = 0; j < 8 && !done; ++j) {
            const int b = 255 - 8 * lane - j;
            if (s.hc[b] > 0) {
                lb = (uint32_t)b;
                la = acc;
                lc = s.hc[b];
                if (acc + s.hm[b] >= t) done = true;
            }
            acc += s.hm[b];
        }
        s.digit = lb;
        s.above = la;
        s.eqc = lc;
    }
}

// top-k: the key threshold that keeps exactly k of the source's tokens (k < n)
template <class Src>
__device__ uint64_t select_by_count(const Src &src, int k, Smem &s) {
    uint32_t prefix = 0, eq = 0;
    uint32_t krem = (uint32_t)k;
    for (int pass = 0; pass < 4; ++pass) {
        const int sh = 24 - 8 * pass;
        const uint32_t hmask = pass == 0 ? 0u : (0xffffffffu << (sh + 8));
        for (int b = threadIdx.x; b < 256; b += NT) s.hc[b] = 0u;
        __syncthreads();
        src.foreach([&](int, float v) {
            const uint32_t kv = vkey(v);
            if ((kv & hmask) == prefix) atomicAdd(&s.hc[(kv >> sh) & 255u], 1u);
        });
        __syncthreads();
        if (threadIdx.x < 32) digit_by_count(s, krem);
        __syncthreads();
        prefix |= s.digit << sh;
        krem -= s.cabove;
        eq = s.eqc;
        __syncthreads();
    }
    if (krem >= eq) return (uint64_t)prefix << 32;   // every token with this logit is kept
    const int j = id_crossing(
        src, [&](int, float v) { return vkey(v) == prefix ? 1.f : 0.f; }, (float)krem, false, false, s);
    return j >= 0 ? ckey(prefix, src.id(j)) : (uint64_t)prefix << 32;
}

// top-p: the key threshold of the shortest prefix (of the tokens at or above `thr`) whose mass
// exp(l - m) reaches `target`
template <class Src>
__device__ uint64_t select_by_mass(const Src &src, uint64_t thr, float m, float target, Smem &s) {
    uint32_t prefix = 0, eq = 0;
    float t = target;
    for (int pass = 0; pass < 4; ++pass) {
        const int sh = 24 - 8 * pass;
        const uint32_t hmask = pass == 0 ? 0u : (0xffffffffu << (sh + 8));
        for (int b = threadIdx.x; b < 256; b += NT) {
            s.hc[b] = 0u;
            s.hm[b] = 0.f;
        }
        __syncthreads();
        src.foreach([&](int j, float v) {
            const uint32_t kv = vkey(v);
            if ((kv & hmask) == prefix && ckey(kv, src.id(j)) >= thr) {
                const uint32_t b = (kv >> sh) & 255u;
                atomicAdd(&s.hc[b], 1u);
                atomicAdd(&s.hm[b], expf(v - m));
            }
        });
        __syncthreads();
        if (threadIdx.x < 32) digit_by_mass(s, t);
        __syncthreads();
        prefix |= s.digit << sh;
        t -= s.above;
        eq = s.eqc;
        __syncthreads();
    }
    if (eq <= 1) return (uint64_t)prefix << 32;
    const int j = id_crossing(
        src,
        [&](int j, float v) {
            const uint32_t kv = vkey(v);
            return kv == prefix && ckey(kv, src.id(j)) >= thr ? expf(v - m) : 0.f;
        },
        t, false, false, s);
    return j >= 0 ? ckey(prefix, src.id(j)) : (uint64_t)prefix << 32;
}

// The chain after top-k (threshold thr): top-p and min-p on the survivors, then temperature and
// the draw (weights exp((l - m) / temp), walked in increasing id). best: the leader's key.
template <class Src>
__device__ int finish(const Src &src, uint64_t thr, uint64_t best, float m, const lcx_sampler &prm, float uu,
                      Smem &s) {
    if (prm.top_p < 1.f) {
        float z = 0.f;
        src.foreach([&](int j, float v) {
            if (ckey(vkey(v), src.id(j)) >= thr) z += expf(v - m);
        });
        z = block_sum(z, s);
        const uint64_t tp = select_by_mass(src, thr, m, prm.top_p * z, s);
        thr = tp > thr ? tp : thr;
    }
    if (prm.min_p > 0.f) {
        const uint64_t tm = (uint64_t)vkey(m + logf(prm.min_p)) << 32;
        thr = tm > thr ? tm : thr;
    }
    thr = thr < best ? thr : best;
    const float temp = prm.temp;
    const int j = id_crossing(
        src, [&](int j, float v) { return ckey(vkey(v), src.id(j)) >= thr ? expf((v - m) / temp) : 0.f; }, uu,
        true, true, s);
    return j >= 0 ? src.id(j) : ckey_id(best);
}

// Candidates kept in shared memory when top-k leaves few: the logits whose top 12 key bits are at
// least those of the k-th largest (so every top-k survivor), at most kCap of them. The same
// dynamic shared memory first holds the 4096-bin histogram of those 12 bits.
constexpr int kCap = 4096;
constexpr int kBins = 4096;
constexpr int kListBytes = kCap * 8;   // values, then ids (>= the histogram's kBins * 4)
static_assert(kListBytes >= kBins * 4, "the histogram shares the list's memory");
static_assert(kBins == 4 * NT, "each thread scans 4 histogram bins");

__global__ void __launch_bounds__(NT, 1) k_sample(const lcx_sampler prm, const float *__restrict__ logits, const int V,
                                                  const int32_t *__restrict__ hist, const int n_hist,
                                                  const float *__restrict__ u, int32_t *__restrict__ out) {
    __shared__ Smem s;
    extern __shared__ __align__(16) unsigned char list_mem[];
    const int r = blockIdx.x;
    Row row{logits + (size_t)r * V, V, nullptr, prm.penalty_repeat};
    // 1. repeat penalty: the history's distinct tokens, as a bitmap
    if (prm.penalty_repeat != 1.f && hist && n_hist > 0) {
        for (int i = threadIdx.x; i < (V + 31) / 32; i += NT) s.pen[i] = 0u;
        __syncthreads();
        for (int j = threadIdx.x; j < n_hist; j += NT) {
            const int t = hist[(size_t)r * n_hist + j];
            if (t >= 0 && t < V) atomicOr(&s.pen[t >> 5], 1u << (t & 31));
        }
        __syncthreads();
        row.pen = s.pen;
    }
    const bool small_k = prm.temp > 0.f && prm.top_k > 0 && prm.top_k < V && prm.top_k <= kCap;
    uint32_t *h12 = reinterpret_cast<uint32_t *>(list_mem);
    if (small_k) {
        for (int b = threadIdx.x; b < kBins; b += NT) h12[b] = 0u;
        __syncthreads();
    }
    // the leader -- every cut-off keeps it, and it is the greedy choice -- and, with a small
    // top-k, the histogram of the top 12 key bits in the same pass
    unsigned long long best = 0;
    row.foreach([&](int i, float v) {
        const uint32_t kv = vkey(v);
        const unsigned long long c = ckey(kv, i);
        best = c > best ? c : best;
        if (small_k) atomicAdd(&h12[kv >> 20], 1u);
    });
    best = block_max(best, s);
    const float m = vkey_val((uint32_t)(best >> 32));
    if (!(prm.temp > 0.f) || !isfinite(m)) {
        if (threadIdx.x == 0) out[r] = ckey_id(best);
        return;
    }
    const float uu = fminf(fmaxf(u[r], 0.f), 1.f);
    if (small_k) {
        // the bin of the k-th largest: thread t sums bins 4095 - 4t .. 4092 - 4t (from the top);
        // the exclusive scan of those sums (exact integers) finds the one thread holding it
        const int t4 = kBins - 1 - 4 * (int)threadIdx.x;
        uint32_t c4 = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) c4 += h12[t4 - j];
        float tot4;
        const uint32_t ex4 = (uint32_t)block_excl_scan((float)c4, s, &tot4);
        const uint32_t k = (uint32_t)prm.top_k;
        if (ex4 < k && k <= ex4 + c4) {
            uint32_t acc = ex4;
            for (int j = 0; j < 4; ++j) {
                const uint32_t hb = h12[t4 - j];
                if (acc + hb >= k) {
                    s.digit = (uint32_t)(t4 - j);
                    s.cabove = acc;
                    s.eqc = hb;
                    break;
                }
                acc += hb;
            }
        }
        __syncthreads();
        const uint32_t d0 = s.digit, n_cand = s.cabove + s.eqc;
        __syncthreads();
        if (n_cand <= (uint32_t)kCap) {
            // 2. the candidates, compacted in id order: each thread takes a contiguous run of ids,
            // counts its candidates, and writes them after those of the threads before it (the
            // histogram's memory is reused from here on: its last reads are before the barriers
            // of the scan below)
            float *lv = reinterpret_cast<float *>(list_mem);
            int *li = reinterpret_cast<int *>(list_mem + kCap * 4);
            const int CH = (V + NT - 1) / NT;
            const int i0 = min(V, (int)threadIdx.x * CH), i1 = min(V, i0 + CH);
            int c = 0;
            row.run(i0, i1, [&](int, float v) { c += (vkey(v) >> 20) >= d0 ? 1 : 0; });
            float tot;
            int off = (int)block_excl_scan((float)c, s, &tot);
            row.run(i0, i1, [&](int i, float v) {
                if ((vkey(v) >> 20) >= d0 && off < kCap) {
                    lv[off] = v;
                    li[off] = i;
                    ++off;
                }
            });
            __syncthreads();
            const ListSrc L{lv, li, min((int)tot, kCap)};
            const uint64_t thr = select_by_count(L, prm.top_k, s);
            const int tok = finish(L, thr, best, m, prm, uu, s);
            if (threadIdx.x == 0) out[r] = tok;
            return;
        }
    }
    // 2. the cut-offs over the whole row
    const RowSrc R{row};
    uint64_t thr = 0;
    if (prm.top_k > 0 && prm.top_k < V) thr = select_by_count(R, prm.top_k, s);
    const int tok = finish(R, thr, best, m, prm, uu, s);
    if (threadIdx.x == 0) out[r] = tok;
}

}  // namespace smp
}  // namespace lcx

extern "C" int32_t lcx_sample(const lcx_sampler *prm, const float *logits, int32_t n_rows, int32_t n_vocab,
                              const int32_t *history, int32_t n_history, const float *u, int32_t *tokens_out,
                              void *cuda_stream) {
    using namespace lcx;
    if (!prm || n_rows < 0 || n_vocab <= 0 || n_vocab > smp::kMaxVocab || n_history < 0) return LCX_INVALID;
    if (!(prm->penalty_repeat > 0.f) || !isfinite(prm->penalty_repeat)) return LCX_INVALID;
    if (n_rows == 0) return LCX_OK;   // nothing to sample: the buffers are not read
    if (!logits || !tokens_out || (n_history > 0 && !history) || (prm->temp > 0.f && !u)) return LCX_INVALID;
    cudaError_t e = cudaFuncSetAttribute(smp::k_sample, cudaFuncAttributeMaxDynamicSharedMemorySize, smp::kListBytes);
    if (e == cudaSuccess) {
        smp::k_sample<<<n_rows, smp::NT, smp::kListBytes, (cudaStream_t)cuda_stream>>>(*prm, logits, n_vocab, history,
                                                                                     n_history, u, tokens_out);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) {
        set_error_text(cudaGetErrorString(e));
        return LCX_COMPUTE_FAILED;
    }
    return LCX_OK;
}
