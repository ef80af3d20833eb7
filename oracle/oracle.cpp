/*
 * ORACLE -- test infrastructure only.
 *
 * A plain, slow, fp64 CPU implementation of the forward pass of a Llama-architecture decoder
 * over one batch, as the article "How inference works in llama.cpp" (romankryvolapov.com,
 * llama-cpp) walks through it. Only the tests, the smoke check and the bench's CPU-baseline
 * leg may load it; the product path never does. It shares no code, header or table with the
 * CUDA library: every formula below is written out from its definition.
 *
 * What it computes, token by token in batch order, over an explicit per-sequence cell store:
 *   x   = dequant(tok_embd[id])                                 (step 13b, build_inp_embd /
 *                                                                ggml_get_rows: the token's row,
 *                                                                dequantized to float)
 *   per layer (step 13c, the per-layer structure of the graph):
 *     xn  = x / sqrt(mean(x^2) + eps) * g_attn                  RMS normalisation
 *     q,k,v = Wq xn, Wk xn, Wv xn                               block-quantized projections
 *     RoPE(q), RoPE(k) at the token's position                  rotary position encoding
 *     store f16(k), f16(v) in the cell (seq, pos)               KV-cache section: the new
 *                                                                token's K and V are written
 *                                                                first, then attended
 *     o_h = sum_j softmax_j(q_h . k_j / sqrt(hd)) v_j           over every cell of the same
 *                                                                sequence with pos_j <= pos
 *                                                                (causal mask), GQA head map
 *                                                                kv = h / (n_head / n_head_kv)
 *     x  += Wo o
 *     xn  = x / sqrt(mean(x^2) + eps) * g_ffn
 *     x  += Wd (silu(Wg xn) * (Wu xn))                          SwiGLU feed-forward
 *   flagged tokens only (step 13c, output rows; step 14, logits buffer in batch order):
 *     logits = Wout (x / sqrt(mean(x^2) + eps) * g_out),  argmax (lowest index on ties)
 *
 * Batch rules (step 12, llama_batch_allocr::init and init_batch; step 13, return codes):
 *   n_tokens <= 0, a token outside [0, n_vocab), a sequence outside [0, n_seq_max), or
 *   positions of a sequence that do not continue from its last position by +1 -> -1;
 *   positions NULL -> filled from the sequence's last position + 1; logits flags NULL ->
 *   only the last token; more new cells than the cache has free -> 1, nothing committed;
 *   a flagged token whose logits are not all finite -> -3, the cells of its ubatch (consecutive
 *   chunks of n_ubatch tokens) removed again; earlier ubatches stay in the cache and their
 *   logits rows stay reported (the decode loop copies each ubatch's rows into the output buffer
 *   before it runs the next ubatch, and a failure returns from inside that loop).
 *
 * Evaluation order: a ubatch runs layer by layer over blocks of at most 256 of its tokens (the
 * way a ubatch's graph runs every layer over all its tokens, step 13c); inside a layer every
 * token's K and V are stored before any token of the block attends, and the causal mask limits
 * token t to the cells of its sequence with pos <= pos_t, so each token computes exactly what it
 * would alone. Every matrix-vector product is one sum in increasing k, whatever the block size.
 * In the last layer a token whose logits are not flagged computes only its K and V: the rest of
 * that layer feeds nothing but its own logits (step 13c, only the output rows go on to the head).
 *
 * Readings where the pages are silent (each is a choice of this implementation):
 *   Q8_0 block = fp16 d + int8 q[32], w = d*q; Q4_0 block = fp16 d + 16 bytes, element j in
 *   the low nibble of byte j and element j+16 in the high nibble, w = d*(q-8); RMS eps 1e-5;
 *   RoPE pairs adjacent elements (2i, 2i+1) with angle pos * theta^(-2i/hd); attention scale
 *   1/sqrt(hd); SiLU(a) = a / (1 + e^-a); K and V are rounded to f16 (nearest even) when
 *   stored; ffn_down rows hold n_ff rounded up to a multiple of 32, the extra inputs are 0.
 *
 * Parity pins: every function here is pinned by tests that do not call it to check itself
 * (hand-computed blocks, closed forms, invariants, brute force on tiny shapes).
 */
#include <algorithm>
#include <atomic>
#include <cmath>
#include <condition_variable>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <functional>
#include <mutex>
#include <thread>
#include <vector>

namespace {

enum { T_F16 = 1, T_Q4_0 = 2, T_Q8_0 = 8 };

/* ------------------------------------------------------------------ fp16 */
double half_to_double(uint16_t h) {
    int sign = (h >> 15) & 1, exp = (h >> 10) & 0x1f, man = h & 0x3ff;
    double v;
    if (exp == 0) v = std::ldexp((double)man, -24);                 /* subnormal: man * 2^-24 */
    else if (exp == 31) v = man ? NAN : INFINITY;
    else v = std::ldexp(1.0 + man / 1024.0, exp - 15);
    return sign ? -v : v;
}

/* Round a double to the nearest binary16 (ties to even), returned as a double. */
double round_to_half(double x) {
    if (std::isnan(x) || std::isinf(x) || x == 0.0) return x;
    double a = std::fabs(x);
    if (a >= 65520.0) return std::copysign(INFINITY, x);            /* rounds past the largest half */
    int e;
    std::frexp(a, &e);                                              /* a = f * 2^e, f in [0.5, 1) */
    int exp_unbiased = e - 1;                                       /* a in [2^exp, 2^(exp+1)) */
    if (exp_unbiased < -14) exp_unbiased = -14;                     /* subnormal spacing 2^-24 */
    double ulp = std::ldexp(1.0, exp_unbiased - 10);
    double q = a / ulp;                                             /* exact: scaling by 2^k */
    double r = std::nearbyint(q);                                   /* default mode: ties to even */
    return std::copysign(r * ulp, x);
}

/* ------------------------------------------------------------------ dequant (one row) */
/* Element i of a stored row: row is the row's first byte. */
void dequant_row(int type, const uint8_t *row, int64_t n, double *out) {
    if (type == T_F16) {
        for (int64_t i = 0; i < n; ++i) {
            uint16_t h = (uint16_t)(row[2 * i] | (row[2 * i + 1] << 8));
            out[i] = half_to_double(h);
        }
        return;
    }
    const int64_t bsz = type == T_Q8_0 ? 34 : 18;
    for (int64_t b = 0; b * 32 < n; ++b) {
        const uint8_t *blk = row + b * bsz;
        const double d = half_to_double((uint16_t)(blk[0] | (blk[1] << 8)));   /* the block's scale */
        const int64_t m = n - b * 32 < 32 ? n - b * 32 : 32;
        for (int64_t e = 0; e < m; ++e) {
            if (type == T_Q8_0) {
                out[b * 32 + e] = d * (double)(int8_t)blk[2 + e];
            } else {
                int q = e < 16 ? (blk[2 + e] & 0x0f) : (blk[2 + e - 16] >> 4);
                out[b * 32 + e] = d * (double)(q - 8);
            }
        }
    }
}

int64_t row_bytes(int type, int64_t k) {
    if (type == T_F16) return 2 * k;
    int64_t nb = (k + 31) / 32;
    return nb * (type == T_Q8_0 ? 34 : 18);
}

/* ------------------------------------------------------------------ thread pool */
class Pool {
  public:
    explicit Pool(int n) { resize(n); }
    ~Pool() { stop(); }
    void resize(int n) {
        stop();
        n_ = n < 1 ? 1 : n;
        quit_ = false;
        const uint64_t start = gen_;                       /* no job runs while resizing */
        for (int t = 1; t < n_; ++t) workers_.emplace_back([this, t, start] { loop(t, start); });
    }
    int size() const { return n_; }
    /* fn(lo, hi) over [0, n) in n_ contiguous chunks; the caller runs chunk 0. Fewer than
     * min_n items run on the calling thread alone. */
    void parallel_for(int64_t n, const std::function<void(int64_t, int64_t)> &fn, int64_t min_n = 64) {
        if (n_ == 1 || n < min_n) { fn(0, n); return; }
        {
            std::unique_lock<std::mutex> lk(m_);
            job_ = &fn; total_ = n; pending_ = n_ - 1; ++gen_;
        }
        cv_.notify_all();
        run_chunk(0);
        std::unique_lock<std::mutex> lk(m_);
        done_cv_.wait(lk, [this] { return pending_ == 0; });
        job_ = nullptr;
    }

  private:
    void run_chunk(int t) {
        int64_t chunk = (total_ + n_ - 1) / n_, lo = t * chunk, hi = lo + chunk < total_ ? lo + chunk : total_;
        if (lo < hi) (*job_)(lo, hi);
    }
    void loop(int t, uint64_t seen) {
        for (;;) {
            {
                std::unique_lock<std::mutex> lk(m_);
                cv_.wait(lk, [&] { return quit_ || gen_ != seen; });
                if (quit_) return;
                seen = gen_;
            }
            run_chunk(t);
            std::unique_lock<std::mutex> lk(m_);
            if (--pending_ == 0) done_cv_.notify_one();
        }
    }
    void stop() {
        { std::unique_lock<std::mutex> lk(m_); quit_ = true; }
        cv_.notify_all();
        for (auto &w : workers_) w.join();
        workers_.clear();
    }
    int n_ = 1;
    std::vector<std::thread> workers_;
    std::mutex m_;
    std::condition_variable cv_, done_cv_;
    const std::function<void(int64_t, int64_t)> *job_ = nullptr;
    int64_t total_ = 0;
    int pending_ = 0;
    uint64_t gen_ = 0;
    bool quit_ = false;
};

Pool &pool() { static Pool p(1); return p; }

/* ------------------------------------------------------------------ ops */
/* Y[t][n] = sum_k W[n][k] X[t][k] for the T rows of X: W stored row-major (row n = the K inputs
 * of output n), X [T][K] and Y [T][N] row-major. Every output is one sum in increasing k of
 * products rounded before they are added (no fused multiply-add), so it does not depend on T or
 * on the thread count. A row is dequantized once per group of 8 tokens (the last tokens of X, fewer
 * than 8, one by one). */
template <int G>
void matmat_group(const double *w, int64_t K, const double *xg, double *s) {
    for (int j = 0; j < G; ++j) s[j] = 0.0;
    for (int64_t k = 0; k < K; ++k)
        for (int j = 0; j < G; ++j) s[j] += w[k] * xg[k * G + j];
}

void matmat(int type, const uint8_t *W, int64_t N, int64_t K, const double *X, int64_t T, double *Y) {
    constexpr int G = 8;
    const int64_t rb = row_bytes(type, K);
    pool().parallel_for(N, [&](int64_t lo, int64_t hi) {
        std::vector<double> w(K), xg((size_t)K * G);
        for (int64_t t0 = 0; t0 < T;) {
            const int g = T - t0 >= G ? G : 1;
            for (int64_t k = 0; k < K; ++k)               /* the group's inputs, side by side per k */
                for (int j = 0; j < g; ++j) xg[k * g + j] = X[(t0 + j) * K + k];
            for (int64_t n = lo; n < hi; ++n) {
                dequant_row(type, W + n * rb, K, w.data());
                double s[G];
                if (g == G) matmat_group<G>(w.data(), K, xg.data(), s);
                else matmat_group<1>(w.data(), K, xg.data(), s);
                for (int j = 0; j < g; ++j) Y[(t0 + j) * N + n] = s[j];
            }
            t0 += g;
        }
    });
}

/* y[n] = sum_k W[n][k] x[k]: one token of matmat. */
void matvec(int type, const uint8_t *W, int64_t N, int64_t K, const double *x, double *y) {
    matmat(type, W, N, K, x, 1, y);
}

void rmsnorm(const double *x, int64_t n, const float *g, double eps, double *y) {
    double ss = 0.0;
    for (int64_t i = 0; i < n; ++i) ss += x[i] * x[i];
    double r = std::sqrt(ss / (double)n + eps);
    for (int64_t i = 0; i < n; ++i) y[i] = x[i] / r * (double)g[i];
}

/* Rotate adjacent pairs of one head vector by pos * theta^(-2i/hd). */
void rope(double *x, int hd, int64_t pos, double theta) {
    for (int i = 0; i < hd / 2; ++i) {
        double freq = std::pow(theta, -2.0 * i / (double)hd);
        double a = (double)pos * freq, c = std::cos(a), s = std::sin(a);
        double x0 = x[2 * i], x1 = x[2 * i + 1];
        x[2 * i] = x0 * c - x1 * s;
        x[2 * i + 1] = x0 * s + x1 * c;
    }
}

double silu(double a) { return a / (1.0 + std::exp(-a)); }

/* One query head against n keys/values (each hd long, stride ld between cells). */
void attend_head(const double *q, const double *K, const double *V, int64_t n, int64_t ld, int hd, double *o) {
    std::vector<double> s(n);
    double scale = 1.0 / std::sqrt((double)hd), mx = -INFINITY;
    for (int64_t j = 0; j < n; ++j) {
        double d = 0.0;
        for (int e = 0; e < hd; ++e) d += q[e] * K[j * ld + e];
        s[j] = d * scale;
        if (s[j] > mx) mx = s[j];
    }
    double den = 0.0;
    for (int64_t j = 0; j < n; ++j) { s[j] = std::exp(s[j] - mx); den += s[j]; }
    for (int e = 0; e < hd; ++e) o[e] = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        double p = s[j] / den;
        for (int e = 0; e < hd; ++e) o[e] += p * V[j * ld + e];
    }
}

/* All n_head query heads; K, V hold n cells of n_head_kv * hd values each. */
void attend_gqa(const double *q, const double *K, const double *V, int64_t n, int n_head, int n_head_kv, int hd,
                double *o) {
    int group = n_head / n_head_kv;
    for (int h = 0; h < n_head; ++h) {
        int kv = h / group;
        attend_head(q + (int64_t)h * hd, K + (int64_t)kv * hd, V + (int64_t)kv * hd, n, (int64_t)n_head_kv * hd, hd,
                    o + (int64_t)h * hd);
    }
}

/* ------------------------------------------------------------------ model / context */
struct Layer { const float *attn_norm, *ffn_norm; const uint8_t *wq, *wk, *wv, *wo, *w_gate, *w_up, *w_down; };

struct Hparams {
    int32_t n_vocab, n_embd, n_layer, n_head, n_head_kv, head_dim, n_ff;
    double rms_eps, rope_theta;
    int32_t t_linear, t_embd, t_out;
};

struct Model {
    Hparams hp;
    const uint8_t *tok_embd, *output;
    const float *output_norm;
    std::vector<Layer> layers;
};

/* One sequence's cells: per layer, [cell][n_head_kv * head_dim] f16-rounded values (as doubles). */
struct Seq { std::vector<std::vector<double>> k, v; int64_t n = 0; };

struct Ctx {
    Model *m;
    uint32_t n_ctx, n_seq_max, n_ubatch;
    std::vector<Seq> seqs;
    int64_t used = 0;
    bool elide = true;   /* last layer: K and V only for tokens whose logits are not flagged */
    bool unified = true; /* one KV store shared by all sequences; else one stream per sequence */
    /* trace of one layer for the most recent token that ran it whole: x in, q after RoPE, o,
     * x after attention */
    int32_t trace_layer = -1;
    std::vector<double> tr_x, tr_q, tr_o, tr_x1;
};

int64_t kv_width(const Hparams &hp) { return (int64_t)hp.n_head_kv * hp.head_dim; }

constexpr int64_t kBlock = 256;   /* tokens evaluated layer by layer together */

/* Runs tokens tok[0..T) (validated; positions continue their sequences) through every layer,
 * appending their cells, and writes the logits and argmax of the flagged ones, in order. */
void run_block(Ctx &c, int64_t T, const int32_t *tok, const int32_t *pos, const int32_t *seq, const int8_t *flag,
               double *logits, int32_t *argmax) {
    const Model &m = *c.m;
    const Hparams &hp = m.hp;
    const int64_t d = hp.n_embd, hd = hp.head_dim, H = hp.n_head, KVH = hp.n_head_kv, KVW = kv_width(hp);
    const int64_t F = hp.n_ff, F_pad = (F + 31) / 32 * 32, L = hp.n_layer;
    std::vector<double> X((size_t)T * d), XN((size_t)T * d), Y((size_t)T * d);
    for (int64_t t = 0; t < T; ++t)
        dequant_row(hp.t_embd, m.tok_embd + (int64_t)tok[t] * row_bytes(hp.t_embd, d), d, &X[t * d]);
    std::vector<int64_t> all(T), out;
    for (int64_t t = 0; t < T; ++t) {
        all[t] = t;
        if (flag[t]) out.push_back(t);
    }
    for (int64_t t = 0; t < T; ++t) {   /* room for the new cells */
        Seq &s = c.seqs[seq[t]];
        s.k.resize(L);
        s.v.resize(L);
    }
    /* gathers rows idx of A [.][w] into B [idx.size()][w] and back */
    auto gather = [](const std::vector<double> &A, int64_t w, const std::vector<int64_t> &idx, std::vector<double> &B) {
        B.resize(idx.size() * w);
        for (size_t i = 0; i < idx.size(); ++i) std::memcpy(&B[i * w], &A[idx[i] * w], w * sizeof(double));
    };

    for (int64_t l = 0; l < L; ++l) {
        const Layer &W = m.layers[l];
        /* the tokens that run the whole layer: all but, in the last layer, the unflagged ones */
        const std::vector<int64_t> &full = (l == L - 1 && c.elide) ? out : all;
        const int64_t nf = (int64_t)full.size();
        for (int64_t t = 0; t < T; ++t) rmsnorm(&X[t * d], d, W.attn_norm, hp.rms_eps, &XN[t * d]);
        std::vector<double> K((size_t)T * KVW), V((size_t)T * KVW), XF, Q((size_t)nf * H * hd);
        matmat(hp.t_linear, W.wk, KVW, d, XN.data(), T, K.data());
        matmat(hp.t_linear, W.wv, KVW, d, XN.data(), T, V.data());
        gather(XN, d, full, XF);
        matmat(hp.t_linear, W.wq, H * hd, d, XF.data(), nf, Q.data());
        for (int64_t i = 0; i < nf; ++i)
            for (int64_t h = 0; h < H; ++h) rope(&Q[(i * H + h) * hd], (int)hd, pos[full[i]], hp.rope_theta);
        for (int64_t t = 0; t < T; ++t) {   /* K after RoPE and V, rounded to f16, into the cells */
            for (int64_t h = 0; h < KVH; ++h) rope(&K[t * KVW + h * hd], (int)hd, pos[t], hp.rope_theta);
            Seq &s = c.seqs[seq[t]];
            const int64_t cell = pos[t];   /* positions of a sequence are 0..n-1 */
            if ((int64_t)s.k[l].size() < (cell + 1) * KVW) {
                s.k[l].resize((size_t)(cell + 1) * KVW);
                s.v[l].resize((size_t)(cell + 1) * KVW);
            }
            for (int64_t e = 0; e < KVW; ++e) {
                s.k[l][cell * KVW + e] = round_to_half(K[t * KVW + e]);
                s.v[l][cell * KVW + e] = round_to_half(V[t * KVW + e]);
            }
        }
        if (nf == 0) continue;
        /* attention: query head h of token t over the cells of its sequence with pos <= pos_t */
        std::vector<double> O((size_t)nf * H * hd);
        const int group = (int)(H / KVH);
        pool().parallel_for(nf * H, [&](int64_t lo, int64_t hi) {
            for (int64_t i = lo; i < hi; ++i) {
                const int64_t f = i / H, h = i % H, t = full[f];
                const Seq &s = c.seqs[seq[t]];
                const int64_t kv = h / group;
                attend_head(&Q[i * hd], s.k[l].data() + kv * hd, s.v[l].data() + kv * hd, pos[t] + 1, KVW, (int)hd,
                            &O[i * hd]);
            }
        }, 2);
        if (l == c.trace_layer) {
            const int64_t f = nf - 1, t = full[f];
            c.tr_x.assign(&X[t * d], &X[t * d] + d);
            c.tr_q.assign(&Q[f * H * hd], &Q[f * H * hd] + H * hd);
            c.tr_o.assign(&O[f * H * hd], &O[f * H * hd] + H * hd);
        }
        matmat(hp.t_linear, W.wo, d, H * hd, O.data(), nf, Y.data());
        for (int64_t i = 0; i < nf; ++i)
            for (int64_t e = 0; e < d; ++e) X[full[i] * d + e] += Y[i * d + e];
        if (l == c.trace_layer) c.tr_x1.assign(&X[full[nf - 1] * d], &X[full[nf - 1] * d] + d);
        /* SwiGLU feed-forward; ffn_down's inputs past n_ff are zero */
        for (int64_t i = 0; i < nf; ++i) rmsnorm(&X[full[i] * d], d, W.ffn_norm, hp.rms_eps, &XN[i * d]);
        std::vector<double> G((size_t)nf * F), U((size_t)nf * F), Hh((size_t)nf * F_pad, 0.0);
        matmat(hp.t_linear, W.w_gate, F, d, XN.data(), nf, G.data());
        matmat(hp.t_linear, W.w_up, F, d, XN.data(), nf, U.data());
        for (int64_t i = 0; i < nf; ++i)
            for (int64_t e = 0; e < F; ++e) Hh[i * F_pad + e] = silu(G[i * F + e]) * U[i * F + e];
        matmat(hp.t_linear, W.w_down, d, F_pad, Hh.data(), nf, Y.data());
        for (int64_t i = 0; i < nf; ++i)
            for (int64_t e = 0; e < d; ++e) X[full[i] * d + e] += Y[i * d + e];
    }
    for (int64_t t = 0; t < T; ++t) {
        Seq &s = c.seqs[seq[t]];
        if (pos[t] + 1 > s.n) s.n = pos[t] + 1;
        c.used += 1;
    }
    if (out.empty()) return;
    /* final norm and the head for the flagged tokens (step 14) */
    const int64_t no = (int64_t)out.size();
    for (int64_t i = 0; i < no; ++i) rmsnorm(&X[out[i] * d], d, m.output_norm, hp.rms_eps, &XN[i * d]);
    const uint8_t *Wout = m.output ? m.output : m.tok_embd;
    const int tout = m.output ? hp.t_out : hp.t_embd;
    matmat(tout, Wout, hp.n_vocab, d, XN.data(), no, logits);
    for (int64_t i = 0; i < no; ++i) {
        const double *lg = logits + i * hp.n_vocab;
        int32_t best = 0;
        for (int32_t j = 1; j < hp.n_vocab; ++j)
            if (lg[j] > lg[best]) best = j;
        argmax[i] = best;
    }
}

/* Removes the cells appended by tokens i0..i1 of a batch (each token appended the cell at its
 * position of its sequence; a sequence's cells stay positions 0..n-1). */
void rollback(Ctx &c, int32_t i0, int32_t i1, const int32_t *seq, const int32_t *pos) {
    const int64_t W = kv_width(c.m->hp);
    for (int32_t j = i0; j <= i1; ++j) {
        Seq &s = c.seqs[seq[j]];
        if (pos[j] < s.n) s.n = pos[j];
        c.used -= 1;
    }
    for (auto &s : c.seqs)
        for (size_t l = 0; l < s.k.size(); ++l) {
            if ((int64_t)s.k[l].size() > s.n * W) s.k[l].resize((size_t)(s.n * W));
            if ((int64_t)s.v[l].size() > s.n * W) s.v[l].resize((size_t)(s.n * W));
        }
}

}  // namespace

/* ====================================================================== C API */
extern "C" {

typedef struct {
    int32_t n_vocab, n_embd, n_layer, n_head, n_head_kv, head_dim, n_ff;
    double rms_eps, rope_theta;
    int32_t t_linear, t_embd, t_out;
} orc_hparams;

typedef struct { const void *attn_norm, *wq, *wk, *wv, *wo, *ffn_norm, *w_gate, *w_up, *w_down; } orc_layer;

void orc_set_threads(int n) { pool().resize(n); }
int orc_get_threads(void) { return pool().size(); }

void *orc_model_create(const orc_hparams *hp, const void *tok_embd, const float *output_norm, const void *output,
                       const orc_layer *layers) {
    if (!hp || !tok_embd || !output_norm || !layers) return nullptr;
    if (hp->n_head <= 0 || hp->n_head_kv <= 0 || hp->n_head % hp->n_head_kv || hp->head_dim % 2) return nullptr;
    Model *m = new Model;
    m->hp = Hparams{hp->n_vocab, hp->n_embd, hp->n_layer, hp->n_head, hp->n_head_kv, hp->head_dim, hp->n_ff,
                    hp->rms_eps, hp->rope_theta, hp->t_linear, hp->t_embd, hp->t_out};
    m->tok_embd = (const uint8_t *)tok_embd;
    m->output = (const uint8_t *)output;
    m->output_norm = output_norm;
    for (int l = 0; l < hp->n_layer; ++l) {
        const orc_layer &s = layers[l];
        m->layers.push_back(Layer{(const float *)s.attn_norm, (const float *)s.ffn_norm, (const uint8_t *)s.wq,
                                  (const uint8_t *)s.wk, (const uint8_t *)s.wv, (const uint8_t *)s.wo,
                                  (const uint8_t *)s.w_gate, (const uint8_t *)s.w_up, (const uint8_t *)s.w_down});
    }
    return m;
}

void orc_model_free(void *m) { delete (Model *)m; }

/* n_ctx is rounded up to a multiple of 256, as the context constructor does (step 10). */
void *orc_ctx_create(void *model, uint32_t n_ctx, uint32_t n_seq_max, uint32_t n_ubatch) {
    if (!model || n_ctx == 0 || n_seq_max == 0 || n_ubatch == 0) return nullptr;
    Ctx *c = new Ctx;
    c->m = (Model *)model;
    c->n_ctx = (n_ctx + 255u) / 256u * 256u;
    c->n_seq_max = n_seq_max;
    c->n_ubatch = n_ubatch;
    c->seqs.resize(n_seq_max);
    return c;
}

void orc_ctx_free(void *c) { delete (Ctx *)c; }
uint32_t orc_n_ctx(const void *c) { return ((const Ctx *)c)->n_ctx; }

void orc_kv_clear(void *cv) {
    Ctx *c = (Ctx *)cv;
    for (auto &s : c->seqs) { s.k.clear(); s.v.clear(); s.n = 0; }
    c->used = 0;
}

int32_t orc_seq_pos_max(const void *cv, int32_t seq) {
    const Ctx *c = (const Ctx *)cv;
    if (seq < 0 || (uint32_t)seq >= c->n_seq_max) return -1;
    return (int32_t)c->seqs[seq].n - 1;
}

/* The stored (f16-rounded) K and V of one cell and layer, as doubles [n_head_kv * head_dim]. */
int32_t orc_kv_get(const void *cv, int32_t seq, int32_t pos, int32_t layer, double *k, double *v) {
    const Ctx *c = (const Ctx *)cv;
    if (seq < 0 || (uint32_t)seq >= c->n_seq_max) return -1;
    const Seq &s = c->seqs[seq];
    const int64_t L = c->m->hp.n_layer, W = kv_width(c->m->hp);
    if (pos < 0 || pos >= s.n || layer < 0 || layer >= L) return -1;
    for (int64_t e = 0; e < W; ++e) {
        k[e] = s.k[layer][(int64_t)pos * W + e];
        v[e] = s.v[layer][(int64_t)pos * W + e];
    }
    return 0;
}

/* Validates, fills, and runs the batch token by token. logits_out: [n_out][n_vocab] doubles
 * (may be NULL), argmax_out: [n_out]. *n_out receives the number of flagged tokens. */
int32_t orc_decode(void *cv, int32_t n_tokens, const int32_t *token, const int32_t *pos_in, const int32_t *seq_in,
                   const int8_t *flags_in, double *logits_out, int32_t *argmax_out, int32_t *n_out) {
    Ctx *c = (Ctx *)cv;
    const Hparams &hp = c->m->hp;
    if (n_out) *n_out = 0;
    if (n_tokens <= 0 || !token) return -1;
    std::vector<int32_t> seq(n_tokens), pos(n_tokens);
    std::vector<int8_t> flag(n_tokens);
    std::vector<int64_t> next(c->n_seq_max);
    for (uint32_t s = 0; s < c->n_seq_max; ++s) next[s] = c->seqs[s].n;
    for (int32_t i = 0; i < n_tokens; ++i) {
        if (token[i] < 0 || token[i] >= hp.n_vocab) return -1;
        seq[i] = seq_in ? seq_in[i] : 0;
        if (seq[i] < 0 || (uint32_t)seq[i] >= c->n_seq_max) return -1;
        int64_t expect = next[seq[i]]++;
        pos[i] = pos_in ? pos_in[i] : (int32_t)expect;
        if ((int64_t)pos[i] != expect) return -1;
        flag[i] = flags_in ? (flags_in[i] != 0) : (int8_t)(i == n_tokens - 1);
    }
    /* capacity (step 10 and init_batch): one shared store of n_ctx cells, or, with a stream per
     * sequence, n_ctx_seq = n_ctx / n_seq_max cells for each sequence */
    if (c->unified) {
        if (c->used + n_tokens > (int64_t)c->n_ctx) return 1;
    } else {
        const int64_t n_ctx_seq = (int64_t)c->n_ctx / c->n_seq_max;
        for (uint32_t s = 0; s < c->n_seq_max; ++s)
            if (next[s] > n_ctx_seq) return 1;
    }
    /* ubatches (step 12, init_batch): with one store, consecutive chunks of n_ubatch tokens
     * (split_simple); with a stream per sequence, split_equal: every ubatch takes the same number
     * of next tokens from each sequence that has tokens left (the lowest sequence ids first, at
     * most n_ubatch sequences): as many as the shortest of them has left, and at most n_ubatch
     * divided by their number; inside the ubatch, sequence by sequence in position order */
    std::vector<std::vector<int32_t>> ubs;
    if (c->unified) {
        for (int32_t u0 = 0; u0 < n_tokens; u0 += (int32_t)c->n_ubatch) {
            std::vector<int32_t> u;
            for (int32_t i = u0; i < n_tokens && i < u0 + (int32_t)c->n_ubatch; ++i) u.push_back(i);
            ubs.push_back(u);
        }
    } else {
        std::vector<std::vector<int32_t>> left(c->n_seq_max);   /* each sequence's tokens, in batch order */
        for (int32_t i = 0; i < n_tokens; ++i) left[seq[i]].push_back(i);
        std::vector<size_t> taken(c->n_seq_max, 0);
        for (;;) {
            std::vector<uint32_t> ss;
            for (uint32_t s = 0; s < c->n_seq_max && ss.size() < c->n_ubatch; ++s)
                if (taken[s] < left[s].size()) ss.push_back(s);
            if (ss.empty()) break;
            size_t k = c->n_ubatch / ss.size();
            for (uint32_t s : ss) k = std::min(k, left[s].size() - taken[s]);
            std::vector<int32_t> u;
            for (uint32_t s : ss)
                for (size_t j = 0; j < k; ++j) u.push_back(left[s][taken[s] + j]);
            for (uint32_t s : ss) taken[s] += k;
            ubs.push_back(u);
        }
    }
    /* output rows in batch order: the row of flagged token i is the number of flagged tokens before it */
    std::vector<int32_t> brow(n_tokens, -1);
    int32_t n_rows = 0;
    for (int32_t i = 0; i < n_tokens; ++i)
        if (flag[i]) brow[i] = n_rows++;
    std::vector<double> tmp;
    int32_t row = 0;   /* rows done, ubatch by ubatch */
    for (const std::vector<int32_t> &u : ubs) {
        const int32_t nt = (int32_t)u.size();
        std::vector<int32_t> ut(nt), up(nt), us(nt);
        std::vector<int8_t> uf(nt);
        int32_t nu = 0;
        for (int32_t i = 0; i < nt; ++i) {
            ut[i] = token[u[i]];
            up[i] = pos[u[i]];
            us[i] = seq[u[i]];
            uf[i] = flag[u[i]];
            nu += uf[i];
        }
        tmp.resize((size_t)(nu > 0 ? nu : 1) * hp.n_vocab);
        std::vector<int32_t> am(nu > 0 ? nu : 1);
        int32_t r = 0;
        for (int32_t b0 = 0; b0 < nt; b0 += (int32_t)kBlock) {
            const int32_t b1 = b0 + (int32_t)kBlock < nt ? b0 + (int32_t)kBlock : nt;
            run_block(*c, b1 - b0, ut.data() + b0, up.data() + b0, us.data() + b0, uf.data() + b0,
                      tmp.data() + (int64_t)r * hp.n_vocab, am.data() + r);
            for (int32_t i = b0; i < b1; ++i) r += uf[i];
        }
        /* a logit that is not finite fails the ubatch (step 13, a failed compute: its cells are
         * removed again); earlier ubatches stay, and so do their rows when they are the first
         * rows of the batch (one store: the ubatches run in batch order); with a stream per
         * sequence the rows of a stopped batch are not reported */
        for (int64_t j = 0; j < (int64_t)nu * hp.n_vocab; ++j)
            if (!std::isfinite(tmp[j])) {
                for (int32_t i = nt - 1; i >= 0; --i) rollback(*c, u[i], u[i], seq.data(), pos.data());
                if (n_out) *n_out = c->unified ? row : 0;
                return -3;
            }
        r = 0;
        for (int32_t i = 0; i < nt; ++i)
            if (uf[i]) {
                if (logits_out)
                    std::memcpy(logits_out + (int64_t)brow[u[i]] * hp.n_vocab, tmp.data() + (int64_t)r * hp.n_vocab,
                                (size_t)hp.n_vocab * sizeof(double));
                if (argmax_out) argmax_out[brow[u[i]]] = am[r];
                ++r;
            }
        row += nu;
    }
    if (n_out) *n_out = row;
    return 0;
}

/* 1: one KV store shared by every sequence (the default); 0: a stream per sequence, each of
 * n_ctx / n_seq_max cells, batches cut by split_equal. Only while the store is empty. */
int32_t orc_set_kv_unified(void *cv, int32_t on) {
    Ctx *c = (Ctx *)cv;
    if (c->used != 0) return -1;
    c->unified = on != 0;
    return 0;
}

/* Last layer: 1 = tokens whose logits are not flagged compute only their K and V (the default),
 * 0 = every token runs the whole layer. The results are the same either way. */
void orc_set_elide(void *cv, int32_t on) { ((Ctx *)cv)->elide = on != 0; }

/* Record intermediates of `layer` for each token run (the last one is kept); -1 = off. */
void orc_set_trace(void *cv, int32_t layer) { ((Ctx *)cv)->trace_layer = layer; }
/* which: 0 = x entering the layer [d], 1 = q after RoPE [H*hd], 2 = attention output [H*hd],
 * 3 = x after the attention residual [d]. Returns the element count, or -1. */
int64_t orc_get_trace(const void *cv, int32_t which, double *out) {
    const Ctx *c = (const Ctx *)cv;
    const std::vector<double> *v = which == 0 ? &c->tr_x : which == 1 ? &c->tr_q : which == 2 ? &c->tr_o
                                 : which == 3 ? &c->tr_x1 : nullptr;
    if (!v || v->empty()) return -1;
    if (out) std::memcpy(out, v->data(), v->size() * sizeof(double));
    return (int64_t)v->size();
}

/* ---------------------------------------------------------------- single operations */
int64_t orc_row_bytes(int32_t type, int64_t k) { return row_bytes(type, k); }
void orc_dequant_row(int32_t type, const void *row, int64_t n, double *out) { dequant_row(type, (const uint8_t *)row, n, out); }
double orc_half_to_double(uint16_t h) { return half_to_double(h); }
double orc_round_to_half(double x) { return round_to_half(x); }
void orc_matvec(int32_t type, const void *W, int64_t N, int64_t K, const double *x, double *y) {
    matvec(type, (const uint8_t *)W, N, K, x, y);
}
void orc_matmat(int32_t type, const void *W, int64_t N, int64_t K, const double *X, int64_t T, double *Y) {
    matmat(type, (const uint8_t *)W, N, K, X, T, Y);
}
void orc_rmsnorm(const double *x, int64_t n, const float *g, double eps, double *y) { rmsnorm(x, n, g, eps, y); }
void orc_rope(double *x, int32_t hd, int64_t pos, double theta) { rope(x, hd, pos, theta); }
double orc_silu(double a) { return silu(a); }
void orc_attend_gqa(const double *q, const double *K, const double *V, int64_t n, int32_t n_head, int32_t n_head_kv,
                    int32_t hd, double *o) {
    attend_gqa(q, K, V, n, n_head, n_head_kv, hd, o);
}

}  // extern "C"
