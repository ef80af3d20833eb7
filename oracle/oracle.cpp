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
 *   chunks of n_ubatch tokens) removed again, earlier ubatches kept, no rows reported.
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
    for (int64_t i = 0; i < n; ++i) {
        int64_t b = i / 32, e = i % 32;
        if (type == T_Q8_0) {
            const uint8_t *blk = row + b * 34;
            double d = half_to_double((uint16_t)(blk[0] | (blk[1] << 8)));
            out[i] = d * (double)(int8_t)blk[2 + e];
        } else {
            const uint8_t *blk = row + b * 18;
            double d = half_to_double((uint16_t)(blk[0] | (blk[1] << 8)));
            int q = e < 16 ? (blk[2 + e] & 0x0f) : (blk[2 + e - 16] >> 4);
            out[i] = d * (double)(q - 8);
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
    /* fn(lo, hi) over [0, n) in n_ contiguous chunks; the caller runs chunk 0. */
    void parallel_for(int64_t n, const std::function<void(int64_t, int64_t)> &fn) {
        if (n_ == 1 || n < 64) { fn(0, n); return; }
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
/* y[n] = sum_k W[n][k] x[k]: W stored row-major, row n = the K inputs of output n. */
void matvec(int type, const uint8_t *W, int64_t N, int64_t K, const double *x, double *y) {
    const int64_t rb = row_bytes(type, K);
    pool().parallel_for(N, [&](int64_t lo, int64_t hi) {
        std::vector<double> w(K);
        for (int64_t n = lo; n < hi; ++n) {
            dequant_row(type, W + n * rb, K, w.data());
            double s = 0.0;
            for (int64_t k = 0; k < K; ++k) s += w[k] * x[k];
            y[n] = s;
        }
    });
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
    /* trace of one layer for the most recent token: x in, q after RoPE, o, x after attention */
    int32_t trace_layer = -1;
    std::vector<double> tr_x, tr_q, tr_o, tr_x1;
};

int64_t kv_width(const Hparams &hp) { return (int64_t)hp.n_head_kv * hp.head_dim; }

/* Runs one validated token through every layer, appending its cell; logits if flagged. */
void forward_token(Ctx &c, int32_t tok, int32_t pos, int32_t seq, double *logits, int32_t *argmax) {
    const Model &m = *c.m;
    const Hparams &hp = m.hp;
    const int64_t d = hp.n_embd, hd = hp.head_dim, H = hp.n_head, KVW = kv_width(hp), F = hp.n_ff;
    const int64_t F_pad = (F + 31) / 32 * 32, L = hp.n_layer;
    std::vector<double> x(d), xn(d), q(H * hd), k(KVW), v(KVW), o(H * hd), y(d), g(F), u(F), h(F_pad, 0.0);
    dequant_row(hp.t_embd, m.tok_embd + (int64_t)tok * row_bytes(hp.t_embd, d), d, x.data());

    Seq &s = c.seqs[seq];
    s.k.resize(L);
    s.v.resize(L);
    const int64_t cell = pos;                                  /* positions of a sequence are 0..n-1 */

    for (int64_t l = 0; l < L; ++l) {
        const Layer &W = m.layers[l];
        rmsnorm(x.data(), d, W.attn_norm, hp.rms_eps, xn.data());
        matvec(hp.t_linear, W.wq, H * hd, d, xn.data(), q.data());
        matvec(hp.t_linear, W.wk, KVW, d, xn.data(), k.data());
        matvec(hp.t_linear, W.wv, KVW, d, xn.data(), v.data());
        for (int64_t hh = 0; hh < H; ++hh) rope(q.data() + hh * hd, (int)hd, pos, hp.rope_theta);
        for (int64_t hh = 0; hh < hp.n_head_kv; ++hh) rope(k.data() + hh * hd, (int)hd, pos, hp.rope_theta);
        s.k[l].resize((size_t)(cell + 1) * KVW);
        s.v[l].resize((size_t)(cell + 1) * KVW);
        for (int64_t e = 0; e < KVW; ++e) {
            s.k[l][cell * KVW + e] = round_to_half(k[e]);
            s.v[l][cell * KVW + e] = round_to_half(v[e]);
        }
        attend_gqa(q.data(), s.k[l].data(), s.v[l].data(), pos + 1, (int)H, hp.n_head_kv, (int)hd, o.data());
        if (l == c.trace_layer) { c.tr_x = x; c.tr_q = q; c.tr_o = o; }
        matvec(hp.t_linear, W.wo, d, H * hd, o.data(), y.data());
        for (int64_t i = 0; i < d; ++i) x[i] += y[i];
        if (l == c.trace_layer) c.tr_x1 = x;
        rmsnorm(x.data(), d, W.ffn_norm, hp.rms_eps, xn.data());
        matvec(hp.t_linear, W.w_gate, F, d, xn.data(), g.data());
        matvec(hp.t_linear, W.w_up, F, d, xn.data(), u.data());
        for (int64_t i = 0; i < F; ++i) h[i] = silu(g[i]) * u[i];
        matvec(hp.t_linear, W.w_down, d, F_pad, h.data(), y.data());
        for (int64_t i = 0; i < d; ++i) x[i] += y[i];
    }
    s.n = pos + 1;
    c.used += 1;

    if (logits) {
        rmsnorm(x.data(), d, m.output_norm, hp.rms_eps, xn.data());
        const uint8_t *Wout = m.output ? m.output : m.tok_embd;
        int tout = m.output ? hp.t_out : hp.t_embd;
        matvec(tout, Wout, hp.n_vocab, d, xn.data(), logits);
        int32_t best = 0;
        for (int32_t i = 1; i < hp.n_vocab; ++i)
            if (logits[i] > logits[best]) best = i;
        *argmax = best;
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
    if (c->used + n_tokens > (int64_t)c->n_ctx) return 1;
    int32_t row = 0;
    for (int32_t i = 0; i < n_tokens; ++i) {
        double *lg = nullptr;
        std::vector<double> tmp;
        int32_t am = -1;
        if (flag[i]) {
            if (logits_out) lg = logits_out + (int64_t)row * hp.n_vocab;
            else { tmp.resize(hp.n_vocab); lg = tmp.data(); }
        }
        forward_token(*c, token[i], pos[i], seq[i], lg, &am);
        if (flag[i]) {
            /* a logit that is not finite fails the ubatch (step 13, a failed compute: its cells
             * are removed again); earlier ubatches stay */
            for (int32_t j = 0; j < hp.n_vocab; ++j)
                if (!std::isfinite(lg[j])) {
                    rollback(*c, i - i % (int32_t)c->n_ubatch, i, seq.data(), pos.data());
                    return -3;
                }
            if (argmax_out) argmax_out[row] = am;
            ++row;
        }
    }
    if (n_out) *n_out = row;
    return 0;
}

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
void orc_rmsnorm(const double *x, int64_t n, const float *g, double eps, double *y) { rmsnorm(x, n, g, eps, y); }
void orc_rope(double *x, int32_t hd, int64_t pos, double theta) { rope(x, hd, pos, theta); }
double orc_silu(double a) { return silu(a); }
void orc_attend_gqa(const double *q, const double *K, const double *V, int64_t n, int32_t n_head, int32_t n_head_kv,
                    int32_t hd, double *o) {
    attend_gqa(q, K, V, n, n_head, n_head_kv, hd, o);
}

}  // extern "C"
