/*
 * Seeded synthetic inputs for the Llama ubatch forward: weights, norm gains, token ids and
 * prompt lengths, plus the encoders that turn f32 weights into the stored block formats.
 *
 * This module is shared by the CPU oracle and by the CUDA path as their common source of
 * inputs. It holds none of the forward's arithmetic: no dequantisation, no norm, no
 * matmul. It only draws numbers and encodes them into the bytes a model file would hold.
 *
 * Random numbers: a counter-based draw. Element i of tensor `tid` under seed `seed` is
 *   key = mix(seed * 0x9E3779B97F4A7C15 + tid),  r = mix(key + (i + 1) * 0x9E3779B97F4A7C15)
 * where mix() is the splitmix64 output function (Steele, Lea and Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014). The two 32-bit halves of r give
 * u1, u2 in (0, 1); a normal draw is sqrt(-2 ln u1) cos(2 pi u2) (Box and Muller, 1958).
 *
 * Block encodings (the bytes the forward reads):
 *   Q8_0: 34 bytes per 32 consecutive elements of a row: fp16 d, then int8 q[32];
 *         d = fp16(amax / 127), q = round-half-away(w / d) clamped to [-127, 127].
 *   Q4_0: 18 bytes per 32 elements: fp16 d, then 16 bytes; element j (0..15) sits in the
 *         low nibble of byte j and element j + 16 in the high nibble.
 *         m = the element with the largest magnitude (sign kept), d = fp16(m / -8),
 *         q = min(15, floor(w / d + 8.5)); all elements zero -> d = 0, q = 8.
 *   F16:  IEEE binary16, round to nearest even.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

uint64_t synth_draw_u64(uint64_t seed, uint64_t tid, uint64_t i) {
    uint64_t key = mix64(seed * GOLDEN + tid);
    return mix64(key + (i + 1) * GOLDEN);
}

static inline double normal_at(uint64_t key, uint64_t i) {
    uint64_t r = mix64(key + (i + 1) * GOLDEN);
    double u1 = ((double)(r >> 32) + 0.5) * (1.0 / 4294967296.0);
    double u2 = ((double)(r & 0xffffffffULL) + 0.5) * (1.0 / 4294967296.0);
    return sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925286766559 * u2);
}

/* ---------------------------------------------------------------- threading */
typedef void (*range_fn)(void *ctx, int64_t lo, int64_t hi);
typedef struct { range_fn fn; void *ctx; int64_t lo, hi; } job_t;
static void *job_main(void *p) { job_t *j = (job_t *)p; j->fn(j->ctx, j->lo, j->hi); return NULL; }

static void run_parallel(range_fn fn, void *ctx, int64_t n, int n_threads) {
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 256) n_threads = 256;
    if (n < 4096 || n_threads == 1) { fn(ctx, 0, n); return; }
    pthread_t th[256];
    job_t jobs[256];
    int64_t chunk = (n + n_threads - 1) / n_threads;
    int started = 0;
    for (int t = 0; t < n_threads; ++t) {
        int64_t lo = t * chunk, hi = lo + chunk < n ? lo + chunk : n;
        if (lo >= hi) break;
        jobs[t] = (job_t){fn, ctx, lo, hi};
        if (pthread_create(&th[t], NULL, job_main, &jobs[t]) != 0) { fn(ctx, lo, hi); jobs[t].fn = NULL; }
        started = t + 1;
    }
    for (int t = 0; t < started; ++t) if (jobs[t].fn) pthread_join(th[t], NULL);
}

/* ---------------------------------------------------------------- fp16 encode */
uint16_t synth_f32_to_f16(float f) {
    uint32_t x; memcpy(&x, &f, 4);
    uint32_t sign = (x >> 16) & 0x8000u;
    uint32_t exp = (x >> 23) & 0xffu;
    uint32_t man = x & 0x7fffffu;
    if (exp == 0xffu) return (uint16_t)(sign | 0x7c00u | (man ? 0x200u : 0));
    int32_t e = (int32_t)exp - 127 + 15;
    if (e >= 31) return (uint16_t)(sign | 0x7c00u);
    if (e <= 0) {                                   /* subnormal or zero half */
        if (e < -10) return (uint16_t)sign;
        man |= 0x800000u;
        uint32_t shift = (uint32_t)(14 - e);
        uint32_t h = man >> shift;
        uint32_t rem = man & ((1u << shift) - 1u), half = 1u << (shift - 1);
        if (rem > half || (rem == half && (h & 1u))) h++;
        return (uint16_t)(sign | h);
    }
    uint32_t h = ((uint32_t)e << 10) | (man >> 13);
    uint32_t rem = man & 0x1fffu;
    if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) h++;   /* may carry into the exponent: correct */
    return (uint16_t)(sign | h);
}

static float f16_bits_to_f32(uint16_t h) {
    uint32_t sign = (uint32_t)(h & 0x8000u) << 16, exp = (h >> 10) & 0x1fu, man = h & 0x3ffu, x;
    if (exp == 0) {
        if (man == 0) x = sign;
        else { int e = -1; do { man <<= 1; e++; } while (!(man & 0x400u)); man &= 0x3ffu;
               x = sign | ((uint32_t)(127 - 15 - e) << 23) | (man << 13); }
    } else if (exp == 31) x = sign | 0x7f800000u | (man << 13);
    else x = sign | ((exp - 15 + 127) << 23) | (man << 13);
    float f; memcpy(&f, &x, 4); return f;
}

/* ---------------------------------------------------------------- draws */
typedef struct { uint64_t key; float mean, std; float *out; } normal_job;
static void normal_range(void *p, int64_t lo, int64_t hi) {
    normal_job *j = (normal_job *)p;
    for (int64_t i = lo; i < hi; ++i) j->out[i] = (float)(j->mean + j->std * normal_at(j->key, (uint64_t)i));
}

/* out[i] = mean + std * N(0,1) draw i of tensor tid, rounded to f32. */
void synth_normal_f32(uint64_t seed, uint64_t tid, int64_t n, float mean, float std, float *out, int n_threads) {
    normal_job j = {mix64(seed * GOLDEN + tid), mean, std, out};
    run_parallel(normal_range, &j, n, n_threads);
}

/* out[i] = lo + (draw_i mod (hi - lo)), a near-uniform integer in [lo, hi). */
void synth_uniform_i32(uint64_t seed, uint64_t tid, int64_t n, int32_t lo, int32_t hi, int32_t *out) {
    uint64_t key = mix64(seed * GOLDEN + tid), span = (uint64_t)((int64_t)hi - lo);
    for (int64_t i = 0; i < n; ++i) out[i] = (int32_t)(lo + (int64_t)(mix64(key + ((uint64_t)i + 1) * GOLDEN) % span));
}

/* ---------------------------------------------------------------- encoders */
typedef struct { const float *w; int64_t k, k_pad; uint8_t *out; } enc_job;

/* Rows of k floats, padded with zeros to k_pad (a multiple of 32), encoded block by block. */
static void q8_0_range(void *p, int64_t lo, int64_t hi) {
    enc_job *j = (enc_job *)p;
    int64_t nb = j->k_pad / 32;
    for (int64_t r = lo; r < hi; ++r) {
        const float *row = j->w + r * j->k;
        for (int64_t b = 0; b < nb; ++b) {
            float v[32]; float amax = 0.f;
            for (int e = 0; e < 32; ++e) {
                int64_t c = b * 32 + e;
                v[e] = c < j->k ? row[c] : 0.f;
                if (fabsf(v[e]) > amax) amax = fabsf(v[e]);
            }
            uint8_t *blk = j->out + (r * nb + b) * 34;
            uint16_t dh = synth_f32_to_f16(amax / 127.f);
            double d = (double)f16_bits_to_f32(dh);
            blk[0] = (uint8_t)(dh & 0xff); blk[1] = (uint8_t)(dh >> 8);
            for (int e = 0; e < 32; ++e) {
                int q = 0;
                if (d != 0.0) {
                    double t = (double)v[e] / d;
                    q = (int)(t >= 0 ? floor(t + 0.5) : -floor(-t + 0.5));
                    if (q > 127) q = 127;
                    if (q < -127) q = -127;
                }
                blk[2 + e] = (uint8_t)(int8_t)q;
            }
        }
    }
}

static void q4_0_range(void *p, int64_t lo, int64_t hi) {
    enc_job *j = (enc_job *)p;
    int64_t nb = j->k_pad / 32;
    for (int64_t r = lo; r < hi; ++r) {
        const float *row = j->w + r * j->k;
        for (int64_t b = 0; b < nb; ++b) {
            float v[32]; float amax = 0.f, m = 0.f;
            for (int e = 0; e < 32; ++e) {
                int64_t c = b * 32 + e;
                v[e] = c < j->k ? row[c] : 0.f;
                if (fabsf(v[e]) > amax) { amax = fabsf(v[e]); m = v[e]; }
            }
            uint8_t *blk = j->out + (r * nb + b) * 18;
            uint16_t dh = synth_f32_to_f16(m / -8.f);
            float d = f16_bits_to_f32(dh);
            blk[0] = (uint8_t)(dh & 0xff); blk[1] = (uint8_t)(dh >> 8);
            uint8_t q[32];
            for (int e = 0; e < 32; ++e) {
                int qi = 8;
                if (d != 0.f) {
                    double t = floor((double)(v[e] / d) + 8.5);
                    qi = t < 0 ? 0 : (t > 15 ? 15 : (int)t);
                }
                q[e] = (uint8_t)qi;
            }
            for (int e = 0; e < 16; ++e) blk[2 + e] = (uint8_t)(q[e] | (q[e + 16] << 4));
        }
    }
}

static void f16_range(void *p, int64_t lo, int64_t hi) {
    enc_job *j = (enc_job *)p;
    uint16_t *o = (uint16_t *)j->out;
    for (int64_t i = lo; i < hi; ++i) o[i] = synth_f32_to_f16(j->w[i]);
}

/* w: n_rows x k floats. out: n_rows x (k_pad / 32) blocks of 34 (Q8_0) or 18 (Q4_0) bytes. */
void synth_encode_q8_0(const float *w, int64_t n_rows, int64_t k, int64_t k_pad, uint8_t *out, int n_threads) {
    enc_job j = {w, k, k_pad, out};
    run_parallel(q8_0_range, &j, n_rows, n_threads);
}
void synth_encode_q4_0(const float *w, int64_t n_rows, int64_t k, int64_t k_pad, uint8_t *out, int n_threads) {
    enc_job j = {w, k, k_pad, out};
    run_parallel(q4_0_range, &j, n_rows, n_threads);
}
void synth_encode_f16(const float *w, int64_t n, uint16_t *out, int n_threads) {
    enc_job j = {w, n, n, (uint8_t *)out};
    run_parallel(f16_range, &j, n, n_threads);
}
