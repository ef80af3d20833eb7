// GEMM for prefill-sized ubatches: out[t][n] = sum_k A[t][k] W[n][k] with A in f16 (the
// RMS-normalised activations) and W in Q4_0 / Q8_0 dequantised on load, f32 accumulation,
// followed by the shared epilogues (RoPE + KV append, residual add, SwiGLU, logits).
//
// This is the CUDA-core tiled version: a CTA computes 16 row tasks (quads, or gate/up quad
// pairs for SwiGLU) x 32 tokens, with the weight tile dequantised once into shared memory.
#include <cstdlib>

#include "epilogue.cuh"

namespace lcx {

namespace {

constexpr int TT = 32;     // tokens per CTA
constexpr int TASKS = 16;  // row tasks per CTA

// element e of block b of row `row` in the quad-interleaved storage (QMat)
template <int QT>
__device__ __forceinline__ float deq(const uint8_t *w, int nb, int row, int b, int e) {
    constexpr int QB = QT == Q8 ? 32 : 16;
    const uint8_t *quad = w + (size_t)(row >> 2) * (nb / 2) * pair_bytes_of(QB);
    const float d = __half2float(*reinterpret_cast<const __half *>(quad + quad_s_off(QB, b) + 2 * (row & 3)));
    const uint8_t *q = quad + quad_q_off(QB, row & 3, b);
    if (QT == Q8) return d * (float)(int8_t)q[e];
    const uint8_t byte = q[e & 15];
    const int v = e < 16 ? (byte & 15) : (byte >> 4);
    return d * (float)(v - 8);
}

template <int QT, int ROWS, int EPI, bool OUT16>
__global__ void __launch_bounds__(256) k_gemm_simt(const uint8_t *__restrict__ w, int N,
                                                   int nb, int n_tasks, int T, const __half *__restrict__ A,
                                                   const __half *__restrict__ A_lo, const FwdArgs a, int layer) {
    __shared__ float Ws[32][TASKS * ROWS + 1];
    __shared__ float Xs[32][TT + 1];
    LCX_PDL_WAIT();
    LCX_PDL_TRIGGER();
    const int task0 = blockIdx.x * TASKS, tok0 = blockIdx.y * TT;
    const int K = nb * 32;
    const int tq = threadIdx.x % TASKS, tp = threadIdx.x / TASKS;   // task in tile, token pair
    float acc[ROWS][2];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) acc[r][0] = acc[r][1] = 0.f;

    // a SwiGLU task (ROWS 8) is a gate quad and the up quad after it: rows 8 task .. 8 task + 7
    auto task_row = [&](int task, int r) -> int { return task * ROWS + r; };

    for (int b = 0; b < nb; ++b) {
        for (int i = threadIdx.x; i < 32 * TASKS * ROWS; i += blockDim.x) {
            const int e = i % 32, rr = i / 32;   // rr = local row (task * ROWS + r)
            const int task = task0 + rr / ROWS;
            Ws[e][rr] = task < n_tasks ? deq<QT>(w, nb, task_row(task, rr % ROWS), b, e) : 0.f;
        }
        for (int i = threadIdx.x; i < 32 * TT; i += blockDim.x) {
            const int e = i % 32, tt = i / 32;
            const size_t ai = (size_t)(tok0 + tt) * K + b * 32 + e;
            Xs[e][tt] = tok0 + tt < T ? __half2float(A[ai]) + __half2float(A_lo[ai]) : 0.f;
        }
        __syncthreads();
#pragma unroll 8
        for (int e = 0; e < 32; ++e) {
            const float x0 = Xs[e][2 * tp], x1 = Xs[e][2 * tp + 1];
#pragma unroll
            for (int r = 0; r < ROWS; ++r) {
                const float w = Ws[e][tq * ROWS + r];
                acc[r][0] = fmaf(w, x0, acc[r][0]);
                acc[r][1] = fmaf(w, x1, acc[r][1]);
            }
        }
        __syncthreads();
    }
    const int task = task0 + tq;
    if (task >= n_tasks) return;
    unsigned long long best[2] = {0ull, 0ull};
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int t = tok0 + 2 * tp + j;
        if (t >= T) continue;
        float v0[4], v1[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            v0[r] = acc[r][j];
            v1[r] = acc[(ROWS == 8 ? 4 : 0) + r][j];
        }
        if (ROWS == 8) {
            epi_swiglu<OUT16>(a, t, 4 * task, v0, v1);
        } else {
            epi_quad<EPI>(a, layer, t, task * 4, N, v0, best[j]);
            if (EPI == EPI_LOGITS && best[j]) atomicMax(&a.amax_key[t], best[j]);
        }
    }
}

template <int QT, int ROWS, int EPI, bool OUT16>
cudaError_t run(const QMat &W, int n_tasks, int T, const __half *A, const __half *A_lo, const FwdArgs &a, int layer,
               cudaStream_t s) {
    dim3 grid((n_tasks + TASKS - 1) / TASKS, (T + TT - 1) / TT);
    return launch_pdl(k_gemm_simt<QT, ROWS, EPI, OUT16>, grid, dim3(256), 0, s, (const uint8_t *)W.w, W.N, W.nb,
                      n_tasks, T, A, A_lo, a, layer);
}

template <int QT>
cudaError_t dispatch(const QMat &W, Epi epi, int T, const __half *A, const __half *A_lo, const FwdArgs &a, int layer,
                     cudaStream_t s) {
    switch (epi) {
        case EPI_QKV: return run<QT, 4, EPI_QKV, false>(W, (W.N + 3) / 4, T, A, A_lo, a, layer, s);
        case EPI_RESID: return run<QT, 4, EPI_RESID, false>(W, (W.N + 3) / 4, T, A, A_lo, a, layer, s);
        case EPI_SWIGLU: return run<QT, 8, EPI_SWIGLU, true>(W, (a.F + 3) / 4, T, A, A_lo, a, layer, s);
        case EPI_LOGITS: return run<QT, 4, EPI_LOGITS, false>(W, (W.N + 3) / 4, T, A, A_lo, a, layer, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_gemm(const QMat &W, Epi epi, int T, const __half *A, const __half *A_lo, const FwdArgs &a,
                        int layer, cudaStream_t s, int64_t &launches, int64_t *wide) {
    // The tensor-core kernel is the GEMM; LCX_GEMM_SIMT=1 selects this CUDA-core version instead
    // (same results up to summation order), for cross-checking the two on a device.
    static const bool simt = [] {
        const char *e = getenv("LCX_GEMM_SIMT");
        return e && e[0] == '1';
    }();
    if (!simt) return launch_gemm_tc(W, epi, T, A, A_lo, a, layer, s, launches, wide);
    ++launches;
    if (W.type == Q4) return dispatch<Q4>(W, epi, T, A, A_lo, a, layer, s);
    if (W.type == Q8) return dispatch<Q8>(W, epi, T, A, A_lo, a, layer, s);
    return cudaErrorInvalidValue;
}

}  // namespace lcx
