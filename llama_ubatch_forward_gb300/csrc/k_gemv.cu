// Entry points of the weight-streaming GEMV (kernel in k_gemv.cuh, instantiations per block
// type in k_gemv_q4.cu / k_gemv_q8.cu).
#include "k_gemv.cuh"

namespace lcx {
namespace gemv_detail {
cudaError_t dispatch_q4(const GemvParams &p, Epi epi, const FwdArgs &a, int layer, cudaStream_t s);
cudaError_t dispatch_q8(const GemvParams &p, Epi epi, const FwdArgs &a, int layer, cudaStream_t s);
}  // namespace gemv_detail

bool gemv_fits(const QMat &W, int T) {
    int nt = T <= 1 ? 1 : T <= 2 ? 2 : T <= 4 ? 4 : 8;
    if (T > kGemvMaxT || (size_t)nt * gemv_detail::stage_bytes_per_token(W.nb) > (size_t)kGemvSmemX) return false;
    const gemv_detail::StagePlan pl = gemv_detail::stage_plan(W.nb, W.type == Q8 ? 32 : 16, nt, false, kGemvSmemTotal);
    return pl.slots >= 2;
}

cudaError_t launch_gemv(const QMat &W, Epi epi, int T, const GemvIn &in, const FwdArgs &a, int layer, cudaStream_t s,
                        int64_t &launches) {
    gemv_detail::GemvParams p;
    p.w = W.w;
    p.N = W.N;
    p.nb = W.nb;
    p.K = W.K;
    p.T = T;
    p.in = in;
    p.n_tasks = epi == EPI_SWIGLU ? (a.F + 1) / 2 : (W.N + 3) / 4;
    ++launches;
    if (W.type == Q4) return gemv_detail::dispatch_q4(p, epi, a, layer, s);
    if (W.type == Q8) return gemv_detail::dispatch_q8(p, epi, a, layer, s);
    return cudaErrorInvalidValue;
}

}  // namespace lcx
