// Instantiations of the weight-streaming GEMV for Q4_0 weights (split from the other block
// type so the two compile in parallel).
#include "k_gemv.cuh"

namespace lcx {
namespace gemv_detail {

template <int QT, int EPI, bool OUT16>
static cudaError_t dispatch_nt(const GemvParams &p, const FwdArgs &a, int layer, cudaStream_t s) {
    if (p.T <= 1) return run<QT, 1, EPI, OUT16>(p, a, layer, s);
    if (p.T <= 2) return run<QT, 2, EPI, OUT16>(p, a, layer, s);
    if (p.T <= 4) return run<QT, 4, EPI, OUT16>(p, a, layer, s);
    return run<QT, 8, EPI, OUT16>(p, a, layer, s);
}

cudaError_t dispatch_q4(const GemvParams &p, Epi epi, const FwdArgs &a, int layer, cudaStream_t s) {
    switch (epi) {
        case EPI_QKV: return dispatch_nt<Q4, EPI_QKV, false>(p, a, layer, s);
        case EPI_RESID: return dispatch_nt<Q4, EPI_RESID, false>(p, a, layer, s);
        case EPI_SWIGLU: return dispatch_nt<Q4, EPI_SWIGLU, false>(p, a, layer, s);
        case EPI_LOGITS: return dispatch_nt<Q4, EPI_LOGITS, false>(p, a, layer, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gemv_detail
}  // namespace lcx
