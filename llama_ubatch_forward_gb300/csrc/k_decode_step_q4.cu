// Instantiations of the persistent decode step for Q4_0 layer weights and a Q8_0 head.
#include "k_decode_step.cuh"

namespace lcx {
namespace step_detail {

const void *step_kernel_q4(int hd, int g) {
#define LCX_STEP_K(HD, G) if (hd == HD && g == G) return (const void *)k_decode_step<Q4, Q8, HD, G>;
    LCX_STEP_K(64, 1) LCX_STEP_K(64, 2) LCX_STEP_K(64, 4) LCX_STEP_K(64, 8)
    LCX_STEP_K(128, 1) LCX_STEP_K(128, 2) LCX_STEP_K(128, 4) LCX_STEP_K(128, 8)
#undef LCX_STEP_K
    return nullptr;
}

}  // namespace step_detail
}  // namespace lcx
