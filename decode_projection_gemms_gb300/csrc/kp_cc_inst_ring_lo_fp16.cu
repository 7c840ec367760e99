// Instantiations of the CUDA-core split-K kernel's shared-memory-ring form for
// M = 1..8, fp16 elements.
#include "kp_cc_kernel.cuh"

namespace kp {
const CCKernelFn cc_ring_lo_fp16[8][kCCVariants] = {
    KP_CC_RING_ROW(1, KP_FP16),
    KP_CC_RING_ROW(2, KP_FP16),
    KP_CC_RING_ROW(3, KP_FP16),
    KP_CC_RING_ROW(4, KP_FP16),
    KP_CC_RING_ROW(5, KP_FP16),
    KP_CC_RING_ROW(6, KP_FP16),
    KP_CC_RING_ROW(7, KP_FP16),
    KP_CC_RING_ROW(8, KP_FP16)};
}  // namespace kp
