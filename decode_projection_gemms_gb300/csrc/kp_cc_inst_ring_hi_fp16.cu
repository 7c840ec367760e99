// Instantiations of the CUDA-core split-K kernel's shared-memory-ring form for
// M = 9..16, fp16 elements.
#include "kp_cc_kernel.cuh"

namespace kp {
const CCKernelFn cc_ring_hi_fp16[8][kCCVariants] = {
    KP_CC_RING_ROW(9, KP_FP16),
    KP_CC_RING_ROW(10, KP_FP16),
    KP_CC_RING_ROW(11, KP_FP16),
    KP_CC_RING_ROW(12, KP_FP16),
    KP_CC_RING_ROW(13, KP_FP16),
    KP_CC_RING_ROW(14, KP_FP16),
    KP_CC_RING_ROW(15, KP_FP16),
    KP_CC_RING_ROW(16, KP_FP16)};
}  // namespace kp
