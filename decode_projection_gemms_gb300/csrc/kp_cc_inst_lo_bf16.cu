// Instantiations of the CUDA-core split-K kernel for M = 1..8, bf16 elements.
#include "kp_cc_kernel.cuh"

namespace kp {
const CCKernelFn cc_table_lo_bf16[8][kCCVariants] = {
    KP_CC_ROW(1, KP_BF16),
    KP_CC_ROW(2, KP_BF16),
    KP_CC_ROW(3, KP_BF16),
    KP_CC_ROW(4, KP_BF16),
    KP_CC_ROW(5, KP_BF16),
    KP_CC_ROW(6, KP_BF16),
    KP_CC_ROW(7, KP_BF16),
    KP_CC_ROW(8, KP_BF16)};
}  // namespace kp
