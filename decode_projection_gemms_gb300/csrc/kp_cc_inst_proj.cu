// Instantiations of the CUDA-core single-launch projection kernel (bf16,
// M = 1..8).
#include "kp_cc_kernel.cuh"

namespace kp {
#define KP_CC_PROJ_ROW(M)                                                                  \
    {                                                                                      \
        cc_pick_proj<M, 0>(), cc_pick_proj<M, 1>(), cc_pick_proj<M, 2>(), cc_pick_proj<M, 3>(), \
            cc_pick_proj<M, 4>(), cc_pick_proj<M, 5>()                                     \
    }
const CCKernelFn cc_table_proj[8][kCCVariants] = {
    KP_CC_PROJ_ROW(1), KP_CC_PROJ_ROW(2), KP_CC_PROJ_ROW(3), KP_CC_PROJ_ROW(4),
    KP_CC_PROJ_ROW(5), KP_CC_PROJ_ROW(6), KP_CC_PROJ_ROW(7), KP_CC_PROJ_ROW(8)};
}  // namespace kp
