// qk_gemv_q80.cu -- instantiations of the GEMV kernel for one weight
// format (its own translation unit so the kernels build in parallel).
#include "qk_gemv_kernel.cuh"

namespace qk {

cudaError_t gemv_launch_q80(int batch, int us, const GemvArgs &a, int grid, int smem, cudaStream_t st, bool pdl)
{
    switch (batch) {
    case 1: QK_GEMV_DISPATCH_US(kFmtQ80, 1, us)
    case 2: QK_GEMV_DISPATCH_US(kFmtQ80, 2, us)
    case 3: QK_GEMV_DISPATCH_US(kFmtQ80, 3, us)
    case 4: QK_GEMV_DISPATCH_US(kFmtQ80, 4, us)
    case 5: QK_GEMV_DISPATCH_US(kFmtQ80, 5, us)
    case 6: QK_GEMV_DISPATCH_US(kFmtQ80, 6, us)
    case 7: QK_GEMV_DISPATCH_US(kFmtQ80, 7, us)
    case 8: QK_GEMV_DISPATCH_US(kFmtQ80, 8, us)
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qk
