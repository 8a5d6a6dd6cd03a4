// qk_gemv_q6k.cu -- instantiations of the GEMV kernel for one weight
// format (its own translation unit so the kernels build in parallel).
#include "qk_gemv_kernel.cuh"

namespace qk {

cudaError_t gemv_launch_q6k(int batch, int us, const GemvArgs &a, int grid, int smem, cudaStream_t st, bool pdl)
{
    switch (batch) {
    case 1: QK_GEMV_DISPATCH_US(kFmtQ6K, 1, us)
    case 2: QK_GEMV_DISPATCH_US(kFmtQ6K, 2, us)
    case 3: QK_GEMV_DISPATCH_US(kFmtQ6K, 3, us)
    case 4: QK_GEMV_DISPATCH_US(kFmtQ6K, 4, us)
    case 5: QK_GEMV_DISPATCH_US(kFmtQ6K, 5, us)
    case 6: QK_GEMV_DISPATCH_US(kFmtQ6K, 6, us)
    case 7: QK_GEMV_DISPATCH_US(kFmtQ6K, 7, us)
    case 8: QK_GEMV_DISPATCH_US(kFmtQ6K, 8, us)
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qk
