// qk_gemv_q6k.cu -- instantiations of the GEMV kernel for one weight
// format (its own translation unit so the kernels build in parallel).
#include "qk_gemv_kernel.cuh"

namespace qk {

cudaError_t gemv_launch_q6k(int batch, bool wide, const GemvArgs &a, int grid, int smem, cudaStream_t st, bool pdl)
{
    switch (batch) {
    case 1:
        if (!a.pair && a.cpa == 0 && a.kw == 1)   // the plain forms (no pair or experts code)
            return wide ? gemv_launch_one<kFmtQ6K, 1, true, kModePlainKw1>(a, grid, smem, st, pdl)
                        : gemv_launch_one<kFmtQ6K, 1, false, kModePlainKw1>(a, grid, smem, st, pdl);
        if (!a.pair && a.cpa == 0)
            return wide ? gemv_launch_one<kFmtQ6K, 1, true, kModePlain>(a, grid, smem, st, pdl)
                        : gemv_launch_one<kFmtQ6K, 1, false, kModePlain>(a, grid, smem, st, pdl);
        return wide ? gemv_launch_one<kFmtQ6K, 1, true>(a, grid, smem, st, pdl)
                    : gemv_launch_one<kFmtQ6K, 1>(a, grid, smem, st, pdl);
    case 2: return gemv_launch_one<kFmtQ6K, 2>(a, grid, smem, st, pdl);
    case 3: return gemv_launch_one<kFmtQ6K, 3>(a, grid, smem, st, pdl);
    case 4: return gemv_launch_one<kFmtQ6K, 4>(a, grid, smem, st, pdl);
    case 5: return gemv_launch_one<kFmtQ6K, 5>(a, grid, smem, st, pdl);
    case 6: return gemv_launch_one<kFmtQ6K, 6>(a, grid, smem, st, pdl);
    case 7: return gemv_launch_one<kFmtQ6K, 7>(a, grid, smem, st, pdl);
    case 8: return gemv_launch_one<kFmtQ6K, 8>(a, grid, smem, st, pdl);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qk
