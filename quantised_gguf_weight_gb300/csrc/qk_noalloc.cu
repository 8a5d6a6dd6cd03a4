// qk_noalloc.cu -- qgemm_q4_k_noalloc: the prefill GEMM without a
// caller-supplied workspace.
//
// Some callers cannot allocate device memory at the point where they run the
// GEMM: a plugin hosted by an inference engine that owns every device
// allocation, or code that must not allocate once it has started (a fixed,
// audited memory footprint).  Such callers cannot provide the workspace that
// qgemm_q4_k takes.  This entry point uses instead a scratch array that lives
// in this file as a __device__ variable: every GPU that loads the library
// holds it (kQkNoallocScratchBytes) until the process exits, and no call
// allocates or frees anything.
//
// In host code the array's name is only a host-side stand-in, not a device
// address, so its device address is looked up with cudaGetSymbolAddress,
// once per device, on the first call made while that device is current.
// That first call should therefore come before any stream capture.  Every
// call shares the one array; calls that overlap on the GPU (for instance on
// two streams at once) race on it.  Nothing in it has to start at zero: the
// bf16 pre-pass rewrites every byte the GEMM reads (padding included).
#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/qk.h"
#include "qk_internal.h"

namespace {

constexpr size_t kQkNoallocScratchBytes = QK_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_qk_noalloc_scratch[kQkNoallocScratchBytes];

// Device address of the scratch array per device; nullptr until looked up.
// Host threads that make their first call on a device at the same time may
// both look it up and store the same address.
std::atomic<void *> g_scratch_addr[64];

void *scratch_address(int dev)
{
    void *cached = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (!cached) {
        if (cudaGetSymbolAddress(&cached, g_qk_noalloc_scratch) != cudaSuccess) return nullptr;
        g_scratch_addr[dev].store(cached, std::memory_order_release);
    }
    return cached;
}

}  // namespace

extern "C" {

int qgemm_q4_k_noalloc(const void *w, int64_t row_offset, int64_t N, int64_t K, const float *x, int64_t M, float *y,
                       int64_t ldy, qk_stream_t stream)
{
    // the same checks, in the same order, as qgemm_q4_k (no workspace)
    int64_t row_bytes = 0;
    const int st = qk::gemm_check_args(qk::kFmtQ4K, w, row_offset, N, K, x, M, y, &ldy, 0, nullptr, 0, false,
                                       &row_bytes);
    if (st != QK_OK) return st;
    // the bf16 copy of x has to fit in the fixed scratch array
    if (qk::gemm_workspace_bytes(M, K) > kQkNoallocScratchBytes) return QK_ERR_TOO_LARGE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return QK_ERR_CUDA;
    void *scratch = scratch_address(dev);
    int *err = qk::library_error_word();
    if (!scratch || !err) return QK_ERR_CUDA;
    const uint8_t *w_rows = static_cast<const uint8_t *>(w) + row_offset * row_bytes;
    bool encode_failed = false;
    cudaError_t e = qk::gemm_q4k_launch(w_rows, N, K, x, M, y, ldy, scratch, reinterpret_cast<cudaStream_t>(stream),
                                        err, qk::library_wait_limit_ns(), qk::library_gemm_skip_chunk(),
                                        &encode_failed);
    if (encode_failed) return QK_ERR_CUDA;
    return e == cudaSuccess ? QK_OK : QK_ERR_CUDA;
}

}  // extern "C"
