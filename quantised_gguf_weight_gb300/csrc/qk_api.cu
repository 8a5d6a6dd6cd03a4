// qk_api.cu -- the extern "C" entry points declared in include/qk.h.
//
// Host side only: argument validation (before any launch, outputs untouched
// on error), row-offset addressing, launch planning, the device error word
// and its read-back.  The compute runs entirely in the kernels of
// qk_gemv.cu and qk_gemm.cu; there is no host fallback of any kind.
#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <cuda_runtime.h>

#include "../../include/qk.h"
#include "qk_device.cuh"
#include "qk_internal.h"

namespace {

// Device error word: bit kErrTimeout is set by a kernel whose bounded wait ran
// out.  One per device (a __device__ variable lives in every context).
__device__ int g_qk_error_word;

std::atomic<uint64_t> g_wait_limit_ns{2000000000ull};
std::atomic<int64_t> g_skip_item{-1};
std::atomic<int> g_programmatic{0};
std::atomic<int> g_gemm_skip_chunk{-1};
// batch 2..8 on the tensor cores: 0 never, 1 where it is the faster form
// (the default), 2 wherever the format and K allow it (tests)
std::atomic<int> g_gemv_tc{1};

// Strict-blocks mode starts on when the environment sets QK_STRICT=1.
int strict_from_env()
{
    const char *v = std::getenv("QK_STRICT");
    return (v && std::strcmp(v, "1") == 0) ? 1 : 0;
}
std::atomic<int> g_strict_blocks{strict_from_env()};

// Device address of the error word per device, looked up once; host threads
// that make their first call on a device at the same time may both look it
// up, and store the same address.
std::atomic<int *> g_error_word_addr[64];

int *error_word_ptr()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    int *cached = g_error_word_addr[dev].load(std::memory_order_acquire);
    if (!cached) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_qk_error_word) != cudaSuccess) return nullptr;
        cached = static_cast<int *>(p);
        g_error_word_addr[dev].store(cached, std::memory_order_release);
    }
    return cached;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int gemv_entry(int fmt, const void *w, int64_t row_offset, int64_t rows, int64_t K,
               const float *x, int batch, float *y, int64_t ldy, qk_stream_t stream,
               int64_t up_offset = -1)
{
    const bool pair = up_offset >= 0;
    if (!w || !x || !y) return QK_ERR_NULL;
    if (rows <= 0 || K <= 0 || row_offset < 0) return QK_ERR_BAD_DIM;
    if (batch < 1 || batch > QK_MAX_BATCH) return QK_ERR_BATCH;
    if (ldy == 0) ldy = rows;
    if (ldy < rows) return QK_ERR_BAD_DIM;
    if (qk::strict_blocks_reject(fmt, K)) return QK_ERR_BAD_DIM;
    if (!aligned(w, fmt == qk::kFmtQ4K ? 16 : 2) || !aligned(x, 4) || !aligned(y, 4))
        return QK_ERR_ALIGN;
    // batch 2..8 of Q8_0 / Q4_K: the tensor-core form where the format and
    // K allow it and it is the faster form: every SM gets at least one whole
    // 128-row tile (the tensor cores work on 128 rows whatever their number)
    // and, for Q4_K, the batch is 4 or more (at batch 2 and 3 the fp32 form
    // keeps up with its 4-bit weights)
    const int tc_mode = g_gemv_tc.load();
    if (!pair && batch >= 2 && tc_mode != 0) {
        qk::GemvTcPlan tp;
        int sms = 0, smem = 0;
        const bool faster = qk::device_limits(&sms, &smem) && rows >= 128LL * sms &&
                            (fmt == qk::kFmtQ80 || batch >= 4);
        if ((tc_mode == 2 || faster) && qk::gemv_tc_plan(fmt, rows, K, &tp)) {
            if (row_offset > (INT64_MAX / tp.row_bytes) - rows) return QK_ERR_BAD_DIM;
            int *err = error_word_ptr();
            if (!err) return QK_ERR_CUDA;
            const uint8_t *w_rows = static_cast<const uint8_t *>(w) + row_offset * tp.row_bytes;
            cudaError_t e = qk::gemv_tc_launch(fmt, w_rows, rows, K, x, batch, y, ldy,
                                               reinterpret_cast<cudaStream_t>(stream), tp, err, g_wait_limit_ns.load(),
                                               g_programmatic.load() != 0, g_skip_item.load());
            return e == cudaSuccess ? QK_OK : QK_ERR_CUDA;
        }
    }
    // the kernel keeps a launch's activation rows in shared memory: a batch
    // whose activations do not fit is cut into launches of fewer rows (as
    // even as possible); only a single row that does not fit is refused
    qk::GemvPlan plan;
    int bmax = batch;
    while (bmax > 0 && !qk::gemv_plan(fmt, rows, K, bmax, pair, &plan)) --bmax;
    if (bmax == 0) {
        // either no usable device or one activation row does not fit
        int dev_count = 0;
        if (cudaGetDeviceCount(&dev_count) != cudaSuccess || dev_count == 0) return QK_ERR_CUDA;
        return QK_ERR_TOO_LARGE;
    }
    const int64_t last = pair ? (row_offset > up_offset ? row_offset : up_offset) : row_offset;
    if (last > (INT64_MAX / plan.row_bytes) - rows) return QK_ERR_BAD_DIM;
    int *err = error_word_ptr();
    if (!err) return QK_ERR_CUDA;
    const uint8_t *w_rows = static_cast<const uint8_t *>(w) + row_offset * plan.row_bytes;
    const int parts = (batch + bmax - 1) / bmax;
    for (int p = 0, b0 = 0, planned = bmax; p < parts; ++p) {
        const int nb = (batch - b0) / (parts - p);
        if (nb != planned) {
            if (!qk::gemv_plan(fmt, rows, K, nb, pair, &plan)) return QK_ERR_CUDA;
            planned = nb;
        }
        cudaError_t e = qk::gemv_launch(fmt, w_rows, rows, K, x + static_cast<int64_t>(b0) * K, nb,
                                        y + static_cast<int64_t>(b0) * ldy, ldy,
                                        reinterpret_cast<cudaStream_t>(stream), plan, err,
                                        g_wait_limit_ns.load(), g_skip_item.load(), g_programmatic.load() != 0,
                                        pair ? up_offset - row_offset : 0);
        if (e != cudaSuccess) return QK_ERR_CUDA;
        b0 += nb;
    }
    return QK_OK;
}

}  // namespace

namespace qk {
int *library_error_word() { return error_word_ptr(); }
uint64_t library_wait_limit_ns() { return g_wait_limit_ns.load(); }
bool strict_blocks_reject(int fmt, int64_t K)
{
    const int64_t qk = fmt == kFmtQ80 ? 32 : 256;
    return g_strict_blocks.load() != 0 && K % qk != 0;
}
}  // namespace qk

extern "C" {

size_t qgemm_q4_k_workspace_bytes(int64_t M, int64_t N, int64_t K)
{
    (void)N;
    if (M <= 0 || K <= 0) return 0;
    return qk::gemm_workspace_bytes(M, K);
}

}  // extern "C"

namespace {

}  // namespace

namespace qk {
// Argument checks of every prefill GEMM entry point, in the order of their
// statuses; the workspace is checked by the caller (between the alignment
// and size checks), so the same checks serve the workspace-free entry point.
int gemm_check_args(int fmt, const void *w, int64_t row_offset, int64_t N, int64_t K, const float *x, int64_t M,
                    const float *y, int64_t *ldy, int64_t up_offset, const void *workspace, size_t workspace_bytes,
                    bool check_workspace, int64_t *row_bytes)
{
    if (!w || !x || !y) return QK_ERR_NULL;
    if (N <= 0 || K <= 0 || M <= 0 || row_offset < 0 || up_offset < 0) return QK_ERR_BAD_DIM;
    if (*ldy == 0) *ldy = N;
    if (*ldy < N) return QK_ERR_BAD_DIM;
    if (strict_blocks_reject(fmt, K)) return QK_ERR_BAD_DIM;
    if (!aligned(w, fmt == kFmtQ4K ? 16 : 2) || !aligned(x, 4) || !aligned(y, 4)) return QK_ERR_ALIGN;
    if (check_workspace &&
        (!workspace || !aligned(workspace, 256) || workspace_bytes < gemm_workspace_bytes(M, K)))
        return QK_ERR_WORKSPACE;
    // tensor-map limits: at most 2^31 tokens and rows per call
    const int64_t last = row_offset > up_offset ? row_offset : up_offset;
    if (M > (1LL << 31) - 1 || K > (1LL << 31) - 1 || last > (1LL << 31) - 1 - N) return QK_ERR_TOO_LARGE;
    *row_bytes = fmt == kFmtQ4K ? ((K + 255) / 256) * 144 : ((K + 31) / 32) * 34;
    if (last > (INT64_MAX / *row_bytes) - N) return QK_ERR_BAD_DIM;
    return QK_OK;
}
int library_gemm_skip_chunk() { return g_gemm_skip_chunk.load(); }
}  // namespace qk

namespace {

int gemm_entry(int fmt, const void *w, int64_t row_offset, int64_t N, int64_t K, const float *x, int64_t M, float *y,
               int64_t ldy, void *workspace, size_t workspace_bytes, qk_stream_t stream, int mode,
               int64_t up_offset)
{
    int64_t row_bytes = 0;
    const int st = qk::gemm_check_args(fmt, w, row_offset, N, K, x, M, y, &ldy, up_offset, workspace,
                                       workspace_bytes, true, &row_bytes);
    if (st != QK_OK) return st;
    int *err = error_word_ptr();
    if (!err) return QK_ERR_CUDA;
    const uint8_t *w_rows = static_cast<const uint8_t *>(w) + row_offset * row_bytes;
    bool encode_failed = false;
    cudaError_t e = qk::gemm_launch(fmt, w_rows, N, K, x, M, y, ldy, workspace,
                                    reinterpret_cast<cudaStream_t>(stream), err, g_wait_limit_ns.load(),
                                    g_gemm_skip_chunk.load(), &encode_failed, mode, up_offset - row_offset);
    if (encode_failed) return QK_ERR_CUDA;
    return e == cudaSuccess ? QK_OK : QK_ERR_CUDA;
}

}  // namespace

extern "C" {

int qgemm_q4_k(const void *w, int64_t row_offset, int64_t N, int64_t K, const float *x, int64_t M, float *y,
               int64_t ldy, void *workspace, size_t workspace_bytes, qk_stream_t stream)
{
    return gemm_entry(qk::kFmtQ4K, w, row_offset, N, K, x, M, y, ldy, workspace, workspace_bytes, stream, 0, 0);
}

int qgemm_q4_k_acc(const void *w, int64_t row_offset, int64_t N, int64_t K, const float *x, int64_t M, float *y,
                   int64_t ldy, void *workspace, size_t workspace_bytes, qk_stream_t stream)
{
    return gemm_entry(qk::kFmtQ4K, w, row_offset, N, K, x, M, y, ldy, workspace, workspace_bytes, stream, 1, 0);
}

int qgemm_q8_0(const void *w, int64_t row_offset, int64_t N, int64_t K, const float *x, int64_t M, float *y,
               int64_t ldy, void *workspace, size_t workspace_bytes, qk_stream_t stream)
{
    return gemm_entry(qk::kFmtQ80, w, row_offset, N, K, x, M, y, ldy, workspace, workspace_bytes, stream, 0, 0);
}

int qgemm_q8_0_acc(const void *w, int64_t row_offset, int64_t N, int64_t K, const float *x, int64_t M, float *y,
                   int64_t ldy, void *workspace, size_t workspace_bytes, qk_stream_t stream)
{
    return gemm_entry(qk::kFmtQ80, w, row_offset, N, K, x, M, y, ldy, workspace, workspace_bytes, stream, 1, 0);
}

int qgemm_swiglu_q8_0(const void *w, int64_t gate_offset, int64_t up_offset, int64_t F, int64_t K, const float *x,
                      int64_t M, float *h, int64_t ldh, void *workspace, size_t workspace_bytes, qk_stream_t stream)
{
    return gemm_entry(qk::kFmtQ80, w, gate_offset, F, K, x, M, h, ldh, workspace, workspace_bytes, stream, 2,
                      up_offset);
}

int qgemm_swiglu_q4_k(const void *w, int64_t gate_offset, int64_t up_offset, int64_t F, int64_t K, const float *x,
                      int64_t M, float *h, int64_t ldh, void *workspace, size_t workspace_bytes, qk_stream_t stream)
{
    return gemm_entry(qk::kFmtQ4K, w, gate_offset, F, K, x, M, h, ldh, workspace, workspace_bytes, stream, 2, up_offset);
}

int qmatvec_q8_0(const void *w, int64_t row_offset, int64_t rows, int64_t K, const float *x,
                 int batch, float *y, int64_t ldy, qk_stream_t stream)
{
    return gemv_entry(qk::kFmtQ80, w, row_offset, rows, K, x, batch, y, ldy, stream);
}

int qmatvec_q4_k(const void *w, int64_t row_offset, int64_t rows, int64_t K, const float *x,
                 int batch, float *y, int64_t ldy, qk_stream_t stream)
{
    return gemv_entry(qk::kFmtQ4K, w, row_offset, rows, K, x, batch, y, ldy, stream);
}

int qmatvec_q6_k(const void *w, int64_t row_offset, int64_t rows, int64_t K, const float *x,
                 int batch, float *y, int64_t ldy, qk_stream_t stream)
{
    return gemv_entry(qk::kFmtQ6K, w, row_offset, rows, K, x, batch, y, ldy, stream);
}

int qmatvec_swiglu_q6_k(const void *w, int64_t gate_offset, int64_t up_offset, int64_t F, int64_t K,
                        const float *x, int batch, float *h, int64_t ldh, qk_stream_t stream)
{
    if (up_offset < 0) return QK_ERR_BAD_DIM;
    return gemv_entry(qk::kFmtQ6K, w, gate_offset, F, K, x, batch, h, ldh, stream, up_offset);
}

int qmatvec_swiglu_q8_0(const void *w, int64_t gate_offset, int64_t up_offset, int64_t F, int64_t K,
                        const float *x, int batch, float *h, int64_t ldh, qk_stream_t stream)
{
    if (up_offset < 0) return QK_ERR_BAD_DIM;
    return gemv_entry(qk::kFmtQ80, w, gate_offset, F, K, x, batch, h, ldh, stream, up_offset);
}

int qmatvec_swiglu_q4_k(const void *w, int64_t gate_offset, int64_t up_offset, int64_t F, int64_t K,
                        const float *x, int batch, float *h, int64_t ldh, qk_stream_t stream)
{
    if (up_offset < 0) return QK_ERR_BAD_DIM;
    return gemv_entry(qk::kFmtQ4K, w, gate_offset, F, K, x, batch, h, ldh, stream, up_offset);
}

}  // extern "C"

namespace {

int experts_entry(int fmt, const void *w, int64_t n_experts, int64_t rows, int64_t K, const float *x, int xk,
                  const int32_t *expert_ids, int64_t n_assign, float *y, int64_t ldy, qk_stream_t stream)
{
    if (!w || !x || !y || !expert_ids) return QK_ERR_NULL;
    if (n_experts <= 0 || rows <= 0 || K <= 0 || xk <= 0 || n_assign <= 0) return QK_ERR_BAD_DIM;
    if (ldy == 0) ldy = rows;
    if (ldy < rows) return QK_ERR_BAD_DIM;
    if (qk::strict_blocks_reject(fmt, K)) return QK_ERR_BAD_DIM;
    if (!aligned(w, fmt == qk::kFmtQ4K ? 16 : 2) || !aligned(x, 4) || !aligned(y, 4) || !aligned(expert_ids, 4))
        return QK_ERR_ALIGN;
    qk::GemvPlan plan;
    if (!qk::gemv_plan(fmt, rows, K, 1, false, &plan, n_assign)) {
        int dev_count = 0;
        if (cudaGetDeviceCount(&dev_count) != cudaSuccess || dev_count == 0) return QK_ERR_CUDA;
        return QK_ERR_TOO_LARGE;
    }
    if (n_experts > (INT64_MAX / plan.row_bytes) / rows) return QK_ERR_BAD_DIM;
    int *err = error_word_ptr();
    if (!err) return QK_ERR_CUDA;
    cudaError_t e = qk::gemv_launch(fmt, static_cast<const uint8_t *>(w), rows, K, x, 1, y, ldy,
                                    reinterpret_cast<cudaStream_t>(stream), plan, err, g_wait_limit_ns.load(),
                                    g_skip_item.load(), g_programmatic.load() != 0, 0, expert_ids, n_experts, xk);
    return e == cudaSuccess ? QK_OK : QK_ERR_CUDA;
}

}  // namespace

extern "C" {

int qmatvec_experts_q8_0(const void *w, int64_t n_experts, int64_t rows, int64_t K, const float *x, int xk,
                         const int32_t *expert_ids, int64_t n_assign, float *y, int64_t ldy, qk_stream_t stream)
{
    return experts_entry(qk::kFmtQ80, w, n_experts, rows, K, x, xk, expert_ids, n_assign, y, ldy, stream);
}

int qmatvec_experts_q4_k(const void *w, int64_t n_experts, int64_t rows, int64_t K, const float *x, int xk,
                         const int32_t *expert_ids, int64_t n_assign, float *y, int64_t ldy, qk_stream_t stream)
{
    return experts_entry(qk::kFmtQ4K, w, n_experts, rows, K, x, xk, expert_ids, n_assign, y, ldy, stream);
}

int qmatvec_experts_q6_k(const void *w, int64_t n_experts, int64_t rows, int64_t K, const float *x, int xk,
                         const int32_t *expert_ids, int64_t n_assign, float *y, int64_t ldy, qk_stream_t stream)
{
    return experts_entry(qk::kFmtQ6K, w, n_experts, rows, K, x, xk, expert_ids, n_assign, y, ldy, stream);
}

int64_t qk_row_bytes_q6_k(int64_t K) { return K <= 0 ? 0 : ((K + 255) / 256) * 210; }

int64_t qk_row_bytes_q8_0(int64_t K) { return K <= 0 ? 0 : ((K + 31) / 32) * 34; }
int64_t qk_row_bytes_q4_k(int64_t K) { return K <= 0 ? 0 : ((K + 255) / 256) * 144; }

const char *qk_status_string(int status)
{
    switch (status) {
    case QK_OK: return "ok";
    case QK_ERR_NULL: return "null pointer argument";
    case QK_ERR_BAD_DIM:
        return "bad dimension (rows/N/M/K <= 0, negative row_offset, ldy too small, or in strict-blocks mode "
               "K not a whole number of blocks)";
    case QK_ERR_ALIGN: return "misaligned pointer";
    case QK_ERR_BATCH: return "batch outside [1, 8]";
    case QK_ERR_CUDA: return "CUDA error";
    case QK_ERR_TIMEOUT: return "a bounded device wait ran out";
    case QK_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case QK_ERR_TOO_LARGE: return "size beyond what the kernels support";
    case QK_ERR_BAD_INDEX: return "an index read from device memory was out of range";
    default: return "unknown status";
    }
}

int qk_device_error(qk_stream_t stream)
{
    int *err = error_word_ptr();
    if (!err) return QK_ERR_CUDA;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return QK_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return QK_ERR_CUDA;
    if (v) {
        const int zero = 0;
        if (cudaMemcpy(err, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return QK_ERR_CUDA;
        return (v & qk::kErrBadIndex) ? QK_ERR_BAD_INDEX : QK_ERR_TIMEOUT;
    }
    return QK_OK;
}

uint64_t qk_set_wait_limit_ns(uint64_t ns)
{
    if (ns == 0) ns = 1;
    return g_wait_limit_ns.exchange(ns);
}

int qk_set_programmatic_launch(int enable) { return g_programmatic.exchange(enable ? 1 : 0); }

int qk_set_strict_blocks(int enable) { return g_strict_blocks.exchange(enable ? 1 : 0); }

int qk_version(void) { return 100; }

// Test hook, not part of the public header: in CTA 0 of every later GEMV
// launch, consumer warp 0's item number `item` (the tensor-core form: the
// CTA's item `item`) is never copied (-1 restores normal operation), so a
// bounded wait runs out and the launch records QK_ERR_TIMEOUT.
int64_t qk_debug_skip_item(int64_t item) { return g_skip_item.exchange(item); }

// Test hook: the launch plan a GEMV call of this shape would use, as
// {SW, R, nkc, rows_w, stages, stage_bytes, smem, grid, XU, cpl, nw, m}; returns the
// number of values written, or -1 if no plan fits.
int qk_debug_gemv_plan(int fmt, int64_t rows, int64_t K, int batch, int64_t *out, int n)
{
    qk::GemvPlan p;
    if (!out || !qk::gemv_plan(fmt, rows, K, batch, false, &p)) return -1;
    const int64_t v[12] = {p.SW, p.R, p.nkc, p.rows_w, p.stages, p.stage_bytes, p.smem, p.grid, p.XU, p.cpl, p.nw, p.m};
    int k = 0;
    for (; k < n && k < 12; ++k) out[k] = v[k];
    return k;
}

// Test hook, not part of the public header: the GEMV plan for an explicit
// device (SM count, shared memory per block), computed on the host only.
// Fields: SW, R, nkc, rows_w, stages, stage_bytes, smem, grid, XU, cpl, nw,
// m, LU, cpa, off_stage, wide, kw.  Returns the number written, -1 if nothing fits.
int qk_debug_gemv_plan_for(int fmt, int64_t rows, int64_t K, int batch, int pair, int64_t n_assign, int sms,
                           int smem_optin, int64_t *out, int n)
{
    qk::GemvPlan p;
    if (!out || fmt < 0 || fmt > 2 || batch < 1 || batch > QK_MAX_BATCH || rows <= 0 || K <= 0 ||
        !qk::gemv_plan_host(fmt, rows, K, batch, pair != 0, n_assign, sms, smem_optin, &p))
        return -1;
    const int64_t v[17] = {p.SW, p.R, p.nkc, p.rows_w, p.stages, p.stage_bytes, p.smem, p.grid,
                           p.XU, p.cpl, p.nw, p.m, p.LU, p.cpa, p.off_stage, p.wide, p.kw};
    int k = 0;
    for (; k < n && k < 17; ++k) out[k] = v[k];
    return k;
}

// Test hook, not part of the public header: the tensor-core form of later
// batch 2..8 GEMV calls: 0 never (the fp32 form), 1 where it is the faster
// form (the default), 2 wherever the format and K allow it.  Returns the
// previous setting.
int qk_debug_gemv_tc(int mode) { return g_gemv_tc.exchange(mode < 0 ? 0 : (mode > 2 ? 2 : mode)); }

// Test hook, not part of the public header: the tensor-core GEMV plan for an
// explicit device, as {G, NC, row_stride, stage_bytes, NS, smem, grid,
// off_stage, off_bop, ks}; -1 when the format and K do not take that form.
int qk_debug_gemv_tc_plan_for(int fmt, int64_t rows, int64_t K, int sms, int smem_optin, int64_t *out, int n)
{
    qk::GemvTcPlan p;
    if (!out || !qk::gemv_tc_plan_for(fmt, rows, K, sms, smem_optin, &p)) return -1;
    const int64_t v[10] = {p.G, p.NC, p.row_stride, p.stage_bytes, p.NS, p.smem, p.grid, p.off_stage, p.off_bop, p.ks};
    int k = 0;
    for (; k < n && k < 10; ++k) out[k] = v[k];
    return k;
}

// Test hook, not part of the public header: CTA 0 of every later GEMM launch
// never loads the activations of K chunk `chunk` (-1 restores normal
// operation), so the MMA issuer's bounded wait runs out (QK_ERR_TIMEOUT).
int qk_debug_gemm_skip_chunk(int chunk) { return g_gemm_skip_chunk.exchange(chunk); }

}  // extern "C"
