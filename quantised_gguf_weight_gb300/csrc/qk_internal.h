// qk_internal.h -- declarations shared by the library's translation units.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace qk {

constexpr int kFmtQ80 = 0;
constexpr int kFmtQ4K = 1;
constexpr int kFmtQ6K = 2;
// Launch plan of one GEMV call (qk_gemv_kernel.cuh): team shape, K chunks,
// stage ring, shared-memory layout and grid.
struct GemvPlan {
    int U, LU, XU, SW, R, cpl, nkc, rows_w, chunk_bytes, row_stride;
    int nw, m, stages, stage_bytes, pair, up_stage_off, cpa;
    int wide;   // batch 1: the 16-warp form (Q4_K: a lane holds half a super-block at a time)
    int kw;     // consumer warps sharing a row group's K chunks (1: no split)
    int off_part;
    int off_x, off_xsum, off_xscale, off_xout, off_stage, smem, grid;
    int64_t row_bytes;
};

// pair: rows are output rows of the SwiGLU form (a gate row and an up row each).
// n_assign > 0: experts mode, `rows` rows per expert and n_assign assignments.
bool gemv_plan(int fmt, int64_t rows, int64_t K, int batch, bool pair, GemvPlan *p, int64_t n_assign = 0);
bool gemv_plan_host(int fmt, int64_t rows, int64_t K, int batch, bool pair, int64_t n_assign, int sms,
                    int smem_optin, GemvPlan *p);
cudaError_t gemv_launch(int fmt, const uint8_t *w_rows, int64_t rows, int64_t K, const float *x,
                        int batch, float *y, int64_t ldy, cudaStream_t st, const GemvPlan &p,
                        int *err, uint64_t wait_ns, int64_t skip_item, bool pdl, int64_t up_rows = 0,
                        const int32_t *expid = nullptr, int64_t n_experts = 0, int xk = 1);

// Plan of the batch 2..8 tensor-core GEMV (qk_gemv_tc.cu): groups of 32
// columns, 256-column items a tile, stage ring and shared-memory layout.
struct GemvTcPlan {
    int G, NC, chunk_bytes, row_stride, stage_bytes, NS;
    int off_bop, off_scale, off_xsum, off_out, off_flag, off_xch, off_stage, smem, grid;
    int ks, off_ksx;       // K split over CTA pairs (clusters of two), and its exchange buffers
    int64_t row_bytes;
};
bool gemv_tc_plan(int fmt, int64_t rows, int64_t K, GemvTcPlan *p);
bool gemv_tc_plan_for(int fmt, int64_t rows, int64_t K, int sms, int smem_optin, GemvTcPlan *p);
cudaError_t gemv_tc_launch(int fmt, const uint8_t *w_rows, int64_t rows, int64_t K, const float *x, int batch,
                           float *y, int64_t ldy, cudaStream_t st, const GemvTcPlan &p, int *err, uint64_t wait_ns,
                           bool pdl, int64_t skip_item = -1);
// The driver's tensor-map encoder (qk_gemm.cu), looked up once.
namespace gemm {
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn();
}  // namespace gemm
// SM count and shared memory per block (opt-in) of the current device.
bool device_limits(int *sms, int *smem_optin);

// The device error word of the current device and the bound of device waits.
int *library_error_word();
uint64_t library_wait_limit_ns();
// Strict-blocks mode: true when it is on and K is not a whole number of the
// format's blocks (32 columns for Q8_0, 256 for Q4_K and Q6_K).
bool strict_blocks_reject(int fmt, int64_t K);

int64_t gemm_k8(int64_t K);
// The argument checks shared by the prefill GEMM entry points (a qk_status;
// sets *ldy when it was 0 and *row_bytes); the workspace is checked only when
// check_workspace is true.
int gemm_check_args(int fmt, const void *w, int64_t row_offset, int64_t N, int64_t K, const float *x, int64_t M,
                    const float *y, int64_t *ldy, int64_t up_offset, const void *workspace, size_t workspace_bytes,
                    bool check_workspace, int64_t *row_bytes);
// The GEMM test hook's K chunk (-1: none).
int library_gemm_skip_chunk();
size_t gemm_workspace_bytes(int64_t M, int64_t K);
// Prefill GEMM of format fmt (kFmtQ4K or kFmtQ80).  mode 0: y = x W^T,
// 1: y += x W^T, 2: y = silu(x Wg^T) * (x Wu^T) with the up rows at
// w_rows + up_rows rows.
cudaError_t gemm_launch(int fmt, const uint8_t *w_rows, int64_t N, int64_t K, const float *x, int64_t M, float *y,
                        int64_t ldy, void *workspace, cudaStream_t st, int *err, uint64_t wait_ns, int skip_chunk,
                        bool *encode_failed, int mode = 0, int64_t up_rows = 0);
// The Q4_K store form (the plain prefill GEMM).
cudaError_t gemm_q4k_launch(const uint8_t *w_rows, int64_t N, int64_t K, const float *x, int64_t M, float *y,
                            int64_t ldy, void *workspace, cudaStream_t st, int *err, uint64_t wait_ns, int skip_chunk,
                            bool *encode_failed);

}  // namespace qk
