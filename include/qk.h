/*
 * qk.h -- C ABI of the GB300 (sm_103a) quantised-weight GEMV / GEMM library.
 *
 * The library multiplies GGUF block-quantised weights by fp32 activations,
 * decoding every block inside the multiply.  That is what the nurllama
 * runtime does with weight types it has a device kernel for: their GGUF bytes
 * go to the device unchanged and each block is decoded inside the matmul
 * (nurllama 0.18.1 API reference, model.nu), through its quantised matvec
 * dispatch `lk_matvec_q ks gt wd xd yd rows cols batch` (same page,
 * kernels.nu).  One entry point per weight format; there is no
 * type dispatch and no host fallback.
 *
 * Operation (every entry point):
 *   y[b][r] = sum_{c < K} W[row_offset + r][c] * x[b][c]
 * with W row-major, the column index fastest: row r of W starts at element
 * r*K (the layout contract of kernels.nu).
 *
 * Block formats (the pages name them, the bytes follow the GGUF layouts):
 *   Q8_0 : 34-byte blocks of 32 weights: fp16 d, then 32 int8 q;  w = d*q.
 *   Q4_K : 144-byte super-blocks of 256 weights: fp16 d, fp16 dmin, 12 bytes
 *          of packed 6-bit sub-block scales sc and mins m (8 sub-blocks of
 *          32), 128 bytes of 4-bit quants q;  w = d*sc*q - dmin*m.
 *   A row holds ceil(K / 32) (Q8_0) or ceil(K / 256) (Q4_K, Q6_K) whole
 *   blocks; columns >= K inside a row's last block are ignored.  In
 *   strict-blocks mode (qk_set_strict_blocks) a K that is not a whole number
 *   of blocks is refused instead (QK_ERR_BAD_DIM).
 *
 * Row addressing: `w` points at the first byte of the whole tensor, and a call
 * uses rows [row_offset, row_offset + rows).  Row r starts at byte
 * r * row_bytes with row_bytes = blocks_per_row * block_bytes.  This is how
 * the parts of a fused tensor are addressed (in nurllama too a weight is a
 * device pointer with a row count and the parts of a fused tensor are ranges
 * of its rows: nurllama README, "What it runs", phi3), and how one expert of
 * a 3-D expert tensor [E][rows_e][K] is addressed: row_offset = e*rows_e + r0.
 *
 * Ownership and execution: every pointer is a device pointer owned by the
 * caller; the library allocates and frees nothing per call and keeps no
 * per-call state.  Calls are asynchronous on `stream` (NULL = the legacy
 * default stream) and never synchronise.
 *
 * Errors: argument errors are detected on the host before any launch and
 * leave every output untouched; a failed launch returns QK_ERR_CUDA.  Device
 * waits are bounded: a kernel whose wait runs out records the fact in a
 * device error word and returns early (its outputs are then unspecified);
 * qk_device_error() reads and clears that word.
 */
#ifndef QK_H
#define QK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *qk_stream_t;

typedef enum {
    QK_OK = 0,
    QK_ERR_NULL = 1,        /* a required pointer is NULL                              */
    QK_ERR_BAD_DIM = 2,     /* rows/N/M <= 0, K <= 0, row_offset < 0, ldy too small;
                               strict-blocks mode: K not a whole number of blocks      */
    QK_ERR_ALIGN = 3,       /* w, x or y misaligned (see each call)                     */
    QK_ERR_BATCH = 4,       /* GEMV batch outside [1, QK_MAX_BATCH]                     */
    QK_ERR_CUDA = 5,        /* a CUDA runtime call or launch failed                     */
    QK_ERR_TIMEOUT = 6,     /* a bounded device wait ran out (from qk_device_error)     */
    QK_ERR_WORKSPACE = 7,   /* workspace NULL, misaligned or smaller than required      */
    QK_ERR_TOO_LARGE = 8,   /* a size exceeds what the kernels support (see each call)  */
    QK_ERR_BAD_INDEX = 9    /* an index read from device memory was out of range        */
                            /* (from qk_device_error; see qmatvec_experts_*)             */
} qk_status;

#define QK_MAX_BATCH 8

/*
 * Q8_0 GEMV, batch 1..8: y[b*ldy + r] = sum_{c<K} W[row_offset + r][c] * x[b*K + c].
 *   w      device, raw Q8_0 block bytes of the whole tensor; 2-byte aligned.
 *   x      device fp32 [batch][K], row stride K; 4-byte aligned.
 *   y      device fp32 [batch][ldy]; writes y[b*ldy + r] for r < rows only;
 *          4-byte aligned.  ldy == 0 means ldy = rows.
 *   K      columns, any K >= 1.  A launch keeps its activation rows (about
 *          4.1 to 4.6 bytes a column each, K rounded up to the block size) in
 *          shared memory next to at least one staged tile of weight rows; a
 *          batch whose activations do not fit in the device's shared memory
 *          per block is computed by several launches of fewer batch rows
 *          (each batch row's result is the same as in a call of that size).
 *          A K for which one activation row does not fit (above about 48000
 *          on GB300) returns QK_ERR_TOO_LARGE before any launch.
 * Accuracy (every GEMV entry point; the tests check these bounds).  The
 * arithmetic is fp32 and a result differs from the exact dot product by at
 * most 1e-5 * S + 1e-6 + A, per element, where
 *   S = sum_c |x[b][c]| * (the magnitudes of the terms the weight is made
 *       of): |w| for Q8_0, |d*sc*q| + |dmin*m| for Q4_K and
 *       |d*scale*q| + 32*|d*scale| for Q6_K.  The kernels sum a Q4_K or Q6_K
 *       weight's two terms separately, so this is sum|w*x| unless the terms
 *       of the weights nearly cancel (then S is the larger);
 *   A is the term of the activation encoding, 0 where x is used as fp32:
 *     - Batch 1 holds each 32-column group of x as 24-bit integers that
 *       share one binary exponent: that of the group's largest magnitude
 *       or, when the largest is at least 2^3 times (in binary exponent)
 *       every other value of the group, that of the second largest, the
 *       largest value then being carried exactly on its own.  A value of
 *       x is thus held within 2^-20 times the second largest magnitude of
 *       its group (the largest within 2^-22 of itself), and
 *       A = 2^-20 * sum_groups (second largest |x| of the group) *
 *                   (sum |w| over the group's columns).
 *       A single outlier per group, at any magnitude, therefore costs
 *       nothing, and A is far inside 1e-5 * S unless a row's weights sit
 *       mostly on values much smaller than their group's second largest
 *       (for instance two values 2^20 times the rest in one group, meeting
 *       zero weights).
 *     - Batch 2..8 takes one of two forms.  Q8_0 with K a multiple of 128
 *       (K up to 4096) and Q4_K (K up to 4864) take the tensor-core form
 *       when the call has at least 128 rows per SM of the device (19456
 *       rows on 152 SMs) and, for Q4_K, batch 4..8; other calls take the
 *       fp32 form, for which A = 0.  The tensor-core form applies the same
 *       rule for a lone outlier (carried exactly), then holds each 32-column
 *       group of a batch row as two fp16 pieces of x scaled by the power of
 *       two that puts the group's largest remaining magnitude M in
 *       [2^14, 2^15) ([2^10, 2^11) for the high-nibble groups of Q4_K): a
 *       value is held within 2^-24 of itself or within 2^-39 (2^-35) * M,
 *       whichever is more (M taken as at least 2^-100), so
 *       A = 2^-35 * sum_groups M * (sum |w| over the group's columns).  Each form's arithmetic for a row depends on K
 *       only: row ranges of a tensor give the bits of the whole call when
 *       both take the same form.
 *   NaN and infinities in x give non-finite results.
 */
int qmatvec_q8_0(const void *w, int64_t row_offset, int64_t rows, int64_t K,
                 const float *x, int batch, float *y, int64_t ldy, qk_stream_t stream);

/*
 * Q4_K GEMV, batch 1..8.  Same contract as qmatvec_q8_0, with w 16-byte
 * aligned (144-byte super-blocks keep every row 16-byte aligned).
 */
int qmatvec_q4_k(const void *w, int64_t row_offset, int64_t rows, int64_t K,
                 const float *x, int batch, float *y, int64_t ldy, qk_stream_t stream);

/*
 * Q6_K GEMV, batch 1..8.  Same contract as qmatvec_q8_0 (w 2-byte aligned:
 * 210-byte super-blocks).  Q6_K is the format of lm_head / ffn_down in the
 * Q4_K_M files people download (their output weight is Q4_K or Q6_K:
 * nx_f32_llm_v4.nx source, lm_head binder comment; kernel `mv_q6_k`,
 * nurllama 0.18.1 API reference, kernels.nu).  Block reading (GGUF):
 * ql[128] | qh[64] | scales[16] int8 | fp16 d per 256 weights; weight i of
 * half n = i/128 (cc = i%128, t = cc/32, l = cc%32) takes its low 4 bits
 * from ql[64n + l + 32*(t%2)] (low nibble if t < 2, else high) and its high
 * 2 bits from (qh[32n + l] >> 2t) & 3;  w = d * scales[i/16] * (q - 32).
 */
int qmatvec_q6_k(const void *w, int64_t row_offset, int64_t rows, int64_t K,
                 const float *x, int batch, float *y, int64_t ldy, qk_stream_t stream);

/*
 * Fused gate/up GEMV with the SwiGLU product, batch 1..8:
 *   g = sum_{c<K} W[gate_offset + p][c] * x[b*K + c]
 *   u = sum_{c<K} W[up_offset + p][c]   * x[b*K + c]
 *   h[b*ldh + p] = silu(g) * u,   silu(z) = z / (1 + e^-z),   for p < F.
 * The SwiGLU of the llama FFN (nurllama README, "What it runs") as silumul
 * g <- silu(g) * u (nurllama 0.18.1 API reference, kernels.nu `lk_silumul`),
 * folded into the matvec as loom's decode matvecs fuse it (loom-port-llm
 * SKILL.md, "Kernel inventory").  Gate and up rows may be row
 * ranges of one fused tensor (phi3's ffn_up: gate_offset 0, up_offset F;
 * nurllama README, "What it runs"), or of two tensors passed as one
 * allocation with the offsets between them.
 *   w            device block bytes holding both row ranges; alignment as the
 *                plain GEMV of the format (Q8_0 2 bytes, Q4_K 16 bytes).
 *   gate_offset, up_offset  first gate / up row (>= 0), in rows of K columns.
 *   x            device fp32 [batch][K];  h  device fp32 [batch][ldh], ldh == 0
 *                means ldh = F; only h[b*ldh + p] for p < F is written.
 * g and u are computed exactly as the plain GEMV's rows (each within the
 * plain GEMV's accuracy bound, see qmatvec_q8_0); silu uses CUDA's expf and its
 * fast division (within 2 ulp; a denominator past 2^126 gives a zero of z's
 * sign, the limit).  Errors: as the plain
 * GEMV; a negative up_offset is QK_ERR_BAD_DIM.
 */
int qmatvec_swiglu_q8_0(const void *w, int64_t gate_offset, int64_t up_offset, int64_t F, int64_t K,
                        const float *x, int batch, float *h, int64_t ldh, qk_stream_t stream);
int qmatvec_swiglu_q4_k(const void *w, int64_t gate_offset, int64_t up_offset, int64_t F, int64_t K,
                        const float *x, int batch, float *h, int64_t ldh, qk_stream_t stream);
int qmatvec_swiglu_q6_k(const void *w, int64_t gate_offset, int64_t up_offset, int64_t F, int64_t K,
                        const float *x, int batch, float *h, int64_t ldh, qk_stream_t stream);

/*
 * Batched expert GEMV over n_assign expert assignments:
 *   y[a*ldy + r] = sum_{c<K} W[expert_ids[a]*rows + r][c] * x[(a / xk)*K + c]
 * for a < n_assign and r < rows: nurllama's batched expert matvec, one call
 * for every assignment, output row a taken from expert expid_dev[a] with
 * input row a/xk (nurllama 0.18.1 API reference, kernels.nu
 * `lk_matvec_experts`); the experts of a projection live in one 3-D tensor
 * [n_experts][rows][K] evaluated as row ranges (nurllama README, "What it
 * runs", llada2).
 *   w           device block bytes of the whole expert tensor (alignment as
 *               the plain GEMV of the format).
 *   x           device fp32 [ceil(n_assign / xk)][K]; xk >= 1 assignments per
 *               input row (e.g. the experts chosen per token).
 *   expert_ids  device int32 [n_assign], 4-byte aligned; it may be written by
 *               the kernel just before this call on the same stream (the
 *               kernel reads it after the previous kernel completes).
 *   y           device fp32 [n_assign][ldy], ldy == 0 means ldy = rows.
 * An id outside [0, n_experts) is not dereferenced: that assignment's rows
 * are set to NaN and qk_device_error() reports QK_ERR_BAD_INDEX.  Error
 * bound as the plain GEMV at batch 1 (see qmatvec_q8_0).
 */
int qmatvec_experts_q8_0(const void *w, int64_t n_experts, int64_t rows, int64_t K, const float *x, int xk,
                         const int32_t *expert_ids, int64_t n_assign, float *y, int64_t ldy, qk_stream_t stream);
int qmatvec_experts_q4_k(const void *w, int64_t n_experts, int64_t rows, int64_t K, const float *x, int xk,
                         const int32_t *expert_ids, int64_t n_assign, float *y, int64_t ldy, qk_stream_t stream);
int qmatvec_experts_q6_k(const void *w, int64_t n_experts, int64_t rows, int64_t K, const float *x, int xk,
                         const int32_t *expert_ids, int64_t n_assign, float *y, int64_t ldy, qk_stream_t stream);

/*
 * Q4_K prefill GEMM on the tensor cores:
 *   y[m*ldy + n] = sum_{c<K} bf16(W[row_offset + n][c]) * bf16(x[m*K + c])
 * for m < M tokens and n < N weight rows, accumulated in fp32.  Each weight
 * is decoded to fp32 (w = d*sc*q - dmin*m) and rounded to bf16, each
 * activation is rounded to bf16 (round to nearest even).  This is the
 * batched (prefill) form of the matvec: the chunked prefill multiplies a
 * whole chunk of positions at once, so a chunk reads each weight only once
 * (nurllama 0.18.1 API reference, model.nu).
 *   w          device Q4_K block bytes of the whole tensor; 16-byte aligned.
 *   x          device fp32 [M][K], row stride K; 4-byte aligned.
 *   y          device fp32 [M][ldy]; writes y[m*ldy + n] for n < N only.
 *              ldy == 0 means ldy = N.
 *   workspace  device scratch of at least qgemm_q4_k_workspace_bytes(M, N, K)
 *              bytes, 256-byte aligned, owned by the caller (it receives the
 *              bf16 copy of x; its contents on return are unspecified).
 * Error bound: |y - exact| <= 1e-2 * sum|w*x| + 1e-6 per element (two bf16
 * roundings); the tests also check it against the bf16-rounded product.
 */
int qgemm_q4_k(const void *w, int64_t row_offset, int64_t N, int64_t K, const float *x, int64_t M,
               float *y, int64_t ldy, void *workspace, size_t workspace_bytes, qk_stream_t stream);

/*
 * Accumulating form of qgemm_q4_k: y[m*ldy + n] += sum_k bf16(W[row_offset+n][k]) * bf16(x[m*K + k]),
 * the acc mode of loom's prefill GEMMs (they come in store, acc and swiglu
 * modes: loom-port-llm SKILL.md, "What the starter generates", gen_gemm.py): the
 * product lands on what y holds (e.g. the residual stream).  Same arguments,
 * errors and bound as qgemm_q4_k, plus one fp32 rounding of the final add.
 */
int qgemm_q4_k_acc(const void *w, int64_t row_offset, int64_t N, int64_t K, const float *x, int64_t M,
                   float *y, int64_t ldy, void *workspace, size_t workspace_bytes, qk_stream_t stream);

/*
 * SwiGLU form of the prefill GEMM (loom's "swiglu" mode, same source): for
 * m < M and p < F
 *   g = sum_k bf16(W[gate_offset + p][k]) * bf16(x[m*K + k])
 *   u = sum_k bf16(W[up_offset + p][k])   * bf16(x[m*K + k])
 *   h[m*ldh + p] = silu(g) * u,   silu(z) = z / (1 + e^-z)  (CUDA expf, fast division as above),
 * g and u accumulated in fp32 on the tensor cores exactly as qgemm_q4_k's
 * outputs.  Gate and up are row ranges of one Q4_K tensor (or of one
 * allocation holding both); gate_offset, up_offset >= 0.  Workspace and
 * errors as qgemm_q4_k (ldh == 0 means ldh = F).
 */
int qgemm_swiglu_q4_k(const void *w, int64_t gate_offset, int64_t up_offset, int64_t F, int64_t K, const float *x,
                      int64_t M, float *h, int64_t ldh, void *workspace, size_t workspace_bytes, qk_stream_t stream);

/*
 * Q8_0 forms of the prefill GEMM (loom's prefill GEMM formats include q8_0,
 * loom-port-llm SKILL.md, "What the starter generates", gen_gemm.py): the same
 * three modes with Q8_0 weights (w = d*q, rounded to bf16), w 2-byte aligned
 * (34-byte blocks); arguments, workspace, errors and bounds as the Q4_K forms.
 */
int qgemm_q8_0(const void *w, int64_t row_offset, int64_t N, int64_t K, const float *x, int64_t M,
               float *y, int64_t ldy, void *workspace, size_t workspace_bytes, qk_stream_t stream);
int qgemm_q8_0_acc(const void *w, int64_t row_offset, int64_t N, int64_t K, const float *x, int64_t M,
                   float *y, int64_t ldy, void *workspace, size_t workspace_bytes, qk_stream_t stream);
int qgemm_swiglu_q8_0(const void *w, int64_t gate_offset, int64_t up_offset, int64_t F, int64_t K, const float *x,
                      int64_t M, float *h, int64_t ldh, void *workspace, size_t workspace_bytes, qk_stream_t stream);

/* Workspace bytes the prefill GEMMs need for M tokens and K columns (N unused). */
size_t qgemm_q4_k_workspace_bytes(int64_t M, int64_t N, int64_t K);

/*
 * qgemm_q4_k for callers that cannot allocate device memory -- for example a
 * plugin inside an inference engine that owns every device allocation, or
 * code that must not allocate once running -- and so cannot pass the
 * workspace qgemm_q4_k needs.  The pages have no counterpart of this call;
 * it exists for such callers only.
 * Same operation, arguments and results as qgemm_q4_k, without the
 * workspace: the scratch is a fixed array of QK_NOALLOC_SCRATCH_BYTES inside
 * the library, held by every GPU that loads the library until the process
 * exits.  No call allocates or frees memory.
 *   Sizes: M * round_up(K, 8) * 2 + 256 must not exceed
 *   QK_NOALLOC_SCRATCH_BYTES, else QK_ERR_TOO_LARGE (before any launch).
 *   The first call on a device looks up the array's device address; make
 *   it before any stream capture.
 *   All calls share the array: calls that overlap on the GPU (for example on
 *   two streams at once) race on it and give undefined results.
 */
#define QK_NOALLOC_SCRATCH_BYTES (8u << 20)
int qgemm_q4_k_noalloc(const void *w, int64_t row_offset, int64_t N, int64_t K, const float *x, int64_t M,
                       float *y, int64_t ldy, qk_stream_t stream);

/*
 * Bytes of one row of a tensor with K columns: ceil(K/32)*34 (Q8_0),
 * ceil(K/256)*144 (Q4_K) or ceil(K/256)*210 (Q6_K).
 */
int64_t qk_row_bytes_q8_0(int64_t K);
int64_t qk_row_bytes_q4_k(int64_t K);
int64_t qk_row_bytes_q6_k(int64_t K);

/* Human-readable name of a status code (static string, never NULL). */
const char *qk_status_string(int status);

/*
 * Reads and clears the device error word of the current device after
 * synchronising `stream`: QK_OK, QK_ERR_TIMEOUT (a bounded wait ran out),
 * QK_ERR_BAD_INDEX (an expert id was out of range) or QK_ERR_CUDA (the
 * synchronisation itself failed).  Meant for tests and
 * debugging; the compute calls never synchronise.
 */
int qk_device_error(qk_stream_t stream);

/*
 * Upper bound, in nanoseconds, of every device-side wait of later launches
 * (default 2e9).  Returns the previous value.  Tests shorten it.
 */
uint64_t qk_set_wait_limit_ns(uint64_t ns);

/*
 * Programmatic dependent launch for later calls (default off; returns the
 * previous setting).  When on, a call may be scheduled while the kernel just
 * before it in the stream is still running: it starts streaming its weights
 * at once and waits for that kernel (griddepcontrol.wait) only before it
 * reads x and writes y.  So the weights of a call must not be written by
 * the kernel directly before it in the stream; x and y keep full stream
 * order.  Meant for decode loops whose weights are loaded once.
 */
int qk_set_programmatic_launch(int enable);

/*
 * Strict-blocks mode for later calls (returns the previous setting).  Off by
 * default, where any K >= 1 is accepted and a row's last block may be
 * partly used; on, every compute call whose K is not a multiple of its
 * format's block (32 columns for Q8_0, 256 for Q4_K and Q6_K) returns
 * QK_ERR_BAD_DIM before any launch.  The library starts with it on when the
 * environment holds QK_STRICT=1 at load time.  A GGUF row always holds whole
 * blocks (nurllama README, "What it runs"); the mode is for callers that want
 * such shapes rejected rather than read with an unused tail.
 */
int qk_set_strict_blocks(int enable);

/* Library version, major*10000 + minor*100 + patch. */
int qk_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QK_H */
