// qk_gemv_kernel.cuh -- the fused dequantise-and-multiply GEMV kernel for
// GGUF Q8_0 / Q4_K weights against fp32 activations, batch 1..8 (sm_103a).
//
// The operation is the quantised matvec of "nurllama 0.18.1 API reference",
// kernels.nu (`lk_matvec_q`, the batched `mv_*_b` forms): every block is
// decoded inside the dot product, y[b][r] = sum_c W[r][c] x[b][c].
//
// Design (one GPU, memory-bound):
//  * Persistent grid, one CTA per SM.  CTA i owns the contiguous row range
//    [rows*i/G, rows*(i+1)/G), i.e. one contiguous byte span of the tensor.
//  * Warp 0 is the producer: one lane streams tiles of whole rows into a ring
//    of shared-memory stages with 1-D bulk copies (cp.async.bulk, completion
//    on an mbarrier, L2 evict-first).  A tile's byte span is widened to
//    16-byte boundaries (Q8_0 rows are 34*nb bytes, not 16-byte multiples);
//    a 16-byte granule that holds a byte of the tensor never crosses a page,
//    so the widened copy stays inside mapped memory.
//  * The other warps are consumers.  A row is cut into units -- 128 weights
//    of Q4_K (half a super-block: four 32-weight sub-blocks) or one 32-weight
//    Q8_0 block -- and a team of SW = units-per-row threads covers one row
//    (the "one warp per output row, the lanes split each block" shape of the
//    nurllama README, "What it runs", generalised to teams of any width).
//    Each thread handles its unit for R rows at once, so each activation
//    value read from shared memory serves R rows.
//  * Activations live in shared memory as float4 groups: group g of unit u
//    of batch row b at float4 index (b*G + g)*XU + u, so threads holding
//    consecutive units read consecutive 16-byte words.  XU (the unit stride)
//    is a compile-time constant US where the kernel is specialised for it,
//    which turns every activation load into a fixed-offset shared load.
//  * Q4_K decoding: a 4-bit field at bit position s of a 32-bit word becomes
//    the exact float 2^23 + q*2^s with one LOP3 (mask | 0x4B000000), and
//    subtracting 2^23 leaves q*2^s exactly.  The activations in shared memory
//    are pre-multiplied by 2^-s for the position their column's nibble has,
//    so (q*2^s)*(x*2^-s) = q*x exactly.  Per 32-weight sub-block j the row
//    contributes d*sc_j * sum(q*x) - dmin*m_j * sum(x) (the identical
//    factorisation of w = d*sc*q - dmin*m); the sub-block sums of x are
//    computed once per CTA.  Int8 Q8_0 quants use the same trick on bytes
//    (bias 128) and contribute d * sum(q*x) per block.  Pairs of weights go
//    through packed f32x2 FADD/FFMA.
//  * Each thread's partial sums go to shared memory; after one named barrier
//    per tile the partials of a row are summed by a warp and written to y.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "qk_device.cuh"
#include "qk_internal.h"

namespace qk {

constexpr uint32_t kMagic = 0x4B000000u;   // 2^23 as an fp32 bit pattern
constexpr float kTwo23 = 8388608.0f;

struct GemvArgs {
    const uint8_t *w;   // first byte of row 0 of this call's row range
    const float *x;     // [B][K], row stride K
    float *y;           // [B][ldy]
    int64_t rows, K, ldy, row_bytes;
    int U;              // units per row
    int XU;             // unit stride of the shared-memory activation layout (>= U)
    int SW;             // threads per row team
    int slots;          // row teams per CTA
    int NTC;            // consumer threads (multiple of 32, >= slots * SW)
    int tile_rows;      // rows per stage = slots * R
    int stages;
    int stage_bytes;
    int off_x, off_xsum, off_xscale, off_red, off_stage;   // shared-memory byte offsets
    int64_t skip_tile;  // test hook: CTA 0 never copies this tile (-1: none)
    uint64_t wait_ns;
    int *err;
};

// Consumer threads per CTA, at most: 512 for batch 1, 256 otherwise (the
// register budget of a thread).
__host__ __device__ constexpr int max_consumers(int /*fmt*/, int batch)
{
    return batch <= 1 ? kMaxConsumers : kMaxConsumers / 2;
}

// Rows each thread handles at once.
__host__ __device__ constexpr int rows_per_thread(int fmt, int batch)
{
    return fmt == kFmtQ4K ? (batch <= 4 ? 2 : 1) : (batch <= 2 ? 4 : 2);
}

// -------------------------------------------------------------------------- Q4_K unit

// Bit position of the nibble that carries local column c (0..127) of a
// 128-weight unit inside its 32-bit qs word, after the (word >> 12) used for
// the upper nibbles.  Low nibbles (first 32 columns of a 64-column chunk) sit
// at 0, 8, 16 and 12; high nibbles at 4, 12, 8 and 16.
__device__ __forceinline__ int q4k_nibble_shift(int c)
{
    const int e = c & 3;
    const bool hi = (c & 32) != 0;
    const int lo_s = e == 0 ? 0 : (e == 1 ? 8 : (e == 2 ? 16 : 12));
    const int hi_s = e == 0 ? 4 : (e == 1 ? 12 : (e == 2 ? 8 : 16));
    return hi ? hi_s : lo_s;
}

// One 128-weight unit (half h of super-block blk) for R rows; adds each
// row's contribution to acc[r][b].  xa: shared address of float4 group 0 of
// unit u (batch row 0); gs: byte stride between groups (16*XU).
template <int B, int R, int US>
__device__ __forceinline__ void q4k_unit(const uint8_t *const (&rowp)[R], int u, uint32_t xa, uint32_t gs_rt,
                                         const float *__restrict__ xsum_u, int xsum_stride,
                                         float (&acc)[R][B])
{
    const uint32_t gs = US ? 16u * US : gs_rt;
    const int blk = u >> 1;
    const int h = u & 1;
    float ds[R][4], dm[R][4];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const uint4 hd = *reinterpret_cast<const uint4 *>(rowp[r] + blk * 144);
        const float d = half_bits_to_float(hd.x);
        const float dmin = half_bits_to_float(hd.x >> 16);
        // 6-bit scales and mins of the four sub-blocks 4h..4h+3, one per byte
        const uint32_t sc_lo = hd.y & 0x3F3F3F3Fu;
        const uint32_t m_lo = hd.z & 0x3F3F3F3Fu;
        const uint32_t sc_hi = (hd.w & 0x0F0F0F0Fu) | ((hd.y >> 2) & 0x30303030u);
        const uint32_t m_hi = ((hd.w >> 4) & 0x0F0F0F0Fu) | ((hd.z >> 2) & 0x30303030u);
        const uint32_t scw = h ? sc_hi : sc_lo;
        const uint32_t mw = h ? m_hi : m_lo;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float sc = __uint_as_float(__byte_perm(scw, kMagic, 0x7440u + j)) - kTwo23;
            const float m = __uint_as_float(__byte_perm(mw, kMagic, 0x7440u + j)) - kTwo23;
            ds[r][j] = d * sc;
            dm[r][j] = dmin * m;
        }
    }
    const uint64_t neg_magic = pack2f(-kTwo23, -kTwo23);
    const uint8_t *qoff[R];
#pragma unroll
    for (int r = 0; r < R; ++r) qoff[r] = rowp[r] + blk * 144 + 16 + 64 * h;
#pragma unroll
    for (int lc = 0; lc < 2; ++lc) {
        uint64_t A[R][B][2];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int b = 0; b < B; ++b) A[r][b][0] = A[r][b][1] = 0ull;
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            uint4 q[R];
#pragma unroll
            for (int r = 0; r < R; ++r) q[r] = *reinterpret_cast<const uint4 *>(qoff[r] + 32 * lc + 16 * p);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int g_lo = 16 * lc + 4 * p + k;
                const int g_hi = g_lo + 8;
                uint64_t qp[R][4];
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const uint32_t wd = k == 0 ? q[r].x : (k == 1 ? q[r].y : (k == 2 ? q[r].z : q[r].w));
                    const uint32_t wd2 = wd >> 12;
                    qp[r][0] = add_f32x2(pack2(magic_field<0xFu>(wd), magic_field<0xF00u>(wd)), neg_magic);
                    qp[r][1] = add_f32x2(pack2(magic_field<0xF0000u>(wd), magic_field<0xF000u>(wd2)), neg_magic);
                    qp[r][2] = add_f32x2(pack2(magic_field<0xF0u>(wd), magic_field<0xF000u>(wd)), neg_magic);
                    qp[r][3] = add_f32x2(pack2(magic_field<0xF00u>(wd2), magic_field<0xF0000u>(wd2)), neg_magic);
                }
#pragma unroll
                for (int b = 0; b < B; ++b) {
                    uint64_t xl0, xl1, xh0, xh1;
                    lds128(xa + static_cast<uint32_t>(b * 32 + g_lo) * gs, xl0, xl1);
                    lds128(xa + static_cast<uint32_t>(b * 32 + g_hi) * gs, xh0, xh1);
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        A[r][b][0] = fma_f32x2(qp[r][0], xl0, A[r][b][0]);
                        A[r][b][0] = fma_f32x2(qp[r][1], xl1, A[r][b][0]);
                        A[r][b][1] = fma_f32x2(qp[r][2], xh0, A[r][b][1]);
                        A[r][b][1] = fma_f32x2(qp[r][3], xh1, A[r][b][1]);
                    }
                }
            }
        }
        // scale this chunk's two sub-blocks (local 2lc = low nibbles, 2lc+1 = high)
        const int xstr = US ? US : xsum_stride;
#pragma unroll
        for (int b = 0; b < B; ++b) {
            const float X0 = xsum_u[(b * 4 + 2 * lc) * xstr];
            const float X1 = xsum_u[(b * 4 + 2 * lc + 1) * xstr];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const float2 a0 = unpack2f(A[r][b][0]);
                const float2 a1 = unpack2f(A[r][b][1]);
                float t = acc[r][b];
                t = fmaf(ds[r][2 * lc], a0.x + a0.y, t);
                t = fmaf(-dm[r][2 * lc], X0, t);
                t = fmaf(ds[r][2 * lc + 1], a1.x + a1.y, t);
                t = fmaf(-dm[r][2 * lc + 1], X1, t);
                acc[r][b] = t;
            }
        }
    }
}

// -------------------------------------------------------------------------- Q8_0 unit

// One 32-weight block (block u) for R rows.  Blocks are 34 bytes, so a
// block starts 0 or 2 bytes past a 4-byte boundary; nine aligned words are
// read and realigned with byte permutes.
template <int B, int R, int US>
__device__ __forceinline__ void q8_unit(const uint8_t *const (&rowp)[R], int u, uint32_t xa, uint32_t gs_rt,
                                        float (&acc)[R][B])
{
    const uint32_t gs = US ? 16u * US : gs_rt;
    uint32_t qw[R][8];
    float d[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const uintptr_t a = reinterpret_cast<uintptr_t>(rowp[r] + 34 * u);
        const uint32_t off = static_cast<uint32_t>(a & 3u);           // 0 or 2
        const uint32_t *wp = reinterpret_cast<const uint32_t *>(a - off);
        uint32_t wv[9];
#pragma unroll
        for (int i = 0; i < 9; ++i) wv[i] = wp[i];
        d[r] = half_bits_to_float(wv[0] >> (8 * off));
        const uint32_t sel = off ? 0x7654u : 0x5432u;
#pragma unroll
        for (int k = 0; k < 8; ++k) qw[r][k] = __byte_perm(wv[k], wv[k + 1], sel) ^ 0x80808080u;
    }
    const uint64_t neg_bias = pack2f(-(kTwo23 + 128.0f), -(kTwo23 + 128.0f));
    uint64_t part[R][B];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int b = 0; b < B; ++b) part[r][b] = 0ull;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        uint64_t q01[R], q23[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint32_t v = qw[r][k];
            q01[r] = add_f32x2(pack2(__byte_perm(v, kMagic, 0x7440u), __byte_perm(v, kMagic, 0x7441u)), neg_bias);
            q23[r] = add_f32x2(pack2(__byte_perm(v, kMagic, 0x7442u), __byte_perm(v, kMagic, 0x7443u)), neg_bias);
        }
#pragma unroll
        for (int b = 0; b < B; ++b) {
            uint64_t x01, x23;
            lds128(xa + static_cast<uint32_t>(b * 8 + k) * gs, x01, x23);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                part[r][b] = fma_f32x2(q01[r], x01, part[r][b]);
                part[r][b] = fma_f32x2(q23[r], x23, part[r][b]);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int b = 0; b < B; ++b) {
            const float2 p2 = unpack2f(part[r][b]);
            acc[r][b] = fmaf(d[r], p2.x + p2.y, acc[r][b]);
        }
}

// -------------------------------------------------------------------------- batch-1 integer units
//
// For batch 1 the activations are held as block floating point: each
// 32-column group has one exponent E and every value becomes the 32-bit
// integer m = rint(x * 2^(30-E)) (|m| < 2^31), stored as four byte planes
// (plane 3 signed, planes 0..2 unsigned).  A weight group then costs one
// 4-way byte dot product per plane, sum_i q_i m_i is assembled exactly in
// integers per plane and x-group scale 2^(E-30) turns it back into a float.
// Values within 2^7 of their group's largest magnitude are represented
// exactly; the error of any other value is below 2^-31 of that magnitude.

// sum(q*m) of one group from its four plane sums, as a float.
__device__ __forceinline__ float planes_to_float(int s0, int s1, int s2, int s3)
{
    const int hi = s3 * 256 + s2;     // exact in int32 for 32-weight groups
    const int lo = s1 * 256 + s0;
    return fmaf(static_cast<float>(hi), 65536.0f, static_cast<float>(lo));
}

// One 128-weight Q4_K unit for R rows, batch 1.
template <int R, int US>
__device__ __forceinline__ void q4k_unit_dig(const uint8_t *const (&rowp)[R], int u, uint32_t xa, uint32_t gs_rt,
                                             const float *__restrict__ xsum_u, const float *__restrict__ xscale_u,
                                             int xstride, float (&acc)[R][1])
{
    const uint32_t gs = US ? 16u * US : gs_rt;
    const int xstr = US ? US : xstride;
    const int blk = u >> 1;
    const int h = u & 1;
    float ds[R][4], dm[R][4];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const uint4 hd = *reinterpret_cast<const uint4 *>(rowp[r] + blk * 144);
        const float d = half_bits_to_float(hd.x);
        const float dmin = half_bits_to_float(hd.x >> 16);
        const uint32_t sc_lo = hd.y & 0x3F3F3F3Fu;
        const uint32_t m_lo = hd.z & 0x3F3F3F3Fu;
        const uint32_t sc_hi = (hd.w & 0x0F0F0F0Fu) | ((hd.y >> 2) & 0x30303030u);
        const uint32_t m_hi = ((hd.w >> 4) & 0x0F0F0F0Fu) | ((hd.z >> 2) & 0x30303030u);
        const uint32_t scw = h ? sc_hi : sc_lo;
        const uint32_t mw = h ? m_hi : m_lo;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float sc = __uint_as_float(__byte_perm(scw, kMagic, 0x7440u + j)) - kTwo23;
            const float m = __uint_as_float(__byte_perm(mw, kMagic, 0x7440u + j)) - kTwo23;
            ds[r][j] = d * sc;
            dm[r][j] = dmin * m;
        }
    }
    const uint8_t *qoff[R];
#pragma unroll
    for (int r = 0; r < R; ++r) qoff[r] = rowp[r] + blk * 144 + 16 + 64 * h;
#pragma unroll
    for (int lc = 0; lc < 2; ++lc) {
        int sl[R][4], sh[R][4];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int k = 0; k < 4; ++k) sl[r][k] = sh[r][k] = 0;
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            uint4 q[R];
#pragma unroll
            for (int r = 0; r < R; ++r) q[r] = *reinterpret_cast<const uint4 *>(qoff[r] + 32 * lc + 16 * p);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int g_lo = 16 * lc + 4 * p + k;
                const uint4 xl = lds128u(xa + static_cast<uint32_t>(g_lo) * gs);
                const uint4 xh = lds128u(xa + static_cast<uint32_t>(g_lo + 8) * gs);
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const uint32_t wd = k == 0 ? q[r].x : (k == 1 ? q[r].y : (k == 2 ? q[r].z : q[r].w));
                    const uint32_t L = wd & 0x0F0F0F0Fu;          // low nibbles: 4 columns of sub-block 2lc
                    const uint32_t H = (wd >> 4) & 0x0F0F0F0Fu;   // high nibbles: same columns of 2lc+1
                    sl[r][0] = dp4a_uu(L, xl.x, sl[r][0]);
                    sl[r][1] = dp4a_uu(L, xl.y, sl[r][1]);
                    sl[r][2] = dp4a_uu(L, xl.z, sl[r][2]);
                    sl[r][3] = dp4a_us(L, xl.w, sl[r][3]);
                    sh[r][0] = dp4a_uu(H, xh.x, sh[r][0]);
                    sh[r][1] = dp4a_uu(H, xh.y, sh[r][1]);
                    sh[r][2] = dp4a_uu(H, xh.z, sh[r][2]);
                    sh[r][3] = dp4a_us(H, xh.w, sh[r][3]);
                }
            }
        }
        const float X0 = xsum_u[(2 * lc) * xstr], X1 = xsum_u[(2 * lc + 1) * xstr];
        const float S0 = xscale_u[(2 * lc) * xstr], S1 = xscale_u[(2 * lc + 1) * xstr];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float F0 = planes_to_float(sl[r][0], sl[r][1], sl[r][2], sl[r][3]);
            const float F1 = planes_to_float(sh[r][0], sh[r][1], sh[r][2], sh[r][3]);
            float t = acc[r][0];
            t = fmaf(ds[r][2 * lc] * S0, F0, t);
            t = fmaf(-dm[r][2 * lc], X0, t);
            t = fmaf(ds[r][2 * lc + 1] * S1, F1, t);
            t = fmaf(-dm[r][2 * lc + 1], X1, t);
            acc[r][0] = t;
        }
    }
}

// One 32-weight Q8_0 block for R rows, batch 1.
template <int R, int US>
__device__ __forceinline__ void q8_unit_dig(const uint8_t *const (&rowp)[R], int u, uint32_t xa, uint32_t gs_rt,
                                            float xscale, float (&acc)[R][1])
{
    const uint32_t gs = US ? 16u * US : gs_rt;
    uint32_t qw[R][8];
    float d[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const uintptr_t a = reinterpret_cast<uintptr_t>(rowp[r] + 34 * u);
        const uint32_t off = static_cast<uint32_t>(a & 3u);           // 0 or 2
        const uint32_t *wp = reinterpret_cast<const uint32_t *>(a - off);
        uint32_t wv[9];
#pragma unroll
        for (int i = 0; i < 9; ++i) wv[i] = wp[i];
        d[r] = half_bits_to_float(wv[0] >> (8 * off));
        const uint32_t sel = off ? 0x7654u : 0x5432u;
#pragma unroll
        for (int k = 0; k < 8; ++k) qw[r][k] = __byte_perm(wv[k], wv[k + 1], sel);
    }
    int sp[R][4];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int k = 0; k < 4; ++k) sp[r][k] = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint4 xv = lds128u(xa + static_cast<uint32_t>(k) * gs);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint32_t v = qw[r][k];
            sp[r][0] = dp4a_su(v, xv.x, sp[r][0]);
            sp[r][1] = dp4a_su(v, xv.y, sp[r][1]);
            sp[r][2] = dp4a_su(v, xv.z, sp[r][2]);
            sp[r][3] = dp4a_ss(v, xv.w, sp[r][3]);
        }
    }
#pragma unroll
    for (int r = 0; r < R; ++r)
        acc[r][0] = fmaf(d[r] * xscale, planes_to_float(sp[r][0], sp[r][1], sp[r][2], sp[r][3]), acc[r][0]);
}

// -------------------------------------------------------------------------- kernel

template <int FMT, int B, int R, int US>
__global__ void __launch_bounds__(32 + max_consumers(FMT, B), 1) gemv_kernel(const GemvArgs a)
{
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int UC = FMT == kFmtQ4K ? 128 : 32;  // columns per unit
    constexpr int G = UC / 4;                      // float4 groups per unit
    const int tid = threadIdx.x;
    const int S = a.stages;
    const uint32_t bar0 = smem_u32(smem);
    const int n_cwarps = a.NTC / 32;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + 16 * kMaxStages);

    const int64_t nG = gridDim.x;
    const int64_t r_begin = (a.rows * blockIdx.x) / nG;
    const int64_t r_end = (a.rows * (blockIdx.x + 1)) / nG;
    const int64_t n_tiles = (r_end - r_begin + a.tile_rows - 1) / a.tile_rows;

    // Programmatic dependent launch: the next grid in the stream may be
    // scheduled now.  (No effect when launched without that attribute.)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(bar0 + 8u * s, 1);                    // full[s]
            mbar_init(bar0 + 8u * (S + s), n_cwarps);       // empty[s]
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    const uint32_t stage0 = smem_u32(smem + a.off_stage);

    // ------------------------------------------------------------------ producer
    if (tid < 32) {
        if (tid == 0) {
            const uint64_t pol = l2_evict_first_policy();
            int64_t j = 0;
            bool ok = true;
            for (; j < n_tiles; ++j) {
                const int s = static_cast<int>(j % S);
                const uint32_t use = static_cast<uint32_t>(j / S);
                if (j >= S && !mbar_wait(bar0 + 8u * (S + s), (use - 1) & 1u, a.wait_ns)) {
                    ok = false;
                    break;
                }
                if (j == a.skip_tile && blockIdx.x == 0) continue;   // test hook
                const int64_t row0 = r_begin + j * a.tile_rows;
                const int64_t n = min(static_cast<int64_t>(a.tile_rows), r_end - row0);
                const uintptr_t gs = reinterpret_cast<uintptr_t>(a.w + row0 * a.row_bytes);
                const uintptr_t ge = gs + static_cast<uintptr_t>(n * a.row_bytes);
                const uintptr_t lo = gs & ~static_cast<uintptr_t>(15);
                const uintptr_t hi = (ge + 15) & ~static_cast<uintptr_t>(15);
                const uint32_t bytes = static_cast<uint32_t>(hi - lo);
                mbar_arrive_expect_tx(bar0 + 8u * s, bytes);
                bulk_g2s(stage0 + static_cast<uint32_t>(s) * a.stage_bytes,
                         reinterpret_cast<const void *>(lo), bytes, bar0 + 8u * s, pol);
            }
            if (!ok) {
                record_error(a.err, kErrTimeout);
                // let the copies already issued land before the CTA exits
                for (int64_t t = j - S; t < j; ++t) {
                    if (t < 0 || (t == a.skip_tile && blockIdx.x == 0)) continue;
                    mbar_wait(bar0 + 8u * (t % S), static_cast<uint32_t>(t / S) & 1u, a.wait_ns);
                }
            }
        }
        return;
    }

    // ------------------------------------------------------------------ consumers
    const int ctid = tid - 32;
    const int lane = tid & 31;
    const int cwarp = ctid >> 5;
    const bool active = ctid < a.slots * a.SW;
    const int slot = active ? ctid / a.SW : 0;
    const int sl = active ? ctid - slot * a.SW : 0;
    const int U = a.U;
    const int XU = US ? US : a.XU;
    const uint32_t xs_addr = smem_u32(smem + a.off_x);
    float *xsum = reinterpret_cast<float *>(smem + a.off_xsum);
    float *xscale = reinterpret_cast<float *>(smem + a.off_xscale);

    // Activations -> shared memory, in one warp-uniform pass: each lane loads
    // float4 group f of batch row b (columns 4f..4f+3; columns >= K are zero)
    // and stores it at its permuted place.  For Q4_K the 8 lanes holding a
    // 32-column sub-block also sum it (unscaled) and the values are
    // pre-multiplied by 2^-s for their nibble position.  The weights do not
    // depend on earlier kernels, x may: with programmatic dependent launch
    // only this part waits for the previous grid (no effect otherwise).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    {
        const int K = static_cast<int>(a.K);
        const int g_total = U * G;                 // float4 groups per batch row incl. padding
        const bool vec = (K % 4 == 0) && ((reinterpret_cast<uintptr_t>(a.x) & 15u) == 0);
        constexpr int UNR = 4;
        for (int b = 0; b < B; ++b) {
            const float *xb = a.x + static_cast<int64_t>(b) * K;
            for (int base = cwarp * 32; base < g_total; base += UNR * a.NTC) {
                float4 v[UNR];
#pragma unroll
                for (int i = 0; i < UNR; ++i) {
                    const int f = base + i * a.NTC + lane;
                    const int c0 = 4 * f;
                    v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (f < g_total) {
                        if (vec && c0 + 3 < K) {
                            v[i] = __ldg(reinterpret_cast<const float4 *>(xb + c0));
                        } else {
                            if (c0 < K) v[i].x = __ldg(xb + c0);
                            if (c0 + 1 < K) v[i].y = __ldg(xb + c0 + 1);
                            if (c0 + 2 < K) v[i].z = __ldg(xb + c0 + 2);
                            if (c0 + 3 < K) v[i].w = __ldg(xb + c0 + 3);
                        }
                    }
                }
#pragma unroll
                for (int i = 0; i < UNR; ++i) {
                    const int f = base + i * a.NTC + lane;
                    if (base + i * a.NTC >= g_total) break;            // warp-uniform
                    const int u = f / G, g = f % G;
                    if constexpr (B == 1) {
                        // block floating point per 32-column group (8 lanes), as four byte planes
                        float amax = fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)), fmaxf(fabsf(v[i].z), fabsf(v[i].w)));
                        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
                        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
                        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 4));
                        float sum = (v[i].x + v[i].y) + (v[i].z + v[i].w);
                        if constexpr (FMT == kFmtQ4K) {
                            sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 1);
                            sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 2);
                            sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 4);
                        }
                        const int ebits = static_cast<int>((__float_as_uint(amax) >> 23) & 255u);
                        const bool finite = ebits != 255;
                        const int E = max(ebits - 127, -96);
                        const float up = __int_as_float((157 - E) << 23);     // 2^(30-E)
                        const float down = __int_as_float((97 + E) << 23);    // 2^(E-30)
                        uint32_t m0 = 0, m1 = 0, m2 = 0, m3 = 0;
                        if (finite) {
                            m0 = static_cast<uint32_t>(__float2int_rn(v[i].x * up));
                            m1 = static_cast<uint32_t>(__float2int_rn(v[i].y * up));
                            m2 = static_cast<uint32_t>(__float2int_rn(v[i].z * up));
                            m3 = static_cast<uint32_t>(__float2int_rn(v[i].w * up));
                        }
                        // byte-plane transpose: plane k holds byte k of the four columns
                        const uint32_t t0 = __byte_perm(m0, m1, 0x5140u), t1 = __byte_perm(m2, m3, 0x5140u);
                        const uint32_t t2 = __byte_perm(m0, m1, 0x7362u), t3 = __byte_perm(m2, m3, 0x7362u);
                        const uint32_t p0 = __byte_perm(t0, t1, 0x5410u), p1 = __byte_perm(t0, t1, 0x7632u);
                        const uint32_t p2 = __byte_perm(t2, t3, 0x5410u), p3 = __byte_perm(t2, t3, 0x7632u);
                        if (f < g_total) {
                            const int grp = FMT == kFmtQ4K ? (g >> 3) : 0;
                            if ((lane & 7) == 0) {
                                xscale[grp * XU + u] = finite ? down : __int_as_float(0x7FC00000);
                                if constexpr (FMT == kFmtQ4K) xsum[grp * XU + u] = sum;
                            }
                            const uint32_t dst = xs_addr + 16u * static_cast<uint32_t>(g * XU + u);
                            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                                         ::"r"(dst), "r"(p0), "r"(p1), "r"(p2), "r"(p3) : "memory");
                        }
                        continue;
                    }
                    if constexpr (FMT == kFmtQ4K) {
                        float sum = (v[i].x + v[i].y) + (v[i].z + v[i].w);
                        sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 1);
                        sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 2);
                        sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 4);
                        if (f < g_total && (lane & 7) == 0) xsum[(b * 4 + (g >> 3)) * XU + u] = sum;
                        const int c = 4 * g;
                        v[i].x *= __int_as_float((127 - q4k_nibble_shift(c)) << 23);
                        v[i].y *= __int_as_float((127 - q4k_nibble_shift(c + 1)) << 23);
                        v[i].z *= __int_as_float((127 - q4k_nibble_shift(c + 2)) << 23);
                        v[i].w *= __int_as_float((127 - q4k_nibble_shift(c + 3)) << 23);
                    }
                    if (f < g_total) {
                        const uint32_t dst = xs_addr + 16u * static_cast<uint32_t>((b * G + g) * XU + u);
                        asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};"
                                     ::"r"(dst), "f"(v[i].x), "f"(v[i].y), "f"(v[i].z), "f"(v[i].w) : "memory");
                    }
                }
            }
        }
    }
    named_bar_sync(1, a.NTC);

    float *red = reinterpret_cast<float *>(smem + a.off_red);
    const int n_out = a.slots * R * B;
    const int red_half = n_out * a.SW;
    const bool warp_team = a.SW <= 32 && (32 % a.SW) == 0;
    const uint32_t gs_rt = 16u * static_cast<uint32_t>(XU);
    for (int64_t j = 0; j < n_tiles; ++j) {
        const int s = static_cast<int>(j % S);
        const bool ok = mbar_wait(bar0 + 8u * s, static_cast<uint32_t>(j / S) & 1u, a.wait_ns);
        if (!ok) *abort_flag = 1;
        const int64_t row0 = r_begin + j * a.tile_rows;
        const int n = static_cast<int>(min(static_cast<int64_t>(a.tile_rows), r_end - row0));
        float acc[R][B];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int b = 0; b < B; ++b) acc[r][b] = 0.f;
        if (ok && active) {
            const uintptr_t gsrc = reinterpret_cast<uintptr_t>(a.w + row0 * a.row_bytes);
            const uint8_t *sbase = smem + a.off_stage + static_cast<int64_t>(s) * a.stage_bytes + (gsrc & 15u);
            const uint8_t *rowp[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int rt = min(r * a.slots + slot, n - 1);
                rowp[r] = sbase + static_cast<int64_t>(rt) * a.row_bytes;
            }
            for (int u = sl; u < U; u += a.SW) {
                const uint32_t xa = xs_addr + 16u * static_cast<uint32_t>(u);
                if constexpr (B == 1 && FMT == kFmtQ4K)
                    q4k_unit_dig<R, US>(rowp, u, xa, gs_rt, xsum + u, xscale + u, XU, acc);
                else if constexpr (B == 1)
                    q8_unit_dig<R, US>(rowp, u, xa, gs_rt, xscale[u], acc);
                else if constexpr (FMT == kFmtQ4K)
                    q4k_unit<B, R, US>(rowp, u, xa, gs_rt, xsum + u, XU, acc);
                else
                    q8_unit<B, R, US>(rowp, u, xa, gs_rt, acc);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar0 + 8u * (S + s));   // stage s may be refilled

        if (warp_team) {
            // teams of SW lanes (SW divides 32): butterfly inside the team,
            // no barrier; a warp whose wait ran out leaves on its own
            if (!ok) {
                if (lane == 0) record_error(a.err, kErrTimeout);
                break;
            }
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int b = 0; b < B; ++b) {
                    float v = acc[r][b];
                    for (int off = a.SW >> 1; off >= 1; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
                    const int rt = r * a.slots + slot;
                    if (active && sl == ((r * B + b) % a.SW) && rt < n) a.y[b * a.ldy + row0 + rt] = v;
                }
            continue;
        }

        // team reduction through shared memory: the partial of (slot, r, b)
        // from team member sl sits at red[((slot*R + r)*B + b)*SW + sl]
        float *rb = red + (j & 1) * red_half;
        if (active) {
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int b = 0; b < B; ++b) rb[((slot * R + r) * B + b) * a.SW + sl] = acc[r][b];
        }
        named_bar_sync(1, a.NTC);
        if (*abort_flag) {
            if (ctid == 0) record_error(a.err, kErrTimeout);
            break;
        }
        for (int o = cwarp; o < n_out; o += n_cwarps) {
            float v = 0.f;
            for (int t = lane; t < a.SW; t += 32) v += rb[o * a.SW + t];
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
            const int b = o % B;
            const int r = (o / B) % R;
            const int sidx = o / (B * R);
            const int rt = r * a.slots + sidx;
            if (lane == 0 && rt < n) a.y[b * a.ldy + row0 + rt] = v;
        }
    }
}

// Launch one instantiation (defined per format in qk_gemv_q4k.cu / qk_gemv_q80.cu).
cudaError_t gemv_launch_q4k(int batch, int us, const GemvArgs &a, int grid, int smem, cudaStream_t st, bool pdl);
cudaError_t gemv_launch_q80(int batch, int us, const GemvArgs &a, int grid, int smem, cudaStream_t st, bool pdl);

template <int FMT, int B, int R, int US>
cudaError_t gemv_launch_one(const GemvArgs &a, int grid, int smem, cudaStream_t st, bool pdl)
{
    auto kern = gemv_kernel<FMT, B, R, US>;
    // raise the dynamic shared-memory limit once per device and size
    static int granted[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (__atomic_load_n(&granted[dev], __ATOMIC_ACQUIRE) < smem) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        __atomic_store_n(&granted[dev], smem, __ATOMIC_RELEASE);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(32 + a.NTC);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, kern, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Instantiations for one format and batch: the activation unit stride is a
// compile-time 32 or 128 where it fits, else a runtime value.
#define QK_GEMV_DISPATCH_US(FMT, B, US_RT)                                                  \
    switch (US_RT) {                                                                        \
    case 32: return gemv_launch_one<FMT, B, rows_per_thread(FMT, B), 32>(a, grid, smem, st, pdl);   \
    case 128: return gemv_launch_one<FMT, B, rows_per_thread(FMT, B), 128>(a, grid, smem, st, pdl); \
    default: return gemv_launch_one<FMT, B, rows_per_thread(FMT, B), 0>(a, grid, smem, st, pdl);    \
    }

}  // namespace qk
