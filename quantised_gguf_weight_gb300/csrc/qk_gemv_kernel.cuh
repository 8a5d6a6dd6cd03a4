// qk_gemv_kernel.cuh -- the GEMV kernel (sm_103a):
// fused dequantise-and-multiply of GGUF Q8_0 / Q4_K / Q6_K rows against fp32
// activations, y[b][r] = sum_c W[r][c] x[b][c], batch 1..8.
//
// The operation is the quantised matvec of "nurllama 0.18.1 API reference",
// kernels.nu (`lk_matvec_q`, the batched `mv_*_b` forms).  Shape of the
// kernel:
//  * Persistent grid, one CTA per SM, CTA i owning the contiguous row range
//    [rows*i/G, rows*(i+1)/G).
//  * The rows of a CTA are cut into row groups of rows_w = (32/SW)*R rows and
//    each row into nkc K-chunks of SW*cpl lane units (a lane unit is one Q4_K
//    super-block of 256 weights, one 32-weight Q8_0 block, or half a Q6_K
//    super-block).  An item is one row group x one K-chunk.
//  * Consumer warp w owns row groups w, w+nw, ... and m shared-memory stages
//    of its own; its t-th item goes to stage w*m + t%m.  Lane w of warp 0 is
//    its producer: it streams the warp's items into its stages with 1-D bulk
//    copies (one per item when the row group is a single chunk -- its rows
//    are contiguous -- else one per row), completion on the stage's "full"
//    mbarrier.  Every stage is filled and drained in order by one producer
//    lane and one warp, so its phase parity is never ambiguous, and the
//    warps' pipelines do not wait on one another.
//  * For each item a lane copies its lane units of its team's R rows from
//    shared memory into registers, the warp hands the stage back at once
//    (its "empty" mbarrier) and the arithmetic runs from registers, so the
//    stages stay in flight.  Partial sums stay in registers across the chunks
//    of a row group and are summed over the SW lanes of a team with shuffles.
//  * Activations are staged once per CTA in shared memory, in the layout of
//    the unit functions: batch 1 as block floating point byte planes (three
//    byte dot products per weight group), batch >= 2 as fp32 (packed f32x2
//    arithmetic).  The layout is unit-major: unit slot us holds its 16-byte
//    slots (every batch row) contiguously plus one padding slot, so lanes
//    reading the same slot of consecutive units and lanes writing
//    consecutive slots of one unit both hit distinct bank groups.  Q4_K half
//    super-blocks are stored h-major (unit slot h*XH + super-block), so lanes
//    holding consecutive super-blocks read consecutive unit slots.
//  * Batch 1 has two forms with the same arithmetic in the same order: 11
//    consumer warps, or 15 at 128 registers a thread (WIDE; Q4_K lanes then
//    hold half a super-block in registers at a time) for calls with more
//    items a CTA than 11 warps, and for every Q6_K call.
//  * Pair mode (SwiGLU): an item holds gate rows and their up rows, and the
//    team sums become silu(g)*u.  Experts mode: each CTA takes part of one
//    assignment's rows, reading the expert id from device memory first.
// Every wait is bounded; a wait that runs out records QK_ERR_TIMEOUT in the
// device error word and the kernel leaves without touching the rest of y.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "qk_device.cuh"
#include "qk_internal.h"

namespace qk {


// Bit position of the nibble that carries local column c (0..127) of a
// 128-weight half super-block inside its 32-bit qs word, after the
// (word >> 12) used for the upper nibbles.  Low nibbles (first 32 columns of
// a 64-column chunk) sit at 0, 8, 16 and 12; high nibbles at 4, 12, 8 and 16.
__device__ __forceinline__ int q4k_nibble_shift(int c)
{
    const int e = c & 3;
    const bool hi = (c & 32) != 0;
    const int lo_s = e == 0 ? 0 : (e == 1 ? 8 : (e == 2 ? 16 : 12));
    const int hi_s = e == 0 ? 4 : (e == 1 ? 12 : (e == 2 ? 8 : 16));
    return hi ? hi_s : lo_s;
}

// Batch 1 holds the activations as block floating point: each 32-column
// group has one exponent E (its largest magnitude lies in [2^E, 2^(E+1)))
// and every value becomes the integer m = rint(x * 2^(21-E)), |m| <= 2^22,
// stored as three byte planes (planes 0 and 1 unsigned, plane 2 signed; a
// fourth byte of each 16-byte slot is unused).  A weight group then costs one
// 4-way byte dot product per plane, sum_i q_i m_i is assembled in integers
// per plane and the group scale 2^(E-21) turns it back into a float.  The
// error of a value is at most 2^(E-22), i.e. 2^-22 of its group's largest
// magnitude; small integers and other values with few significant bits are
// represented exactly.


// sum(q*m) of one group from its three plane sums, as a float.
__device__ __forceinline__ float planes_to_float(int s0, int s1, int s2)
{
    const int lo = s1 * 256 + s0;     // exact in int32 for 32-weight groups
    return fmaf(static_cast<float>(s2), 65536.0f, static_cast<float>(lo));
}

constexpr int kGemvMaxStages = 32;
constexpr int kGemvBarBytes = 768;   // full[32] at 0, empty[32] at 256, abort flag at 512, issued_use[32] at 528,
                                     // "first activation loads issued" at 656

struct GemvArgs {
    const uint8_t *w;   // first byte of row 0 of this call's row range
    const float *x;     // [B][K], row stride K
    float *y;           // [B][ldy]
    int64_t rows, K, ldy, row_bytes;
    int U;              // activation units per row (Q4_K: 128-column halves, Q8_0: blocks)
    int LU;             // lane units per row (Q4_K: super-blocks, Q8_0: blocks)
    int XU;             // unit slots of the shared-memory activation layout (Q4_K: 2 halves of XU/2)
    int SW;             // lanes per row team (power of two, <= 32)
    int lsw;            // log2(SW)
    int cpl;            // lane units per lane per item
    int nkc;            // K chunks per row group (chunk = SW * cpl lane units)
    int rows_w;         // rows per item = (32/SW) * R
    int chunk_bytes;    // bytes of one row's full chunk (nkc > 1)
    int row_stride;     // bytes between rows of a stage (nkc > 1)
    int nw;             // consumer warps that get row groups (<= the launched ones)
    int m;              // stages per consumer warp (stage w*m + t%m holds warp w's item t)
    int kw;             // consumer warps per row group: its K chunks c with c % kw == the warp's
                        // share (kw > 1: every warp has one row group at most)
    int off_part;       // kw > 1: per-lane chunk sums [group][chunk][lane][R][B] (fp32)
    int stage_bytes;
    int off_x, off_xsum, off_xscale, off_xout, off_stage;
    int pair;           // 1: output row p = silu(row p) * row (p + up_rows), both rows in one item
    int64_t up_rows;    // pair mode: distance in rows from a gate row to its up row
    int up_stage_off;   // pair mode, whole rows: stage offset of the up rows' span
    const int32_t *expid;  // experts mode (cpa > 0): expert of each assignment, device memory
    int64_t n_experts;  // experts mode: experts in the tensor (rows of each: `rows`)
    int xk;             // experts mode: assignments per input row of x
    int cpa;            // experts mode: CTAs per assignment (0: plain mode)
    int64_t skip_item;  // test hook: in CTA 0 warp 0's item with this number is never copied (-1: none)
    uint64_t wait_ns;
    int *err;
};

// Consumer warps per CTA and rows per thread of the ring kernel.
// (B = 1: 12 warps in all, three per scheduler, which leaves 168 registers a
// thread; the wide Q4_K batch-1 form: 16 warps, four per scheduler, 128
// registers, a lane holding half a super-block at a time; B >= 2: 9 warps.)
__host__ __device__ constexpr int gemv_warps(int /*fmt*/, int batch, bool wide = false)
{
    return batch == 1 ? (wide ? 15 : 11) : 8;
}
__host__ __device__ constexpr int gemv_rows(int fmt, int batch)
{
    return fmt != kFmtQ80 ? (batch <= 4 ? 2 : 1) : (batch == 1 ? 2 : (batch == 2 ? 4 : 2));
}
// Lane units a lane takes per item (Q4_K: one super-block of R rows; Q6_K:
// one half super-block; Q8_0: up to 4 blocks, held in registers one at a time).
__host__ __device__ constexpr int gemv_cpl_max(int fmt, int batch)
{
    return fmt != kFmtQ80 ? 1 : 4;
}

// -------------------------------------------------------------------------- Q4_K, batch 1
//
// Byte i (0..31) of the 32 bytes held in a (bytes 0..15) and b (16..31),
// selected without indexing registers.
__device__ __forceinline__ uint32_t byte_of32(const uint4 &a, const uint4 &b, int i)
{
    const int wi = i >> 2;
    uint32_t w = a.x;
    w = wi == 1 ? a.y : w;
    w = wi == 2 ? a.z : w;
    w = wi == 3 ? a.w : w;
    w = wi == 4 ? b.x : w;
    w = wi == 5 ? b.y : w;
    w = wi == 6 ? b.z : w;
    w = wi == 7 ? b.w : w;
    return (w >> (8 * (i & 3))) & 0xFFu;
}

// d*sc and -dmin*m of sub-block 4H + j from a super-block's first 16 bytes
// hd: the 6-bit field placed in a float's mantissa is 2^23 + v, and one FMA
// against the matching offset gives the exact product.  For odd j the scale
// is d/16*sc, since those weights are used as 16 q (the high nibbles in place).
template <int H>
__device__ __forceinline__ void q4k_scales(const uint4 &hd, float d, float dmin, float (&ds)[4], float (&dmn)[4])
{
    uint32_t scw, mw;
    if (H == 0) {
        scw = hd.y & 0x3F3F3F3Fu;
        mw = hd.z & 0x3F3F3F3Fu;
    } else {
        scw = (hd.w & 0x0F0F0F0Fu) | ((hd.y >> 2) & 0x30303030u);
        mw = ((hd.w >> 4) & 0x0F0F0F0Fu) | ((hd.z >> 2) & 0x30303030u);
    }
    const float dlo = d, dhi = d * 0.0625f;
    const float clo = dlo * -kTwo23, chi = dhi * -kTwo23, cm = dmin * kTwo23;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float fs = __uint_as_float(__byte_perm(scw, kMagic, 0x7440u + j));
        const float fm = __uint_as_float(__byte_perm(mw, kMagic, 0x7440u + j));
        ds[j] = (j & 1) ? fmaf(dhi, fs, chi) : fmaf(dlo, fs, clo);
        dmn[j] = fmaf(-dmin, fm, cm);
    }
}

// One 128-column half H of a super-block of R rows from registers:
// hd = bytes 0..15 (d, dmin, scales[12]); qs[r][Q0 + 2lc + p] holds bytes
// 16p..16p+15 of the half's 32-byte quant chunk lc (its low nibbles are
// sub-block 4H + 2lc, its high nibbles sub-block 4H + 2lc + 1).  x:
// block-floating-point byte planes of the half, float4 group g at xa + 16g;
// per 32-column group j the plain sum is xsum_h[j] and the plane scale
// 2^(E-21) is |xsc_h[j]| (a negative scale marks a group whose outlier is in
// neither the planes nor the plain sum; the caller adds its term).  The
// high nibbles are used in place (byte & 0xF0 = 16 q), which is folded into
// their sub-block scale as d/16 (exact: a power of two).
template <int R, int H, int N, int Q0>
__device__ __forceinline__ void q4k_half(const float (&d)[R], const float (&dmin)[R], const uint4 (&hd)[R],
                                         const uint4 (&qs)[R][N], const uint8_t *xa, const float *xsum_h,
                                         const float *xsc_h, float (&acc)[R][1])
{
    const float4 xsum4 = *reinterpret_cast<const float4 *>(xsum_h);
    const float4 xsc4 = *reinterpret_cast<const float4 *>(xsc_h);
    float ds[R][4], dmn[R][4];
#pragma unroll
    for (int r = 0; r < R; ++r) q4k_scales<H>(hd[r], d[r], dmin[r], ds[r], dmn[r]);
#pragma unroll
    for (int lc = 0; lc < 2; ++lc) {
        int sl[R][3], sh[R][3];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int k = 0; k < 3; ++k) sl[r][k] = sh[r][k] = 0;
#pragma unroll
        for (int p = 0; p < 2; ++p) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int g_lo = 16 * lc + 4 * p + k;
                const uint4 xl = *reinterpret_cast<const uint4 *>(xa + 16 * g_lo);
                const uint4 xh = *reinterpret_cast<const uint4 *>(xa + 16 * (g_lo + 8));
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const uint4 q = qs[r][Q0 + 2 * lc + p];
                    const uint32_t wd = k == 0 ? q.x : (k == 1 ? q.y : (k == 2 ? q.z : q.w));
                    const uint32_t L = wd & 0x0F0F0F0Fu;   // q of sub-block 2lc
                    const uint32_t Hn = wd & 0xF0F0F0F0u;  // 16 q of sub-block 2lc+1
                    sl[r][0] = dp4a_uu(L, xl.x, sl[r][0]);
                    sl[r][1] = dp4a_uu(L, xl.y, sl[r][1]);
                    sl[r][2] = dp4a_us(L, xl.z, sl[r][2]);
                    sh[r][0] = dp4a_uu(Hn, xh.x, sh[r][0]);
                    sh[r][1] = dp4a_uu(Hn, xh.y, sh[r][1]);
                    sh[r][2] = dp4a_us(Hn, xh.z, sh[r][2]);
                }
            }
        }
        const float X0 = lc ? xsum4.z : xsum4.x, X1 = lc ? xsum4.w : xsum4.y;
        const float S0 = fabsf(lc ? xsc4.z : xsc4.x), S1 = fabsf(lc ? xsc4.w : xsc4.y);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float F0 = planes_to_float(sl[r][0], sl[r][1], sl[r][2]);
            const float F1 = planes_to_float(sh[r][0], sh[r][1], sh[r][2]);
            float t = acc[r][0];
            t = fmaf(ds[r][2 * lc] * S0, F0, t);
            t = fmaf(dmn[r][2 * lc], X0, t);
            t = fmaf(ds[r][2 * lc + 1] * S1, F1, t);
            t = fmaf(dmn[r][2 * lc + 1], X1, t);
            acc[r][0] = t;
        }
    }
}

// A whole super-block of R rows (qs = its 128 quant bytes): half 0, then
// half 1 when the row has columns there.
template <int R>
__device__ __forceinline__ void q4k_sb_dig(const uint4 (&hd)[R], const uint4 (&qs)[R][8], bool has_hi,
                                           const uint8_t *xa0, const uint8_t *xa1, const float *xsum0,
                                           const float *xsum1, const float *xsc0, const float *xsc1,
                                           float (&acc)[R][1])
{
    float d[R], dmin[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        d[r] = half_bits_to_float(hd[r].x);
        dmin[r] = half_bits_to_float(hd[r].x >> 16);
    }
    q4k_half<R, 0, 8, 0>(d, dmin, hd, qs, xa0, xsum0, xsc0, acc);
    if (has_hi) q4k_half<R, 1, 8, 4>(d, dmin, hd, qs, xa1, xsum1, xsc1, acc);
}

// One half HH of the super-block, its 64 quant bytes in qs (the wide
// batch-1 form); the same arithmetic in the same order as q4k_sb_dig.
template <int R, int HH>
__device__ __forceinline__ void q4k_half_dig(const uint4 (&hd)[R], const uint4 (&qs)[R][4], const uint8_t *xa,
                                             const float *xsum_h, const float *xsc_h, float (&acc)[R][1])
{
    float d[R], dmin[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        d[r] = half_bits_to_float(hd[r].x);
        dmin[r] = half_bits_to_float(hd[r].x >> 16);
    }
    q4k_half<R, HH, 4, 0>(d, dmin, hd, qs, xa, xsum_h, xsc_h, acc);
}

// -------------------------------------------------------------------------- Q4_K, batch >= 2
//
// One super-block of R rows from registers against fp32 activations that are
// pre-multiplied by 2^-s for their nibble position (see q4k_nibble_shift):
// a nibble at bit s of a word becomes the exact float 2^23 + q*2^s with one
// LOP3, 2^23 is subtracted, and (q*2^s)*(x*2^-s) = q*x exactly.  Float4
// group g of batch row b of half h is at xa_h + 16*(32b + g); the sum of
// 32-column group j of batch row b at xsum_h[(4b + j)*xstr].
template <int B, int R>
__device__ __forceinline__ void q4k_sb_fp(const uint4 (&hd)[R], const uint4 (&qs)[R][8], bool has_hi,
                                            const uint8_t *xa0, const uint8_t *xa1, const float *xsum0,
                                            const float *xsum1, int xstr, float (&acc)[R][B])
{
    const uint64_t neg_magic = pack2f(-kTwo23, -kTwo23);
    float d[R], dmin[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        d[r] = half_bits_to_float(hd[r].x);
        dmin[r] = half_bits_to_float(hd[r].x >> 16);
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        if (h == 1 && !has_hi) break;
        const uint8_t *xa = h ? xa1 : xa0;
        const float *xsum_u = h ? xsum1 : xsum0;
        float ds[R][4], dmn[R][4];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            uint32_t scw, mw;
            if (h == 0) {
                scw = hd[r].y & 0x3F3F3F3Fu;
                mw = hd[r].z & 0x3F3F3F3Fu;
            } else {
                scw = (hd[r].w & 0x0F0F0F0Fu) | ((hd[r].y >> 2) & 0x30303030u);
                mw = ((hd[r].w >> 4) & 0x0F0F0F0Fu) | ((hd[r].z >> 2) & 0x30303030u);
            }
            const float cs = d[r] * -kTwo23, cm = dmin[r] * kTwo23;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                ds[r][j] = fmaf(d[r], __uint_as_float(__byte_perm(scw, kMagic, 0x7440u + j)), cs);
                dmn[r][j] = fmaf(-dmin[r], __uint_as_float(__byte_perm(mw, kMagic, 0x7440u + j)), cm);
            }
        }
#pragma unroll
        for (int lc = 0; lc < 2; ++lc) {
            uint64_t A[R][B][2];
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int b = 0; b < B; ++b) A[r][b][0] = A[r][b][1] = 0ull;
#pragma unroll
            for (int p = 0; p < 2; ++p) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int g_lo = 16 * lc + 4 * p + k;
                    const int g_hi = g_lo + 8;
                    uint64_t qp[R][4];
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const uint4 q = qs[r][4 * h + 2 * lc + p];
                        const uint32_t wd = k == 0 ? q.x : (k == 1 ? q.y : (k == 2 ? q.z : q.w));
                        const uint32_t wd2 = wd >> 12;
                        qp[r][0] = add_f32x2(pack2(magic_field<0xFu>(wd), magic_field<0xF00u>(wd)), neg_magic);
                        qp[r][1] = add_f32x2(pack2(magic_field<0xF0000u>(wd), magic_field<0xF000u>(wd2)), neg_magic);
                        qp[r][2] = add_f32x2(pack2(magic_field<0xF0u>(wd), magic_field<0xF000u>(wd)), neg_magic);
                        qp[r][3] = add_f32x2(pack2(magic_field<0xF00u>(wd2), magic_field<0xF0000u>(wd2)), neg_magic);
                    }
#pragma unroll
                    for (int b = 0; b < B; ++b) {
                        const ulonglong2 xl = *reinterpret_cast<const ulonglong2 *>(xa + 16 * (b * 32 + g_lo));
                        const ulonglong2 xh = *reinterpret_cast<const ulonglong2 *>(xa + 16 * (b * 32 + g_hi));
                        const uint64_t xl0 = xl.x, xl1 = xl.y, xh0 = xh.x, xh1 = xh.y;
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
#pragma unroll
            for (int b = 0; b < B; ++b) {
                const float X0 = xsum_u[(4 * b + 2 * lc) * xstr];
                const float X1 = xsum_u[(4 * b + 2 * lc + 1) * xstr];
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const float2 a0 = unpack2f(A[r][b][0]);
                    const float2 a1 = unpack2f(A[r][b][1]);
                    float t = acc[r][b];
                    t = fmaf(ds[r][2 * lc], a0.x + a0.y, t);
                    t = fmaf(dmn[r][2 * lc], X0, t);
                    t = fmaf(ds[r][2 * lc + 1], a1.x + a1.y, t);
                    t = fmaf(dmn[r][2 * lc + 1], X1, t);
                    acc[r][b] = t;
                }
            }
        }
    }
}

// -------------------------------------------------------------------------- Q8_0
//
// A 34-byte block starts 0 or 2 bytes past a 4-byte boundary; the lane keeps
// the nine aligned words that cover it and realigns them with byte permutes.
template <int R>
__device__ __forceinline__ void q8_realign(const uint32_t (&wv)[R][9], const uint32_t (&off)[R], float (&d)[R],
                                           uint32_t (&qw)[R][8])
{
#pragma unroll
    for (int r = 0; r < R; ++r) {
        d[r] = half_bits_to_float(wv[r][0] >> (8 * off[r]));
        const uint32_t sel = off[r] ? 0x7654u : 0x5432u;
#pragma unroll
        for (int k = 0; k < 8; ++k) qw[r][k] = __byte_perm(wv[r][k], wv[r][k + 1], sel);
    }
}

// Batch 1: block-floating-point planes of the block's 32 columns, float4
// group k at xa + 16k, plane scale |xscale| (a negative scale marks an
// outlier that is not in the planes; the caller adds its term).
template <int R>
__device__ __forceinline__ void q8_blk_dig(const uint32_t (&wv)[R][9], const uint32_t (&off)[R], const uint8_t *xa,
                                            float xscale, float (&acc)[R][1])
{
    float d[R];
    uint32_t qw[R][8];
    q8_realign<R>(wv, off, d, qw);
    int sp[R][3];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int k = 0; k < 3; ++k) sp[r][k] = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint4 xv = *reinterpret_cast<const uint4 *>(xa + 16 * k);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint32_t v = qw[r][k];
            sp[r][0] = dp4a_su(v, xv.x, sp[r][0]);
            sp[r][1] = dp4a_su(v, xv.y, sp[r][1]);
            sp[r][2] = dp4a_ss(v, xv.z, sp[r][2]);
        }
    }
    const float S = fabsf(xscale);
#pragma unroll
    for (int r = 0; r < R; ++r)
        acc[r][0] = fmaf(d[r] * S, planes_to_float(sp[r][0], sp[r][1], sp[r][2]), acc[r][0]);
}

// Batch >= 2: int8 quants through the magic-exponent trick (bias 128), fp32 x
// (float4 group k of batch row b at xa + 16*(8b + k)).
template <int B, int R>
__device__ __forceinline__ void q8_blk_fp(const uint32_t (&wv)[R][9], const uint32_t (&off)[R], const uint8_t *xa,
                                           float (&acc)[R][B])
{
    float d[R];
    uint32_t qw[R][8];
    q8_realign<R>(wv, off, d, qw);
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
            const uint32_t v = qw[r][k] ^ 0x80808080u;
            q01[r] = add_f32x2(pack2(__byte_perm(v, kMagic, 0x7440u), __byte_perm(v, kMagic, 0x7441u)), neg_bias);
            q23[r] = add_f32x2(pack2(__byte_perm(v, kMagic, 0x7442u), __byte_perm(v, kMagic, 0x7443u)), neg_bias);
        }
#pragma unroll
        for (int b = 0; b < B; ++b) {
            const ulonglong2 xv = *reinterpret_cast<const ulonglong2 *>(xa + 16 * (b * 8 + k));
            const uint64_t x01 = xv.x, x23 = xv.y;
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

// -------------------------------------------------------------------------- Q6_K
//
// A Q6_K super-block (210 bytes, 256 weights): ql[128] | qh[64] |
// scales[16] int8 | fp16 d; weight i of half n = i/128 (cc = i%128,
// t = cc/32, l = cc%32) takes 4 low bits from ql[64n + l + 32*(t%2)] (low
// nibble for t < 2, high for t >= 2) and 2 high bits (qh[32n + l] >> 2t) & 3;
// w = d * scales[i/16] * (q - 32).  The lane unit is half a super-block (128
// weights).  Blocks start 0 or 2 bytes past a 4-byte boundary, so a lane
// loads the aligned words around each field and realigns them with byte
// permutes.

// N words of a field starting at the 2-byte-aligned shared address p, read as
// N+1 aligned words (up to 4 bytes past the field, inside the stage slack).
template <int N>
__device__ __forceinline__ void lds_realign(const uint8_t *p, uint32_t (&out)[N])
{
    // (the aligned word address is formed in the shared window, so that the
    // loads are shared-memory loads, not generic ones)
    const uint32_t sa = static_cast<uint32_t>(__cvta_generic_to_shared(p));
    const uint32_t o = sa & 3u;
    const uint32_t *wp = static_cast<const uint32_t *>(__cvta_shared_to_generic(sa - o));
    const uint32_t sel = o ? 0x5432u : 0x3210u;
    uint32_t prev = wp[0];
#pragma unroll
    for (int i = 0; i < N; ++i) {
        const uint32_t nx = wp[i + 1];
        out[i] = __byte_perm(prev, nx, sel);
        prev = nx;
    }
}

// One half super-block in registers: its ql (64 bytes), qh (32 bytes), the 8
// scales (int8) and the word holding d in its low 16 bits.
struct Q6Half {
    uint32_t ql[16], qh[8], sc[2], dw;
};

__device__ __forceinline__ void q6_load(const uint8_t *blk, int n, Q6Half &h)
{
    lds_realign<16>(blk + 64 * n, h.ql);
    lds_realign<8>(blk + 128 + 32 * n, h.qh);
    lds_realign<2>(blk + 192 + 8 * n, h.sc);
    uint32_t dw[1];
    lds_realign<1>(blk + 208, dw);
    h.dw = dw[0];
}

// The 6-bit quants of columns 32t + 4k .. 32t + 4k + 3, one per byte.
__device__ __forceinline__ uint32_t q6_quad(const Q6Half &h, int t, int k)
{
    const uint32_t a = h.ql[k + 8 * (t & 1)];
    const uint32_t b = h.qh[k];
    const uint32_t lo = (t < 2 ? a : (a >> 4)) & 0x0F0F0F0Fu;
    const uint32_t hi = (t == 0 ? (b << 4) : t == 1 ? (b << 2) : t == 2 ? b : (b >> 2)) & 0x30303030u;
    return lo | hi;
}

// d * scales[j] (j < 8 of this half); exact (11 x 8 significant bits).
__device__ __forceinline__ float q6_dscale(const Q6Half &h, float d, int j)
{
    const int s = static_cast<int8_t>((h.sc[j >> 2] >> (8 * (j & 3))) & 0xFFu);
    return d * static_cast<float>(s);
}

// Batch 1: block-floating-point planes of the half's 128 columns (float4
// group g at xa + 16g); per 16-column sub-block j the plain sum x16[j] (for
// the -32 offset) and per 32-column group the plane scale xsc[j/2].
// |xsc[j]| is the plane scale of 32-column group j; a negative xsc[j] marks
// an outlier of the group, in neither the planes nor the 16-column sums (the
// caller adds its term with q6k_outlier_term).
template <int R>
__device__ __forceinline__ void q6k_half_dig(const Q6Half (&hr)[R], const uint8_t *xa, const float *x16,
                                             const float *xsc, float (&acc)[R][1])
{
    float d[R];
#pragma unroll
    for (int r = 0; r < R; ++r) d[r] = half_bits_to_float(hr[r].dw);
    const float4 x16a = *reinterpret_cast<const float4 *>(x16);
    const float4 x16b = *reinterpret_cast<const float4 *>(x16 + 4);
    const float4 xsc4 = *reinterpret_cast<const float4 *>(xsc);
    const float x16v[8] = {x16a.x, x16a.y, x16a.z, x16a.w, x16b.x, x16b.y, x16b.z, x16b.w};
    const float xscv[4] = {xsc4.x, xsc4.y, xsc4.z, xsc4.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        int sp[R][2][3];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int k = 0; k < 3; ++k) sp[r][h][k] = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint4 xv = *reinterpret_cast<const uint4 *>(xa + 16 * (8 * t + k));
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const uint32_t q = q6_quad(hr[r], t, k);
                const int h = k >> 2;                   // 16-column sub-block 2t + h
                sp[r][h][0] = dp4a_uu(q, xv.x, sp[r][h][0]);
                sp[r][h][1] = dp4a_uu(q, xv.y, sp[r][h][1]);
                sp[r][h][2] = dp4a_us(q, xv.z, sp[r][h][2]);
            }
        }
        const float S = fabsf(xscv[t]);
        const float X0 = x16v[2 * t], X1 = x16v[2 * t + 1];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float ds0 = q6_dscale(hr[r], d[r], 2 * t), ds1 = q6_dscale(hr[r], d[r], 2 * t + 1);
            float a = acc[r][0];
            a = fmaf(ds0 * S, planes_to_float(sp[r][0][0], sp[r][0][1], sp[r][0][2]), a);
            a = fmaf(ds0 * -32.0f, X0, a);
            a = fmaf(ds1 * S, planes_to_float(sp[r][1][0], sp[r][1][1], sp[r][1][2]), a);
            a = fmaf(ds1 * -32.0f, X1, a);
            acc[r][0] = a;
        }
    }
}

// The outlier term d*scale*(q - 32)*x of 32-column group t (its column i)
// of half n of the Q6_K super-block at `blk` in shared memory (a rare path,
// kept out of the unrolled arithmetic: the field bytes are read directly).
static __device__ __noinline__ float q6k_outlier_term(const uint8_t *blk, int n, int t, int i, float xv)
{
    const uint32_t lo = blk[64 * n + i + 32 * (t & 1)];
    const uint32_t hi = blk[128 + 32 * n + i];
    const int q = static_cast<int>(((t < 2 ? lo : (lo >> 4)) & 15u) | (((hi >> (2 * t)) & 3u) << 4));
    const float d = half_bits_to_float(static_cast<uint32_t>(blk[208]) | (static_cast<uint32_t>(blk[209]) << 8));
    const float sc = static_cast<float>(static_cast<int8_t>(blk[192 + 8 * n + 2 * t + (i >> 4)]));
    return (d * sc * static_cast<float>(q - 32)) * xv;
}

// The outlier term (d*sc*q - dmin*m)*x of column i of sub-block j of the
// Q4_K super-block at `sb` in shared memory; the weight is formed with one
// rounding (d*sc*q and dmin*m are exact).
static __device__ __noinline__ float q4k_outlier_term(const uint8_t *sb, int j, int i, float xv)
{
    const float d = half_bits_to_float(static_cast<uint32_t>(sb[0]) | (static_cast<uint32_t>(sb[1]) << 8));
    const float dmin = half_bits_to_float(static_cast<uint32_t>(sb[2]) | (static_cast<uint32_t>(sb[3]) << 8));
    const uint8_t *sc = sb + 4;
    uint32_t s6, m6;
    if (j < 4) {
        s6 = sc[j] & 63u;
        m6 = sc[j + 4] & 63u;
    } else {
        s6 = (sc[j + 4] & 15u) | ((sc[j - 4] >> 6) << 4);
        m6 = (sc[j + 4] >> 4) | ((sc[j] >> 6) << 4);
    }
    const uint32_t byte = sb[16 + 32 * (j >> 1) + i];
    const float q = static_cast<float>((j & 1) ? (byte >> 4) : (byte & 15u));
    const float w = fmaf(d * static_cast<float>(s6), q, -(dmin * static_cast<float>(m6)));
    return w * xv;
}

// The outlier term d*q*x of column i of the Q8_0 block at `blk` in shared
// memory (2-byte aligned).
static __device__ __noinline__ float q8_outlier_term(const uint8_t *blk, int i, float xv)
{
    const float d = half_bits_to_float(static_cast<uint32_t>(blk[0]) | (static_cast<uint32_t>(blk[1]) << 8));
    return (d * static_cast<float>(static_cast<int8_t>(blk[2 + i]))) * xv;
}

// Batch >= 2: fp32 x; each 6-bit quant becomes the exact float 2^23 + q (one
// byte permute into the magic pattern) and 2^23 + 32 is subtracted, giving
// q - 32 exactly; packed f32x2 arithmetic (float4 group g of batch row b at
// xa + 16*(32b + g)).
template <int B, int R>
__device__ __forceinline__ void q6k_half_fp(const Q6Half (&hr)[R], const uint8_t *xa, float (&acc)[R][B])
{
    const uint64_t neg_bias = pack2f(-(kTwo23 + 32.0f), -(kTwo23 + 32.0f));
    float d[R];
#pragma unroll
    for (int r = 0; r < R; ++r) d[r] = half_bits_to_float(hr[r].dw);
#pragma unroll
    for (int j = 0; j < 8; ++j) {                      // 16-column sub-block j: t = j/2, k = 4*(j%2) ..
        uint64_t part[R][B];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int b = 0; b < B; ++b) part[r][b] = 0ull;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const int t = j >> 1, k = 4 * (j & 1) + kk;
            uint64_t q01[R], q23[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const uint32_t q = q6_quad(hr[r], t, k);
                q01[r] = add_f32x2(pack2(__byte_perm(q, kMagic, 0x7440u), __byte_perm(q, kMagic, 0x7441u)), neg_bias);
                q23[r] = add_f32x2(pack2(__byte_perm(q, kMagic, 0x7442u), __byte_perm(q, kMagic, 0x7443u)), neg_bias);
            }
#pragma unroll
            for (int b = 0; b < B; ++b) {
                const ulonglong2 xv = *reinterpret_cast<const ulonglong2 *>(xa + 16 * (b * 32 + 8 * t + k));
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    part[r][b] = fma_f32x2(q01[r], xv.x, part[r][b]);
                    part[r][b] = fma_f32x2(q23[r], xv.y, part[r][b]);
                }
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float ds = q6_dscale(hr[r], d[r], j);
#pragma unroll
            for (int b = 0; b < B; ++b) {
                const float2 p2 = unpack2f(part[r][b]);
                acc[r][b] = fmaf(ds, p2.x + p2.y, acc[r][b]);
            }
        }
    }
}

// -------------------------------------------------------------------------- activations -> shared memory
//
// Layout (unit-major): unit slot us (Q4_K: h*XH + super-block for unit
// u = 2*super-block + h; else us = u) owns SU = B*G + 1 consecutive 16-byte
// slots, slot b*G + g holding float4 group g (columns 4g..4g+3 of the unit)
// of batch row b; the last slot is padding.  Sums of x: Q4_K batch 1 per 32
// columns at xsum[us*4 + j], batch >= 2 at xsum[(4b + j)*XU + us]; Q6_K
// (batch 1) per 16 columns at xsum[us*8 + j].  Batch 1 group scales at
// xscale[us*NJ + j].  (Per-unit sums and scales are read as one 16-byte
// vector, the batch >= 2 sums one scalar at a time, lanes on consecutive us.)
//
// One warp-uniform pass per batch row: each lane loads float4 group f of the
// row (columns 4f..4f+3; columns >= K are zero), consecutive lanes
// consecutive groups (coalesced), four groups a lane per round with the next
// round's loads in flight, and stores it at its slot; the 8 lanes of a
// 32-column group reduce it with shuffles, the four groups' shuffles
// interleaved.  Batch 1 stores block-floating-point byte planes (one
// exponent per 32 columns; a NaN or infinity in a group makes its scale
// NaN), batch >= 2 fp32 pre-multiplied by 2^-s for the Q4_K nibble position.
// The sum of eight values in a fixed order, the one at index `skip` left out.
__device__ __forceinline__ float sum8_skip(const float (&v)[8], int skip)
{
    float t[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) t[k] = k == skip ? 0.f : v[k];
    return ((t[0] + t[1]) + (t[2] + t[3])) + ((t[4] + t[5]) + (t[6] + t[7]));
}

// Batch 1: the activations as block-floating-point byte planes.  A lane
// takes 8 consecutive columns (two float4 slots of a unit) per piece, so a
// 32-column group is 4 lanes and its reductions are two shuffle levels.  Per
// group: its largest magnitude (exponent e1) and its plain sum (Q4_K: 32
// columns, Q6_K: its two 16-column halves).  An outlier is the only value of
// the group with an exponent >= e1 - 2 (so it is at least 2^3 times every
// other value).  One ballot finds groups where a single lane holds values
// that large; only a warp with such a group counts them exactly and redoes
// the reductions with the outlier left out.  The group's exponent is then
// that of its largest other value, the outlier's value and column go to
// xout for the exact side term, and the group scale's sign bit marks it.
// Each value becomes m = rint(x * 2^(21-E)), |m| <= 2^22, stored as three
// byte planes (planes 0, 1 unsigned, plane 2 signed; the fourth byte of each
// 16-byte slot unused); a group holding a NaN or an infinity gets a NaN
// scale (its planes then do not matter).
template <int FMT, int NTH>
__device__ __forceinline__ void stage_x1(const GemvArgs &a, const float *x0, uint32_t cwarp, uint32_t lane,
                                         uint32_t xs_addr, float *xsum, float *xscale, float *xout, uint32_t xgo)
{
    constexpr uint32_t UC = FMT == kFmtQ80 ? 32 : 128;
    constexpr uint32_t PU = UC / 8;         // 8-column pieces of a unit
    constexpr uint32_t NJ = UC / 32;
    constexpr uint32_t SU = UC / 4 + 1;     // 16-byte slots a unit slot owns
    constexpr uint32_t UNR = 2;
    static_assert(NTH % 32 == 0, "whole warps");
    const uint32_t XH = static_cast<uint32_t>(a.XU) >> 1;
    const uint32_t K = static_cast<uint32_t>(a.K);
    const uint32_t p_total = static_cast<uint32_t>(a.U) * PU;
    const bool vec = (K % 4 == 0) && ((reinterpret_cast<uintptr_t>(x0) & 15u) == 0);
    // pieces base + i*NTH + lane (i < UNR) of a round; the next round's loads
    // are issued before this round's arithmetic
    auto load = [&](uint32_t base, float (&v)[UNR][8]) {
        const uint32_t ns = min(UNR, (p_total - base + NTH - 1) / NTH);
#pragma unroll
        for (uint32_t i = 0; i < UNR; ++i) {
            const uint32_t pc = base + i * NTH + lane;
            const uint32_t c0 = 8 * pc;
#pragma unroll
            for (int k = 0; k < 8; ++k) v[i][k] = 0.f;
            if (i < ns && pc < p_total) {
                if (vec && c0 + 7 < K) {
                    const float4 lo = __ldg(reinterpret_cast<const float4 *>(x0 + c0));
                    const float4 hi = __ldg(reinterpret_cast<const float4 *>(x0 + c0) + 1);
                    v[i][0] = lo.x; v[i][1] = lo.y; v[i][2] = lo.z; v[i][3] = lo.w;
                    v[i][4] = hi.x; v[i][5] = hi.y; v[i][6] = hi.z; v[i][7] = hi.w;
                } else {
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        if (c0 + k < K) v[i][k] = __ldg(x0 + c0 + k);
                }
            }
        }
    };
    float v[UNR][8], nx[UNR][8];
    if (cwarp * 32 < p_total) load(cwarp * 32, v);
    if (cwarp == 0 && lane == 0) mbar_arrive(xgo);      // the first activation loads are out
    for (uint32_t base = cwarp * 32; base < p_total; base += UNR * NTH) {
        if (base + UNR * NTH < p_total) load(base + UNR * NTH, nx);   // the same for the warp
        // slots of this round with any piece in range (the same for the warp)
        const uint32_t ns = min(UNR, (p_total - base + NTH - 1) / NTH);
        uint32_t pc[UNR];
#pragma unroll
        for (uint32_t i = 0; i < UNR; ++i) pc[i] = base + i * NTH + lane;
        // magnitudes as bit patterns (their order is that of the values; a
        // NaN is above every number), the group maximum, the plain sums
        uint32_t ab[UNR][8], lmax[UNR], gmax[UNR], gref[UNR];
        float F[UNR];
        int oslot[UNR];
        bool outl[UNR];
        auto reduce = [&](uint32_t (&e)[UNR], float (&f)[UNR]) {
#pragma unroll
            for (int o = 1; o <= 2; o <<= 1)
#pragma unroll
                for (uint32_t i = 0; i < UNR; ++i)
                    if (i < ns) {
                        e[i] = max(e[i], __shfl_xor_sync(0xFFFFFFFFu, e[i], o));
                        if (FMT == kFmtQ4K || (FMT == kFmtQ6K && o < 2)) f[i] += __shfl_xor_sync(0xFFFFFFFFu, f[i], o);
                    }
        };
#pragma unroll
        for (uint32_t i = 0; i < UNR; ++i) {
#pragma unroll
            for (int k = 0; k < 8; ++k) ab[i][k] = __float_as_uint(v[i][k]) & 0x7FFFFFFFu;
            lmax[i] = max(max(max(ab[i][0], ab[i][1]), max(ab[i][2], ab[i][3])),
                          max(max(ab[i][4], ab[i][5]), max(ab[i][6], ab[i][7])));
            gmax[i] = lmax[i];
            F[i] = sum8_skip(v[i], -1);
        }
        reduce(gmax, F);
        // an outlier needs a group where one lane alone holds values with an
        // exponent >= e1 - 2 (one ballot); only a warp with such a group
        // counts them exactly
        bool cand_any = false;
        uint32_t thr[UNR];
#pragma unroll
        for (uint32_t i = 0; i < UNR; ++i) {
            const uint32_t e1 = gmax[i] >> 23;
            thr[i] = (e1 - 2u) << 23;
            const uint32_t g1 = (__ballot_sync(0xFFFFFFFFu, lmax[i] >= thr[i]) >> (lane & 28u)) & 0xFu;
            outl[i] = i < ns && e1 < 255u && e1 >= 2u && __popc(g1) == 1;   // candidate so far
            cand_any |= outl[i];
            oslot[i] = -1;
            gref[i] = gmax[i];
        }
        if (__any_sync(0xFFFFFFFFu, cand_any)) {
            // exact test: the group's one candidate lane holds a single such value
#pragma unroll
            for (uint32_t i = 0; i < UNR; ++i) {
                uint32_t c = 0;
                int first = -1;
#pragma unroll
                for (int k = 7; k >= 0; --k)
                    if (ab[i][k] >= thr[i]) {
                        ++c;
                        first = k;
                    }
                const uint32_t g2 = (__ballot_sync(0xFFFFFFFFu, c >= 2u) >> (lane & 28u)) & 0xFu;
                outl[i] = outl[i] && g2 == 0u;
                oslot[i] = (outl[i] && c == 1u) ? first : -1;
                // the reductions without the outlier (a group that has none gets
                // the same values again)
                uint32_t m = 0;
#pragma unroll
                for (int k = 0; k < 8; ++k) m = max(m, k == oslot[i] ? 0u : ab[i][k]);
                gref[i] = m;
                F[i] = sum8_skip(v[i], oslot[i]);
            }
            reduce(gref, F);
        }
#pragma unroll
        for (uint32_t i = 0; i < UNR; ++i) {
            if (!(i < ns) || pc[i] >= p_total) continue;
            const bool finite = (gmax[i] >> 23) != 255u;
            const int E = max(static_cast<int>(gref[i] >> 23) - 127, -96);
            const float up = __int_as_float((148 - E) << 23);     // 2^(21-E)
            const float d21 = __int_as_float((106 + E) << 23);    // 2^(E-21)
            const float dn = !finite ? __int_as_float(0x7FC00000) : (outl[i] ? -d21 : d21);
            // m = rint(x * 2^(21-E)): adding 1.5 * 2^23 in one fp32 FMA rounds
            // the exact x * 2^(21-E) to the nearest integer (ties to even); the
            // sum's bits minus those of 1.5 * 2^23 are m.  The outlier's m is 0.
            constexpr float kRound = 12582912.0f;
            constexpr uint32_t kRoundBits = 0x4B400000u;
            // (a group with a NaN or an infinity gets meaningless planes and a NaN scale)
            uint32_t mm[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
                mm[k] = (__float_as_uint(fmaf(v[i][k], up, kRound)) - kRoundBits) & (k == oslot[i] ? 0u : 0xFFFFFFFFu);
            const uint32_t u = pc[i] / PU, pu = pc[i] % PU;
            const uint32_t us = FMT == kFmtQ4K ? ((u & 1) * XH + (u >> 1)) : u;   // unit slot
            const uint32_t j = pu >> 2;                                          // 32-column group
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                // byte-plane transpose: plane k holds byte k of the four columns
                const uint32_t t0 = __byte_perm(mm[4 * h], mm[4 * h + 1], 0x5140u);
                const uint32_t t1 = __byte_perm(mm[4 * h + 2], mm[4 * h + 3], 0x5140u);
                const uint32_t t2 = __byte_perm(mm[4 * h], mm[4 * h + 1], 0x7362u);
                const uint32_t t3 = __byte_perm(mm[4 * h + 2], mm[4 * h + 3], 0x7362u);
                const uint32_t dst = xs_addr + 16u * (us * SU + 2 * pu + h);
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(__byte_perm(t0, t1, 0x5410u)),
                             "r"(__byte_perm(t0, t1, 0x7632u)), "r"(__byte_perm(t2, t3, 0x5410u)),
                             "r"(__byte_perm(t2, t3, 0x7632u))
                             : "memory");
            }
            if ((lane & 3) == 0) {
                xscale[us * NJ + j] = dn;
                if constexpr (FMT == kFmtQ4K) xsum[us * 4 + j] = F[i];
            }
            if constexpr (FMT == kFmtQ6K)
                if ((lane & 1) == 0) xsum[us * 8 + (pu >> 1)] = F[i];
            if (oslot[i] >= 0) {
                uint32_t xb = 0u;      // the outlier's bits, picked without indexing registers
#pragma unroll
                for (int k = 0; k < 8; ++k) xb |= __float_as_uint(v[i][k]) & (k == oslot[i] ? 0xFFFFFFFFu : 0u);
                xout[2 * (us * NJ + j)] = __uint_as_float(xb);
                xout[2 * (us * NJ + j) + 1] = __int_as_float(static_cast<int>(8 * (pu & 3)) + oslot[i]);
            }
        }
#pragma unroll
        for (uint32_t i = 0; i < UNR; ++i)
#pragma unroll
            for (int k = 0; k < 8; ++k) v[i][k] = nx[i][k];
    }
}

template <int FMT, int B, int NTH>
__device__ __forceinline__ void stage_x(const GemvArgs &a, const float *x0, uint32_t cwarp, uint32_t lane,
                                        uint32_t xs_addr, float *xsum, float *xscale, float *xout)
{
    constexpr uint32_t UC = FMT == kFmtQ80 ? 32 : 128;
    constexpr uint32_t G = UC / 4;          // float4 groups of a unit (a power of two)
    constexpr uint32_t SU = B * G + 1;
    constexpr uint32_t UNR = 4;
    static_assert(NTH % 32 == 0, "whole warps");
    const uint32_t XH = static_cast<uint32_t>(a.XU) >> 1;
    const uint32_t K = static_cast<uint32_t>(a.K);
    const uint32_t g_total = static_cast<uint32_t>(a.U) * G;
    const bool vec = (K % 4 == 0) && ((reinterpret_cast<uintptr_t>(x0) & 15u) == 0);
    for (uint32_t b = 0; b < B; ++b) {
        const float *xb = x0 + static_cast<uint64_t>(b) * K;
        // the float4 groups base + i*NTH + lane (i < UNR) of a round; when the
        // whole round lies inside K and x is 16-byte aligned the loads are
        // unconditional (the same test for every lane of the warp)
        auto load = [&](uint32_t base, float4 (&v)[UNR]) {
            const uint32_t last = base + (UNR - 1) * NTH + 31;
            if (vec && last < g_total && 4 * last + 3 < K) {
                const float4 *p = reinterpret_cast<const float4 *>(xb) + base + lane;
#pragma unroll
                for (uint32_t i = 0; i < UNR; ++i) v[i] = __ldg(p + i * NTH);
                return;
            }
#pragma unroll
            for (uint32_t i = 0; i < UNR; ++i) {
                const uint32_t f = base + i * NTH + lane;
                const uint32_t c0 = 4 * f;
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
        };
        float4 v[UNR], nx[UNR];
        uint32_t base = cwarp * 32;
        if (base < g_total) load(base, v);
        for (; base < g_total; base += UNR * NTH) {
            if (base + UNR * NTH < g_total) load(base + UNR * NTH, nx);   // warp-uniform
            uint32_t us[UNR], g[UNR];
            bool in[UNR];
#pragma unroll
            for (uint32_t i = 0; i < UNR; ++i) {
                const uint32_t f = base + i * NTH + lane;
                const uint32_t u = f / G;
                g[i] = f % G;
                in[i] = f < g_total;
                us[i] = FMT == kFmtQ4K ? ((u & 1) * XH + (u >> 1)) : u;   // unit slot
            }
            // plain sums: per float4, then over 4 lanes (16 columns) and 8 (32)
            float sum[UNR], sum16[UNR];
            auto plain_sums = [&](const float4 (&w)[UNR]) {
#pragma unroll
                for (uint32_t i = 0; i < UNR; ++i) sum[i] = (w[i].x + w[i].y) + (w[i].z + w[i].w);
                if constexpr (FMT != kFmtQ80) {
#pragma unroll
                    for (uint32_t i = 0; i < UNR; ++i) sum[i] += __shfl_xor_sync(0xFFFFFFFFu, sum[i], 1);
#pragma unroll
                    for (uint32_t i = 0; i < UNR; ++i) sum[i] += __shfl_xor_sync(0xFFFFFFFFu, sum[i], 2);
#pragma unroll
                    for (uint32_t i = 0; i < UNR; ++i) sum16[i] = sum[i];
                    if constexpr (FMT == kFmtQ4K) {
#pragma unroll
                        for (uint32_t i = 0; i < UNR; ++i) sum[i] += __shfl_xor_sync(0xFFFFFFFFu, sum[i], 4);
                    }
                }
            };
            {
                static_assert(B >= 2, "batch 1 is staged by stage_x1");
                plain_sums(v);
#pragma unroll
                for (uint32_t i = 0; i < UNR; ++i) {
                    float4 w = v[i];
                    if constexpr (FMT == kFmtQ4K) {
                        if (in[i] && (lane & 7) == 0) xsum[(b * 4 + (g[i] >> 3)) * static_cast<uint32_t>(a.XU) + us[i]] = sum[i];
                        const int c = static_cast<int>(4 * g[i]);
                        w.x *= __int_as_float((127 - q4k_nibble_shift(c)) << 23);
                        w.y *= __int_as_float((127 - q4k_nibble_shift(c + 1)) << 23);
                        w.z *= __int_as_float((127 - q4k_nibble_shift(c + 2)) << 23);
                        w.w *= __int_as_float((127 - q4k_nibble_shift(c + 3)) << 23);
                    }
                    if (in[i]) {
                        const uint32_t dst = xs_addr + 16u * (us[i] * SU + b * G + g[i]);
                        asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};"
                                     ::"r"(dst), "f"(w.x), "f"(w.y), "f"(w.z), "f"(w.w) : "memory");
                    }
                }
            }
#pragma unroll
            for (uint32_t i = 0; i < UNR; ++i) v[i] = nx[i];
        }
    }
}

// -------------------------------------------------------------------------- kernel

// Copy the item of rows [row0, row0+n) (pair mode: n gate rows and their n up
// rows), K chunk c, into the stage at `dst`; completion on `bar`.  Whole rows
// are contiguous: one 1-D bulk copy per span (the up span at up_stage_off),
// else one per row (row lr at lr*row_stride; pair mode: up row lr at
// (rows_w/2 + lr)*row_stride).  Spans are widened to 16-byte boundaries; a
// 16-byte granule holding a byte of the tensor never crosses a page, so the
// widened copy stays in mapped memory.
__device__ __forceinline__ uint32_t span16(uintptr_t gs, uintptr_t ge)
{
    return static_cast<uint32_t>(((ge + 15) & ~static_cast<uintptr_t>(15)) - (gs & ~static_cast<uintptr_t>(15)));
}

__device__ __forceinline__ void copy_item(const GemvArgs &a, bool pair, const uint8_t *w0, int64_t row0, int n,
                                          uint32_t c, uint32_t dst, uint32_t bar, uint64_t pol)
{
    const uint8_t *g0 = w0 + row0 * a.row_bytes;
    const uint8_t *u0 = pair ? g0 + a.up_rows * a.row_bytes : nullptr;
    if (a.nkc == 1) {
        const uintptr_t gs = reinterpret_cast<uintptr_t>(g0), ge = gs + static_cast<uintptr_t>(n * a.row_bytes);
        uint32_t bytes = span16(gs, ge);
        uint32_t ubytes = 0;
        uintptr_t us = 0;
        if (pair) {
            us = reinterpret_cast<uintptr_t>(u0);
            ubytes = span16(us, us + static_cast<uintptr_t>(n * a.row_bytes));
        }
        mbar_arrive_expect_tx(bar, bytes + ubytes);
        bulk_g2s(dst, reinterpret_cast<const void *>(gs & ~static_cast<uintptr_t>(15)), bytes, bar, pol);
        if (pair)
            bulk_g2s(dst + static_cast<uint32_t>(a.up_stage_off),
                     reinterpret_cast<const void *>(us & ~static_cast<uintptr_t>(15)), ubytes, bar, pol);
        return;
    }
    const int64_t cb = static_cast<int64_t>(c) * a.chunk_bytes;
    const int64_t cl = min(static_cast<int64_t>(a.chunk_bytes), a.row_bytes - cb);
    const int spans = pair ? 2 : 1;
    const int P = a.rows_w >> 1;
    uint32_t total = 0;
    for (int h = 0; h < spans; ++h)
        for (int q = 0; q < n; ++q) {
            const uintptr_t gs = reinterpret_cast<uintptr_t>((h ? u0 : g0) + q * a.row_bytes + cb);
            total += span16(gs, gs + static_cast<uintptr_t>(cl));
        }
    mbar_arrive_expect_tx(bar, total);
    for (int h = 0; h < spans; ++h)
        for (int q = 0; q < n; ++q) {
            const uintptr_t gs = reinterpret_cast<uintptr_t>((h ? u0 : g0) + q * a.row_bytes + cb);
            const int lr = h ? P + q : q;
            bulk_g2s(dst + static_cast<uint32_t>(lr * a.row_stride),
                     reinterpret_cast<const void *>(gs & ~static_cast<uintptr_t>(15)),
                     span16(gs, gs + static_cast<uintptr_t>(cl)), bar, pol);
        }
}

// MODE: kModeAny, or a plain call (no SwiGLU pair, no experts mode) whose
// row groups are split over warps (kModePlain) or not (kModePlainKw1).  The
// code a plain instantiation does not need is left out: a smaller kernel
// costs less instruction fetch when calls of different shapes alternate.
constexpr int kModeAny = 0, kModePlain = 1, kModePlainKw1 = 2;

template <int FMT, int B, bool WIDE = false, int MODE = kModeAny>
__global__ void __launch_bounds__(32 * (gemv_warps(FMT, B, WIDE) + 1), 1) gemv_kernel(const GemvArgs a)
{
    constexpr bool PLAIN = MODE != kModeAny;
    const bool pair = !PLAIN && a.pair != 0;
    const bool experts = !PLAIN && a.cpa > 0;
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int R = gemv_rows(FMT, B);
    constexpr int NW = gemv_warps(FMT, B, WIDE);
    constexpr int CM = gemv_cpl_max(FMT, B);
    constexpr int UB = FMT == kFmtQ4K ? 144 : 34;    // bytes per lane unit (Q4_K, Q8_0)
    const int tid = threadIdx.x;
    const uint32_t nw = static_cast<uint32_t>(a.nw);  // consumer warps with row groups
    const uint32_t m = static_cast<uint32_t>(a.m);    // stages per consumer warp
    const uint32_t bar_full = smem_u32(smem);
    const uint32_t bar_empty = bar_full + 256u;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + 512);
    const uint32_t bar_xgo = bar_full + 656u;
    int *issued_use = reinterpret_cast<int *>(smem + 528);   // per stage: use of its last copy, -1 none

    // this CTA's rows, weights, activations and outputs
    const uint8_t *w0 = a.w;
    const float *x0 = a.x;
    float *y0 = a.y;
    int64_t r_begin, r_end;
    if (experts) {
        // experts mode: CTA -> (assignment, part of the expert's rows); the
        // expert id comes from an earlier kernel, so wait for it first
        const int64_t asg = blockIdx.x / a.cpa, j = blockIdx.x - asg * a.cpa;
        r_begin = (a.rows * j) / a.cpa;
        r_end = (a.rows * (j + 1)) / a.cpa;
        asm volatile("griddepcontrol.wait;" ::: "memory");
        const int64_t e = a.expid[asg];
        y0 = a.y + asg * a.ldy;
        if (e < 0 || e >= a.n_experts) {
            // an id outside the tensor: nothing is read, the rows are NaN
            for (int64_t r = r_begin + tid; r < r_end; r += blockDim.x) y0[r] = __int_as_float(0x7FC00000);
            if (tid == 0) record_error(a.err, kErrBadIndex);
            return;
        }
        w0 = a.w + e * a.rows * a.row_bytes;
        x0 = a.x + (asg / a.xk) * a.K;
    } else {
        const int64_t nG = gridDim.x;
        r_begin = (a.rows * blockIdx.x) / nG;
        r_end = (a.rows * (blockIdx.x + 1)) / nG;
    }
    const int gr = pair ? (a.rows_w >> 1) : a.rows_w;   // output rows per row group
    const uint32_t n_groups = static_cast<uint32_t>((r_end - r_begin + gr - 1) / gr);
    const uint32_t nkc = static_cast<uint32_t>(a.nkc);
    const uint32_t kw = MODE == kModePlainKw1 ? 1u : static_cast<uint32_t>(a.kw);

    // programmatic dependent launch: the next grid in the stream may start
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (tid == 0) {
        for (uint32_t s = 0; s < nw * m; ++s) {
            mbar_init(bar_full + 8u * s, 1);
            mbar_init(bar_empty + 8u * s, 1);
            issued_use[s] = -1;
        }
        mbar_init(bar_xgo, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    const uint32_t stage0 = smem_u32(smem + a.off_stage);

    // ------------------------------------------------------------------ producer
    // Lane w of warp 0 feeds consumer warp w: row groups w, w+nw, ..., each
    // as nkc K-chunk items; item t of the warp goes to stage w*m + t%m.  The
    // warps' pipelines are independent, so no warp waits behind another.
    if (tid < 32) {
        const uint32_t w = static_cast<uint32_t>(tid);
        if (w < nw) {
            const uint64_t pol = l2_evict_first_policy();
            bool ok = true;
            uint32_t t = 0, tm = 0, use = 0;                 // item number, its stage offset and use
            // Batch 1: only the first items' copies (about 48 KB a CTA, what
            // lands while the CTA waits for the previous grid) go out before
            // the activations' loads; the others wait until those are issued,
            // so that the activations do not queue behind them.  (Measured on
            // the Llama-8B layer set: gate+up 15.5 -> 14.9 us, ffn_down 11.7 ->
            // 11.5 us; 24 KB held qkv back, 80 KB gained less.)
            const uint32_t p1 = max(1u, 49152u / static_cast<uint32_t>(a.stage_bytes));
            bool held = B == 1 && w >= p1;
            for (uint32_t g = w / kw; ok && g < n_groups; g += nw / kw) {
                const int64_t row0 = r_begin + static_cast<int64_t>(g) * gr;
                const int n = static_cast<int>(min(static_cast<int64_t>(gr), r_end - row0));
                for (uint32_t c = w % kw; c < nkc; c += kw, ++t) {
                    const uint32_t st = w * m + tm;
                    const uint32_t bar = bar_full + 8u * st;
                    if (held) {
                        held = false;
                        if (!mbar_wait_sleep(bar_xgo, 0, a.wait_ns)) {
                            ok = false;
                            break;
                        }
                    }
                    if (*abort_flag || (use > 0 && !mbar_wait_sleep(bar_empty + 8u * st, (use - 1) & 1u, a.wait_ns))) {
                        ok = false;
                        break;
                    }
                    const bool skip = w == 0 && t == a.skip_item && blockIdx.x == 0;   // test hook
                    if (!skip) {
                        copy_item(a, pair, w0, row0, n, c, stage0 + st * static_cast<uint32_t>(a.stage_bytes), bar, pol);
                        issued_use[st] = static_cast<int>(use);
                    }
                    if (++tm == m) {
                        tm = 0;
                        ++use;
                    }
                }
            }
            if (!ok) {
                *abort_flag = 1;
                record_error(a.err, kErrTimeout);
                // let this warp's copies already issued land before the CTA exits
                for (uint32_t q = 0; q < m; ++q) {
                    const int u = issued_use[w * m + q];
                    if (u >= 0) mbar_wait(bar_full + 8u * (w * m + q), static_cast<uint32_t>(u) & 1u, a.wait_ns);
                }
            }
        }
        return;
    }

    // ------------------------------------------------------------------ consumers
    const uint32_t cwarp = static_cast<uint32_t>((tid >> 5) - 1);
    const int lane = tid & 31;
    const int SW = a.SW;
    const int team = lane >> a.lsw;
    const int sl = lane & (SW - 1);
    const int cpl = a.cpl;
    const int XH = a.XU >> 1;
    constexpr int SU = B * (FMT == kFmtQ80 ? 8 : 32) + 1;   // 16-byte slots a unit slot owns
    const uint8_t *xs = smem + a.off_x;
    const float *xsum = reinterpret_cast<const float *>(smem + a.off_xsum);
    const float *xscale = reinterpret_cast<const float *>(smem + a.off_xscale);
    const float *xout = reinterpret_cast<const float *>(smem + a.off_xout);

    // the weights do not depend on earlier kernels, x may: with programmatic
    // dependent launch only this part waits for the previous grid
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if constexpr (B == 1)
        stage_x1<FMT, 32 * NW>(a, x0, cwarp, static_cast<uint32_t>(lane), smem_u32(xs),
                               reinterpret_cast<float *>(smem + a.off_xsum),
                               reinterpret_cast<float *>(smem + a.off_xscale),
                               reinterpret_cast<float *>(smem + a.off_xout), bar_xgo);
    else
        stage_x<FMT, B, 32 * NW>(a, x0, cwarp, static_cast<uint32_t>(lane), smem_u32(xs),
                                 reinterpret_cast<float *>(smem + a.off_xsum),
                                 reinterpret_cast<float *>(smem + a.off_xscale),
                                 reinterpret_cast<float *>(smem + a.off_xout));
    named_bar_sync(1, 32 * NW);
    if (cwarp >= nw) return;

    // the team sums of a row group and its outputs
    auto finish = [&](int64_t row0, int n, const float (&acc)[R][B]) {
        // sum over the SW lanes of each team (every lane of the team gets it)
        float v[R][B];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int b = 0; b < B; ++b) {
                float t = acc[r][b];
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1)
                    if (o < SW) t += __shfl_xor_sync(0xFFFFFFFFu, t, o);   // SW is the same for the warp
                v[r][b] = t;
            }
        if (!pair) {
            // lane 0 of the team writes its rows
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int b = 0; b < B; ++b) {
                    const int lr = team * R + r;
                    if (sl == 0 && lr < n) y0[b * a.ldy + row0 + lr] = v[r][b];
                }
        } else if (SW == 32) {
            // one team: rows r < R/2 are gate rows, r + R/2 their up rows
#pragma unroll
            for (int r = 0; r < R / 2; ++r)
#pragma unroll
                for (int b = 0; b < B; ++b)
                    if (sl == 0 && r < n) y0[b * a.ldy + row0 + r] = silu(v[r][b]) * v[r + R / 2][b];
        } else {
            // teams t < T/2 hold gate rows, team t + T/2 (lanes + 16) the up rows
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int b = 0; b < B; ++b) {
                    const float u = __shfl_down_sync(0xFFFFFFFFu, v[r][b], 16);
                    const int lr = team * R + r;
                    if (lane < 16 && sl == 0 && lr < n) y0[b * a.ldy + row0 + lr] = silu(v[r][b]) * u;
                }
        }
    };
    float *part = reinterpret_cast<float *>(smem + a.off_part);
    const uintptr_t wbase = reinterpret_cast<uintptr_t>(w0);
    const int chunk_lu = SW * cpl;                 // lane units per chunk
    const uint32_t st0 = cwarp * m;                // this warp's stages st0 .. st0+m-1
    uint32_t tm = 0, par = 0;                      // stage offset and parity of the next item
    bool failed = false;
    const uint32_t g_first = cwarp / kw, g_step = nw / kw, c_first = cwarp % kw;
    // batch 1: bit c set when this lane's units of chunk c have a group with
    // an outlier (a sign bit of a group scale), found once after staging
    uint64_t omask = 0;
    if constexpr (B == 1) {
        for (uint32_t c = c_first; c < nkc && c < 64; c += kw) {
            uint32_t sg = 0;
            for (int i = 0; i < cpl; ++i) {
                const int lu = static_cast<int>(c) * SW * cpl + i * SW + sl;
                if (lu >= a.LU) break;
                if constexpr (FMT == kFmtQ80) {
                    sg |= __float_as_uint(xscale[lu]);
                } else {
                    const uint4 s0 = *reinterpret_cast<const uint4 *>(xscale + 4 * lu);
                    sg |= s0.x | s0.y | s0.z | s0.w;
                    if constexpr (FMT == kFmtQ4K) {
                        const uint4 s1 = *reinterpret_cast<const uint4 *>(xscale + 4 * (XH + lu));
                        sg |= s1.x | s1.y | s1.z | s1.w;
                    }
                }
            }
            if (sg >> 31) omask |= 1ull << c;
        }
        if (nkc > 64) omask = ~0ull;                 // (beyond 64 chunks: every chunk is checked)
    }
    for (uint32_t g = g_first; g < n_groups && !failed; g += g_step) {
        const int64_t row0 = r_begin + static_cast<int64_t>(g) * gr;
        const int n = static_cast<int>(min(static_cast<int64_t>(gr), r_end - row0));
        float acc[R][B];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int b = 0; b < B; ++b) acc[r][b] = 0.f;
        for (uint32_t c = c_first; c < nkc; c += kw) {
            const uint32_t st = st0 + tm;
            const bool ochunk = B == 1 && ((omask >> (c < 64 ? c : 63)) & 1u) != 0;
            bool ok = mbar_wait_sleep(bar_full + 8u * st, par, a.wait_ns);
            ok = __all_sync(0xFFFFFFFFu, ok);   // the warp leaves together or not at all
            if (!ok) {
                if (lane == 0) {
                    *abort_flag = 1;
                    record_error(a.err, kErrTimeout);
                }
                failed = true;
                break;
            }
            const uint8_t *stage = smem + a.off_stage + st * static_cast<uint32_t>(a.stage_bytes);
            // where this lane's rows start their chunk in the stage (rows past
            // the group's end read its last row and are not stored)
            // (pair mode: the item's rows lr < P are gate rows, the rest their up rows)
            const uint8_t *rowp[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                int lr = team * R + r;
                const bool up = pair && lr >= gr;
                const int q = min(up ? lr - gr : lr, n - 1);      // output row within the group
                const int64_t grow = row0 + q + (up ? a.up_rows : 0);   // weight row
                if (nkc == 1) {
                    const uintptr_t gsrc = wbase + static_cast<uintptr_t>((row0 + (up ? a.up_rows : 0)) * a.row_bytes);
                    rowp[r] = stage + (up ? a.up_stage_off : 0) + (gsrc & 15u) + static_cast<int64_t>(q) * a.row_bytes;
                } else {
                    lr = up ? gr + q : q;
                    const uintptr_t gsrc = wbase + static_cast<uintptr_t>(grow * a.row_bytes) +
                                           static_cast<uintptr_t>(c) * a.chunk_bytes;
                    rowp[r] = stage + lr * a.row_stride + (gsrc & 15u);
                }
            }
            // lane units of this lane in this chunk: i*SW + sl (i < cpl) from
            // the chunk's start, lane unit c*chunk_lu + i*SW + sl of the row
            // this chunk's sums, started from zero: the row's sum adds them up
            // in chunk order (the same order when the chunks of a row group
            // are shared by kw warps)
            float pacc[R][B];
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int b = 0; b < B; ++b) pacc[r][b] = 0.f;
            const int lu0 = static_cast<int>(c) * chunk_lu + sl;
            // batch 1: the exact terms of the outliers of this lane's groups,
            // read from the stage before it is handed back (rare: a sign bit
            // of a group scale), added after the unit's plane terms
            float oterm[R];
#pragma unroll
            for (int r = 0; r < R; ++r) oterm[r] = 0.f;
            if constexpr (FMT == kFmtQ4K) {
                // a lane past the row's last unit (only in a row's last chunk)
                // works on that last unit and its sums are dropped
                const bool valid = lu0 < a.LU;
                const int lu = valid ? lu0 : a.LU - 1;
                const int su = lu - static_cast<int>(c) * chunk_lu;   // the unit within the chunk
                const bool has_hi = 2 * lu + 1 < a.U;
                auto outliers = [&]() {
                    if (ochunk && valid) {
                        const float4 s0 = *reinterpret_cast<const float4 *>(xscale + 4 * lu);
                        const float4 s1 = *reinterpret_cast<const float4 *>(xscale + 4 * (XH + lu));
                        const float sv[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
                        for (int j = 0; j < 8; ++j)
                            if (sv[j] < 0.f && (j < 4 || has_hi)) {
                                const int slot = 8 * ((j < 4 ? 0 : XH) + lu) + 2 * (j & 3);
                                const float xv = xout[slot];
                                const int i = __float_as_int(xout[slot + 1]);
#pragma unroll
                                for (int r = 0; r < R; ++r)
                                    oterm[r] += q4k_outlier_term(rowp[r] + su * UB, j, i, xv);
                            }
                    }
                };
              if constexpr (B == 1 && WIDE) {
                // one 128-column half at a time: the stage is handed back once
                // the second half is in registers
                uint4 hd[R], q4[R][4];
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const uint4 *p = reinterpret_cast<const uint4 *>(rowp[r] + su * UB);
                    hd[r] = p[0];
#pragma unroll
                    for (int i = 0; i < 4; ++i) q4[r][i] = p[1 + i];
                }
                q4k_half_dig<R, 0>(hd, q4, xs + 16 * SU * lu, xsum + 4 * lu, xscale + 4 * lu, pacc);
                if (has_hi) {
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const uint4 *p = reinterpret_cast<const uint4 *>(rowp[r] + su * UB);
#pragma unroll
                        for (int i = 0; i < 4; ++i) q4[r][i] = p[5 + i];
                    }
                }
                outliers();
                __syncwarp();
                mbar_arrive_if(bar_empty + 8u * st, lane == 0);   // the stage may be refilled
                if (has_hi)
                    q4k_half_dig<R, 1>(hd, q4, xs + 16 * SU * (XH + lu), xsum + 4 * (XH + lu),
                                       xscale + 4 * (XH + lu), pacc);
              } else {
                uint4 hd[R], qs[R][8];
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const uint4 *p = reinterpret_cast<const uint4 *>(rowp[r] + su * UB);
                    hd[r] = p[0];
#pragma unroll
                    for (int i = 0; i < 8; ++i) qs[r][i] = p[1 + i];
                }
                outliers();
                __syncwarp();
                mbar_arrive_if(bar_empty + 8u * st, lane == 0);   // the stage may be refilled
                const uint8_t *xa0 = xs + 16 * SU * lu;
                const uint8_t *xa1 = xs + 16 * SU * (XH + lu);
                if constexpr (B == 1)
                    q4k_sb_dig<R>(hd, qs, has_hi, xa0, xa1, xsum + 4 * lu, xsum + 4 * (XH + lu),
                                  xscale + 4 * lu, xscale + 4 * (XH + lu), pacc);
                else if (valid)
                    q4k_sb_fp<B, R>(hd, qs, has_hi, xa0, xa1, xsum + lu, xsum + XH + lu, a.XU, pacc);
              }
                if constexpr (B == 1) {
#pragma unroll
                    for (int r = 0; r < R; ++r) pacc[r][0] = valid ? pacc[r][0] + oterm[r] : 0.f;
                }
            } else if constexpr (FMT == kFmtQ6K) {
                // lane unit = half super-block: block li/2 of the chunk, half li%2
                // (a chunk holds whole super-blocks: chunk_lu is even when nkc > 1)
                Q6Half hr[R];
                const bool valid = lu0 < a.LU;
                const int lu = valid ? lu0 : a.LU - 1;     // past the row's end: its last unit, sums dropped
                const int su = lu - static_cast<int>(c) * chunk_lu;
#pragma unroll
                for (int r = 0; r < R; ++r) q6_load(rowp[r] + (su >> 1) * 210, lu & 1, hr[r]);
                if constexpr (B == 1) {
                    if (ochunk && valid) {
                        const float4 sc4 = *reinterpret_cast<const float4 *>(xscale + 4 * lu);
                        const float scv[4] = {sc4.x, sc4.y, sc4.z, sc4.w};
                        for (int t = 0; t < 4; ++t)
                            if (scv[t] < 0.f) {
                                const float xv = xout[8 * lu + 2 * t];
                                const int i = __float_as_int(xout[8 * lu + 2 * t + 1]);
#pragma unroll
                                for (int r = 0; r < R; ++r)
                                    oterm[r] += q6k_outlier_term(rowp[r] + (su >> 1) * 210, lu & 1, t, i, xv);
                            }
                    }
                }
                __syncwarp();
                mbar_arrive_if(bar_empty + 8u * st, lane == 0);   // the stage may be refilled
                const uint8_t *xa = xs + 16 * SU * lu;
                if constexpr (B == 1) {
                    q6k_half_dig<R>(hr, xa, xsum + 8 * lu, xscale + 4 * lu, pacc);
#pragma unroll
                    for (int r = 0; r < R; ++r) pacc[r][0] = valid ? pacc[r][0] + oterm[r] : 0.f;
                } else if (valid) {
                    q6k_half_fp<B, R>(hr, xa, pacc);
                }
            } else {
                // one block at a time (words in registers, realigned), the stage
                // handed back once the lane's last block of the item is loaded
#pragma unroll
                for (int i = 0; i < CM; ++i) {
                    if (i >= cpl) break;
                    const int lu = lu0 + i * SW;
                    const bool has = lu < a.LU;
                    uint32_t wv[R][9], off[R];
                    if (has) {
#pragma unroll
                        for (int r = 0; r < R; ++r) {
                            const uint32_t sa = static_cast<uint32_t>(
                                __cvta_generic_to_shared(rowp[r] + (i * SW + sl) * UB));
                            off[r] = sa & 3u;          // 0 or 2
                            // (formed in the shared window: shared-memory loads, not generic ones)
                            const uint32_t *wp = static_cast<const uint32_t *>(__cvta_shared_to_generic(sa - off[r]));
#pragma unroll
                            for (int k = 0; k < 9; ++k) wv[r][k] = wp[k];
                        }
                        if (B == 1 && ochunk && xscale[lu] < 0.f) {
                            const float xv = xout[2 * lu];
                            const int ic = __float_as_int(xout[2 * lu + 1]);
#pragma unroll
                            for (int r = 0; r < R; ++r)
                                oterm[r] += q8_outlier_term(rowp[r] + (i * SW + sl) * UB, ic, xv);
                        }
                    }
                    if (i == cpl - 1) {
                        __syncwarp();
                        mbar_arrive_if(bar_empty + 8u * st, lane == 0);   // the stage may be refilled
                    }
                    if (has) {
                        const uint8_t *xa = xs + 16 * SU * lu;
                        if constexpr (B == 1)
                            q8_blk_dig<R>(wv, off, xa, xscale[lu], pacc);
                        else
                            q8_blk_fp<B, R>(wv, off, xa, pacc);
                    }
                }
                if constexpr (B == 1) {
#pragma unroll
                    for (int r = 0; r < R; ++r) pacc[r][0] += oterm[r];
                }
            }
            if (kw == 1) {
#pragma unroll
                for (int r = 0; r < R; ++r)
#pragma unroll
                    for (int b = 0; b < B; ++b) acc[r][b] += pacc[r][b];
            } else {
                float *pp = part + ((g * nkc + c) * 32u + static_cast<uint32_t>(lane)) * (R * B);
#pragma unroll
                for (int r = 0; r < R; ++r)
#pragma unroll
                    for (int b = 0; b < B; ++b) pp[r * B + b] = pacc[r][b];
            }
            if (++tm == m) {
                tm = 0;
                par ^= 1u;
            }
        }
        if (failed) break;
        if (kw == 1) finish(row0, n, acc);
    }
    if (kw > 1) {
        // the warps of a row group meet; its first warp adds the chunk sums
        // in chunk order and writes the outputs
        named_bar_sync(2, 32 * static_cast<int>(nw));
        const uint32_t g = cwarp / kw;
        if (!failed && cwarp % kw == 0 && g < n_groups) {
            const int64_t row0 = r_begin + static_cast<int64_t>(g) * gr;
            const int n = static_cast<int>(min(static_cast<int64_t>(gr), r_end - row0));
            float acc[R][B];
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int b = 0; b < B; ++b) acc[r][b] = 0.f;
            for (uint32_t c = 0; c < nkc; ++c) {
                const float *pp = part + ((g * nkc + c) * 32u + static_cast<uint32_t>(lane)) * (R * B);
#pragma unroll
                for (int r = 0; r < R; ++r)
#pragma unroll
                    for (int b = 0; b < B; ++b) acc[r][b] += pp[r * B + b];
            }
            finish(row0, n, acc);
        }
    }
}

// Launch one instantiation (defined per format in qk_gemv_q4k.cu / qk_gemv_q80.cu / qk_gemv_q6k.cu).
cudaError_t gemv_launch_q4k(int batch, bool wide, const GemvArgs &a, int grid, int smem, cudaStream_t st, bool pdl);
cudaError_t gemv_launch_q80(int batch, const GemvArgs &a, int grid, int smem, cudaStream_t st, bool pdl);
cudaError_t gemv_launch_q6k(int batch, bool wide, const GemvArgs &a, int grid, int smem, cudaStream_t st, bool pdl);

template <int FMT, int B, bool WIDE = false, int MODE = kModeAny>
cudaError_t gemv_launch_one(const GemvArgs &a, int grid, int smem, cudaStream_t st, bool pdl)
{
    auto kern = gemv_kernel<FMT, B, WIDE, MODE>;
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
    cfg.blockDim = dim3(32 * (gemv_warps(FMT, B, WIDE) + 1));
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

}  // namespace qk
