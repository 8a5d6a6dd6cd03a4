// qk_gemv_tc.cu -- the batch 2..8 GEMV of Q8_0 and Q4_K weights on the
// tensor cores (tcgen05, kind::f16, A operand in tensor memory).
//
// y[b][r] = sum_c W[r][c] * x[b][c] for 2..8 activation rows.  The weights
// are still read once from HBM; what changes against the fp32 form is where
// the multiply-adds run:
//
//   x (the B operand, shared memory): every batch row b and 32-column group g
//     is scaled by a power of two S[g][b] chosen from the group's largest
//     magnitude (one outlier per group, by the batch-1 rule, is set aside
//     and added exactly), and split into two fp16 pieces hi + lo, which hold
//     the scaled value to 2^-24 of itself.  Row b of the B matrix holds the
//     hi pieces of batch row b, row B + b its lo pieces (MMA N = 16).
//   W (the A operand, tensor memory): each thread of the 16 converter warps
//     (4 per tensor-memory lane quarter, each taking 2 of an item's 8
//     groups, or 1 of a Q8_0 row's last half item) decodes its part of one weight row of a 128-row tile into
//     exact fp16 integers (Q8_0: q; Q4_K: q, or 16q for the high nibbles,
//     whose x pieces are scaled down by 16 to match) and stores them into
//     its tensor-memory lane.
//   MMA: per 32-column group two kind::f16 MMAs (K = 16 each) write
//     sum_c q[r][c] * piece[n][c] into the group's own 16 accumulator columns;
//     the block scale differs per row and group, so groups are not summed on
//     the tensor core.
//   Epilogue: the converter threads read their lane's accumulators back,
//     add the two pieces, undo S and apply d (Q8_0) or d*sc and dmin*m with
//     the group's sum of x (Q4_K), in the same order for every row; at the
//     end of a tile the 4 warps of a lane quarter add their sums in order.
//
// A tile's 256-column items flow through a ring of stages (TMA boxes of 64
// or 128 rows issued by one producer thread: a bulk copy a row, or 16-byte
// copies, would be too many operations to keep HBM busy), two tensor-memory
// buffers for A and two for the accumulators: converting item i overlaps
// the MMAs of item i-1, whose accumulators are read back right after.
// Each weight row's arithmetic depends on K only, never on where the row
// sits in a tile or which CTA holds it, so row ranges of a tensor give the
// same bits as one call.
#include <cstdint>
#include <cstring>
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "qk_device.cuh"
#include "qk_internal.h"
#include "qk_tc.cuh"

namespace qk {

namespace {

constexpr int kTcM = 128;              // weight rows a tile (MMA M)
constexpr int kTcKC = 256;             // columns an item
constexpr int kTcCW = 4;               // converter warps a tensor-memory lane quarter
constexpr int kTcGPW = 8 / kTcCW;      // 32-column groups a converter warp takes of each item
constexpr int kTcConvWarps = 4 * kTcCW;
constexpr int kTcIssuer = 0;           // the MMA issuer's warp (it also holds the tensor memory)
constexpr int kTcProducer = 1;         // the stage producer's warp; the converters follow
constexpr int kTcThreads = 32 * (2 + kTcConvWarps);
constexpr int kQ8Half = 64 * 144;      // Q8_0 stage: four boxes of 64 rows x 144 bytes
constexpr int kTcMaxStages = 8;
constexpr uint32_t kTcCols = 512;      // tensor memory: A x2 (128 columns each), accumulators x2 (128 each)
constexpr int kTcBarBytes = 1024;

struct GemvTcArgs {
    const uint8_t *w;      // first weight row of the call
    const float *x;        // [B][K]
    float *y;              // [B][ldy]
    int64_t rows, K, ldy, row_bytes;
    int G;                 // 32-column groups of K padded to whole blocks
    int NC;                // items a tile: 256-column chunks
    int chunk_bytes;       // bytes of a whole chunk of a row
    int row_stride;        // bytes a row takes in a stage
    int stage_bytes, NS;
    int off_bop, off_scale, off_xsum, off_out, off_flag, off_xch, off_stage;
    int ks;                // 1: K split over a cluster of two CTAs (the odd CTA takes the items
                           // c >= NC/2 of every tile and hands its row sums to the even one)
    int off_ksx;           // ks: the odd CTA's row sums of a tile [2 buffers][128 rows][8], in the even CTA
    int ph0, ph1;          // Q8_0: 16-byte phase of the rows of even / odd index within their boxes
    int64_t skip_item;     // test hook: CTA 0 never loads this item (-1: off)
    uint64_t wait_ns;
    int *err;
};

// barrier block (offsets from the 1024-aligned base)
static_assert((kTcCW & (kTcCW - 1)) == 0, "the exchange counts arrivals modulo kTcCW");
// (kXCount: per tile parity and lane quarter, the converter warps that have
// left their partial sums of a tile)
// (kKsFull, kKsEmpty: K split over a cluster, per buffer of the odd CTA's row
// sums: written (in the even CTA), and read (in the odd CTA))
constexpr uint32_t kBarFull = 0, kBarEmpty = 64, kBarAFull = 128, kBarMma = 144, kKsFull = 160, kKsEmpty = 176,
                   kTmemSlot = 192, kAbort = 196, kXCount = 200;

// One lane of the (converged) warp is elected.
__device__ __forceinline__ bool elect_one()
{
    uint32_t r;
    asm volatile("{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}" : "=r"(r));
    return r != 0;
}

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t m, uint32_t o)
{
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "r"(m), "r"(o));   // (a & m) | o
    return r;
}

__device__ __forceinline__ uint32_t hadd2_bits(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// Position within a group of the x value that the MMA's K index kp meets:
// the Q4_K conversion below pairs nibbles (l, l+2) and (l+1, l+3) of a word,
// which swaps bits 0 and 1 of the position; Q8_0 keeps the natural order.
template <int FMT>
__host__ __device__ constexpr int tc_kperm(int kp)
{
    return FMT == kFmtQ4K ? ((kp & ~3) | ((kp & 1) << 1) | ((kp >> 1) & 1)) : kp;
}

// Byte offset in the B operand (128-byte swizzled K-major rows of 64
// columns, 8-row atoms, 16 rows: 2 KB per 64 columns) of the 16-byte chunk
// holding columns [k, k+8) of B row n.
__device__ __forceinline__ uint32_t bop_chunk(int k, int n)
{
    const int kb = k >> 6, c16 = (k >> 3) & 7;
    return static_cast<uint32_t>(kb * 2048 + (n >> 3) * 1024 + (n & 7) * 128 + ((c16 ^ (n & 7)) << 4));
}

// x -> B operand, per-group scales, Q4_K group sums, outliers.  Four lanes
// take one (batch row, group) unit, eight columns each; a warp takes 8 units
// a round.  The loads of up to kStageBatch rounds are issued together (two
// 16-byte loads a lane and round where x allows it) before any of them is
// used, so a call pays about one memory latency per kStageBatch rounds.
constexpr int kStageBatch = 4;

template <int FMT, int B>
__device__ __forceinline__ void tc_stage_x(const GemvTcArgs &a, uint8_t *sm, int cw, int lane, int g_lo, int g_hi)
{
    // the groups g_lo .. g_hi - 1 (the CTA's part of K)
    const int q4 = lane & 3;
    const int Gh = g_hi - g_lo;
    const int units = B * Gh;
    constexpr int kRound = 8 * kTcConvWarps;                 // units a round (all converter warps)
    float *stab = reinterpret_cast<float *>(sm + a.off_scale);
    float *xtab = reinterpret_cast<float *>(sm + a.off_xsum);
    float *otab = reinterpret_cast<float *>(sm + a.off_out);
    uint8_t *ftab = sm + a.off_flag;
    const bool vec = (a.K % 4 == 0) && ((reinterpret_cast<uintptr_t>(a.x) & 15u) == 0);
    for (int base0 = cw * 8; base0 < units; base0 += kStageBatch * kRound) {
        float vb[kStageBatch][8];
#pragma unroll
        for (int r = 0; r < kStageBatch; ++r) {
            const int u = base0 + r * kRound + (lane >> 2);
            const bool act = u < units;
            const int b = act ? u / Gh : 0;
            const int g = g_lo + (act ? u - b * Gh : 0);
            const int64_t c0 = 32LL * g + 8 * q4;
            const float *src = a.x + b * a.K + c0;
            if (act && vec && c0 + 8 <= a.K) {
                const float4 lo = __ldg(reinterpret_cast<const float4 *>(src));
                const float4 hi = __ldg(reinterpret_cast<const float4 *>(src) + 1);
                vb[r][0] = lo.x; vb[r][1] = lo.y; vb[r][2] = lo.z; vb[r][3] = lo.w;
                vb[r][4] = hi.x; vb[r][5] = hi.y; vb[r][6] = hi.z; vb[r][7] = hi.w;
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) vb[r][e] = (act && c0 + e < a.K) ? __ldg(src + e) : 0.f;
            }
        }
#pragma unroll
        for (int r = 0; r < kStageBatch; ++r) {
            if (base0 + r * kRound >= units) break;              // the same for the warp
            const float (&v)[8] = vb[r];
            const int u = base0 + r * kRound + (lane >> 2);
            const bool act = u < units;
            const int b = act ? u / Gh : 0;
            const int g = g_lo + (act ? u - b * Gh : 0);
            uint32_t ab[8], lmax = 0;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                ab[e] = __float_as_uint(v[e]) & 0x7FFFFFFFu;
                lmax = max(lmax, ab[e]);
            }
            uint32_t gmax = max(lmax, __shfl_xor_sync(0xFFFFFFFFu, lmax, 1));
            gmax = max(gmax, __shfl_xor_sync(0xFFFFFFFFu, gmax, 2));
            const bool nonfinite = gmax >= 0x7F800000u;
            // the batch-1 outlier rule: the only value whose exponent is within
            // 2 of the group's largest is carried exactly, off the pieces
            const int e1 = static_cast<int>(gmax >> 23);
            const uint32_t thr = e1 >= 2 ? static_cast<uint32_t>(e1 - 2) << 23 : 0u;
            int cnt = 0;
#pragma unroll
            for (int e = 0; e < 8; ++e) cnt += ab[e] >= thr ? 1 : 0;
            int gcnt = cnt + __shfl_xor_sync(0xFFFFFFFFu, cnt, 1);
            gcnt += __shfl_xor_sync(0xFFFFFFFFu, gcnt, 2);
            const bool has_out = !nonfinite && gcnt == 1;
            int oe = -1;
            if (has_out && cnt == 1) {
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    if (ab[e] >= thr) oe = e;
            }
            uint32_t lm2 = 0;
#pragma unroll
            for (int e = 0; e < 8; ++e)
                if (e != oe) lm2 = max(lm2, ab[e]);
            uint32_t gm2 = max(lm2, __shfl_xor_sync(0xFFFFFFFFu, lm2, 1));
            gm2 = max(gm2, __shfl_xor_sync(0xFFFFFFFFu, gm2, 2));
            // scale: the largest kept magnitude lands in [2^14, 2^15) (Q4_K high
            // nibbles: [2^10, 2^11)); groups below 2^-100 keep the scale of 2^-100
            int E = static_cast<int>(gm2 >> 23) - 127;
            if (E < -100) E = -100;
            const int k = 14 - E;                                  // in [-113, 114]
            const int kx = (FMT == kFmtQ4K && (g & 1)) ? k - 4 : k;
            const float f = __int_as_float((127 + kx) << 23);
            float sum = 0.f;
            uint32_t ob = 0;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                if (e != oe) sum += v[e];
                ob |= (e == oe) ? __float_as_uint(v[e]) : 0u;
            }
            sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 1);
            sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 2);
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t hp = 0, lp = 0;
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    const int e = tc_kperm<FMT>(2 * j + t);
                    const float xs = (e == oe || nonfinite) ? 0.f : v[e] * f;
                    const __half hh = __float2half_rn(xs);
                    const __half hl = __float2half_rn(xs - __half2float(hh));
                    hp |= static_cast<uint32_t>(__half_as_ushort(hh)) << (16 * t);
                    lp |= static_cast<uint32_t>(__half_as_ushort(hl)) << (16 * t);
                }
                hw[j] = hp;
                lw[j] = lp;
            }
            if (act) {
                // B rows: the hi pieces of batch row b in row b, its lo pieces in
                // row B + b (columns counted from the CTA's first staged one)
                const int kc = 32 * (g - g_lo) + 8 * q4;
                *reinterpret_cast<uint4 *>(sm + a.off_bop + bop_chunk(kc, b)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                *reinterpret_cast<uint4 *>(sm + a.off_bop + bop_chunk(kc, B + b)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                if (b == 0) {
#pragma unroll
                    for (int n = 2 * B; n < 16; ++n)
                        *reinterpret_cast<uint4 *>(sm + a.off_bop + bop_chunk(kc, n)) = make_uint4(0, 0, 0, 0);
                }
                if (q4 == 0) {
                    stab[g * 8 + b] = nonfinite ? __int_as_float(0x7FC00000) : __int_as_float((127 - k) << 23);
                    if (FMT == kFmtQ4K) xtab[g * 8 + b] = sum;
                    if (!has_out) ftab[g * 8 + b] = 0;
                }
                if (oe >= 0) {
                    // the group's one outlier: its value, and its column + 1 as the flag
                    otab[g * 8 + b] = __uint_as_float(ob);
                    ftab[g * 8 + b] = static_cast<uint8_t>(8 * q4 + oe + 1);
                }
            }
        }
    }
}

// Q4_K, one 32-byte chunk of qs (sub-block 2m in its low nibbles, 2m+1 in
// its high nibbles): exact fp16 q and 16q into tensor memory, the low
// sub-block at column col, the high one at col + 16.
__device__ __forceinline__ void q4k_tc_store_a(const uint4 &q0, const uint4 &q1, uint32_t taddr)
{
    constexpr uint32_t kOne = 0x64006400u, kMinus = 0xE400E400u;   // fp16 1024 and -1024
#pragma unroll
    for (int e = 0; e < 2; ++e) {                // low nibbles (sub-block 2m), then high (2m+1): one store each
        const uint32_t mask = e ? 0x00F000F0u : 0x000F000Fu;
        uint32_t r[16];
#pragma unroll
        for (int w8 = 0; w8 < 8; ++w8) {
            const uint4 &v = w8 < 4 ? q0 : q1;
            const uint32_t w = (w8 & 3) == 0 ? v.x : (w8 & 3) == 1 ? v.y : (w8 & 3) == 2 ? v.z : v.w;
            r[2 * w8] = hadd2_bits(lop3_and_or(w, mask, kOne), kMinus);
            r[2 * w8 + 1] = hadd2_bits(lop3_and_or(w >> 8, mask, kOne), kMinus);
        }
        tmem_st_32x32b_x16(taddr + 16u * e, r);
    }
}

// Q8_0, one block whose first byte sits PH bytes past the 16-byte boundary
// w0 of a row's 288-byte span (its first 144 bytes at sp0, the rest at sp1):
// the block's exact fp16 q (pairs) and its d.  Only the 16-byte words the
// block touches are read, so the last word ends inside the span.  Registers
// only: the tensor-memory store comes after the caller's branch on PH, with
// the warp converged.
template <int PH>
__device__ __forceinline__ void q80_tc_convert(const uint8_t *sp0, const uint8_t *sp1, int w0, uint32_t (&r)[16],
                                               float &d)
{
    constexpr int NLD = (PH + 34 + 15) / 16;
    uint32_t wx[4 * NLD];
#pragma unroll
    for (int i = 0; i < NLD; ++i) {
        const int off = w0 + 16 * i;
        const uint4 v = *reinterpret_cast<const uint4 *>(off < 144 ? sp0 + off : sp1 + (off - 144));
        wx[4 * i] = v.x ^ 0x80808080u;
        wx[4 * i + 1] = v.y ^ 0x80808080u;
        wx[4 * i + 2] = v.z ^ 0x80808080u;
        wx[4 * i + 3] = v.w ^ 0x80808080u;
    }
    constexpr uint32_t kBias = 0x64646464u, kMinus = 0xE480E480u;   // fp16 high bytes of 1024+u; -1152
    d = half_bits_to_float(((wx[PH >> 2] >> (8 * (PH & 3))) ^ 0x8080u) & 0xFFFFu);
#pragma unroll
    for (int pi = 0; pi < 16; ++pi) {
        const int bo = PH + 2 + 2 * pi;
        r[pi] = hadd2_bits(prmt(wx[bo >> 2], kBias, (bo & 3) ? 0x4342u : 0x4140u), kMinus);
    }
}

template <int FMT, int B, bool KS>
__global__ void __launch_bounds__(kTcThreads, 1) gemv_tc_kernel(const __grid_constant__ CUtensorMap tm0,
                                                                 const __grid_constant__ CUtensorMap tm1,
                                                                 const GemvTcArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    uint8_t *sm = smem_raw + (((raw_u32 + 1023u) & ~1023u) - raw_u32);
    const uint32_t sb = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + kAbort);

    // this CTA's rows (K split: the rows of its cluster); Q8_0 tiles start on
    // a row of even index (the even and odd rows come from two tensor maps,
    // 64 rows of each a tile)
    constexpr bool ks = KS;                                  // (a.ks: the plan's choice, launched as KS)
    const uint32_t rank = ks ? cluster_ctarank() : 0u;
    const int64_t nG = ks ? gridDim.x / 2 : gridDim.x;
    const int64_t gid = ks ? blockIdx.x / 2 : blockIdx.x;
    int64_t r_begin, r_end;
    if (FMT == kFmtQ80) {
        const int64_t pairs = (a.rows + 1) / 2;
        r_begin = min(a.rows, 2 * ((pairs * gid) / nG));
        r_end = min(a.rows, 2 * ((pairs * (gid + 1)) / nG));
    } else {
        r_begin = (a.rows * gid) / nG;
        r_end = (a.rows * (gid + 1)) / nG;
    }
    const int T = static_cast<int>((r_end - r_begin + kTcM - 1) / kTcM);
    const int NC = a.NC, NS = a.NS;
    // the items c_lo .. c_hi - 1 of every tile (K split: one half each)
    const int c_lo = ks && rank ? NC / 2 : 0, c_hi = ks && !rank ? NC / 2 : NC;
    const int items = T * (c_hi - c_lo);

    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(sb + kBarFull + 8u * s, 1);                  // the producer's arrival with the boxes' bytes
            mbar_init(sb + kBarEmpty + 8u * s, kTcConvWarps);
        }
        for (int p = 0; p < 2; ++p) {
            mbar_init(sb + kBarAFull + 8u * p, kTcConvWarps);
            mbar_init(sb + kBarMma + 8u * p, 1);
            mbar_init(sb + kKsFull + 8u * p, 4);                   // the odd CTA's four lane quarters
            mbar_init(sb + kKsEmpty + 8u * p, 4);                  // the even CTA's four lane quarters
        }
        for (int q = 0; q < 8; ++q) reinterpret_cast<uint32_t *>(sm + kXCount)[q] = 0u;
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kTcIssuer) {
        tmem_alloc_1(sb + kTmemSlot, kTcCols);
        tmem_relinquish_1();
    }
    tc_fence_before();
    if constexpr (ks)
        cluster_sync();      // both CTAs' barriers are initialised before either signals the other
    else
        __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(sm + kTmemSlot);
    int last_issued = -1;                                        // producer: its last item

    if (warp == kTcProducer) {
        // ------------------------------------------------------------ producer
        // item i = (tile i / NC, chunk i % NC) into stage i % NS, once the
        // converters have read the item that held the stage before.  The
        // weights do not depend on earlier kernels, so this starts at once.
        if (lane == 0) {
            tma_prefetch_desc(&tm0);
            if (FMT == kFmtQ80) tma_prefetch_desc(&tm1);
            const uint64_t pol = l2_evict_first_policy();
            const uint32_t stage0 = sb + static_cast<uint32_t>(a.off_stage);
            bool ok = true;
            int s = 0, use = 0, t = 0, c = c_lo;                 // stage and its use; tile and chunk of item i
            for (int i = 0; i < items; ++i) {
                if (use > 0 && (*abort_flag || !mbar_wait_sleep(sb + kBarEmpty + 8u * s, (use - 1) & 1, a.wait_ns))) {
                    ok = false;
                    break;
                }
                const int64_t row0 = r_begin + static_cast<int64_t>(t) * kTcM;
                const uint32_t bar = sb + kBarFull + 8u * s;
                const uint32_t dst = stage0 + static_cast<uint32_t>(s * a.stage_bytes);
                if (blockIdx.x == 0 && i == a.skip_item) {
                    // test hook: this item is never loaded, so the converters' bounded wait runs out
                } else if (FMT == kFmtQ4K) {
                    // 128 rows x one super-block (rows past the call read as zeros)
                    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(kTcM * a.chunk_bytes));
                    tma_load_2d(dst, &tm0, c * a.chunk_bytes, static_cast<int32_t>(row0), bar, pol);
                } else {
                    // rows of even and of odd index (64 each), each row's
                    // chunk as the 288 bytes from the 16-byte boundary below it
                    // (bytes past a row read as zeros)
                    const int32_t y = static_cast<int32_t>(row0 >> 1), x = 272 * c;
                    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(4 * kQ8Half));
                    tma_load_2d(dst, &tm0, x, y, bar, pol);
                    tma_load_2d(dst + kQ8Half, &tm0, x + 144, y, bar, pol);
                    tma_load_2d(dst + 2 * kQ8Half, &tm1, x, y, bar, pol);
                    tma_load_2d(dst + 3 * kQ8Half, &tm1, x + 144, y, bar, pol);
                }
                last_issued = i;
                if (++s == NS) { s = 0; ++use; }
                if (++c == c_hi) { c = c_lo; ++t; }
            }
            if (!ok) {
                *abort_flag = 1;
                record_error(a.err, kErrTimeout);
            }
            // the boxes issued land before the CTA leaves
            for (int i = max(0, last_issued - NS + 1); i <= last_issued; ++i)
                if (!(blockIdx.x == 0 && i == a.skip_item))
                    mbar_wait(sb + kBarFull + 8u * (i % NS), (i / NS) & 1, a.wait_ns);
        }
        __syncwarp();
    } else if (warp == kTcIssuer) {
        // ------------------------------------------------------------ MMA issuer
        // the whole warp runs the loop (its values stay warp-uniform); one
        // elected lane issues each MMA and the commits
        const uint32_t idesc = idesc_f16_f32(128, 16);
        // B descriptor of column k0: the 64-column block k0/64 (2 KB each)
        // and 32 bytes a 16-column step inside it (start address >> 4 in
        // the low bits)
        const uint64_t bdesc0 = smem_desc_sw128_kmajor(sb + static_cast<uint32_t>(a.off_bop));
        int last = -1;
        bool ok = true;
        int c = c_lo;                                            // chunk of item i
        for (int i = 0; i < items; ++i, c = (c + 1 == c_hi) ? c_lo : c + 1) {
            const int p = i & 1;
            bool w_ok = !*abort_flag && mbar_wait_sleep(sb + kBarAFull + 8u * p, (i >> 1) & 1, a.wait_ns);
            if (!__all_sync(0xFFFFFFFFu, w_ok)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int ng = min(8, a.G - 8 * c);
            const uint64_t bd_item = bdesc0 + static_cast<uint64_t>((c - c_lo) * (4 * 2048 / 16));
            const uint32_t d0 = tmem + 256u + 128u * p, a0 = tmem + 128u * p;
            if (elect_one()) {
#pragma unroll
                for (int gi = 0; gi < 8; ++gi) {
                    if (gi < ng) {
                        // group gi: columns 32 gi .. 32 gi + 31 of the item = block gi/2, steps 2(gi&1), +1
                        const uint64_t bd = bd_item + static_cast<uint64_t>((gi >> 1) * (2048 / 16) + (gi & 1) * 4);
                        tc_mma_f16_tmem_a(d0 + 16u * gi, a0 + 16u * gi, bd, idesc, 0);
                        tc_mma_f16_tmem_a(d0 + 16u * gi, a0 + 16u * gi + 8u, bd + 2, idesc, 1);
                    }
                }
                tc_commit_1(sb + kBarMma + 8u * p);
            }
            __syncwarp();
            last = i;
        }
        if (!ok && lane == 0) {
            *abort_flag = 1;
            record_error(a.err, kErrTimeout);
        }
        // the MMAs issued complete before the tensor memory is freed
        if (last >= 0) mbar_wait(sb + kBarMma + 8u * (last & 1), (last >> 1) & 1, a.wait_ns);
        __syncwarp();
    } else {
        // ------------------------------------------------------------ converters
        const int cw = warp - (kTcProducer + 1);
        const int h = cw >> 2;                                   // part of each item: groups kTcGPW*h ..
        const int qd = warp & 3;                                 // tensor-memory lane quarter
        const int L = 32 * qd + lane;                            // MMA row of this thread
        // tile row it holds: Q8_0 rows of one parity a warp (rows of one warp
        // then share their 16-byte phase); Q4_K rows in order
        const int rho = FMT == kFmtQ80 ? 64 * (qd >> 1) + 2 * lane + (qd & 1) : L;
        const uint32_t tl = tmem + (static_cast<uint32_t>(32 * qd) << 16);

        // x may be written by the previous kernel in the stream
        asm volatile("griddepcontrol.wait;" ::: "memory");
        tc_stage_x<FMT, B>(a, sm, cw, lane, 8 * c_lo, min(a.G, 8 * c_hi));
        fence_proxy_async_smem();                                // the B operand, for the tensor cores
        named_bar_sync(1, 32 * kTcConvWarps);                   // the tables, for every converter

        const float *stab = reinterpret_cast<const float *>(sm + a.off_scale);
        const float *xtab = reinterpret_cast<const float *>(sm + a.off_xsum);
        const float *otab = reinterpret_cast<const float *>(sm + a.off_out);
        const uint8_t *ftab = sm + a.off_flag;
        float acc[B], ocur[B], oprev[B];
        float scur[2 * kTcGPW], sprev[2 * kTcGPW];              // Q8_0: d; Q4_K: d*sc, then dmin*m
#pragma unroll
        for (int b = 0; b < B; ++b) acc[b] = ocur[b] = oprev[b] = 0.f;
#pragma unroll
        for (int j = 0; j < 2 * kTcGPW; ++j) scur[j] = sprev[j] = 0.f;
        bool failed = false;
        auto fail = [&]() {
            if (lane == 0) {
                *abort_flag = 1;
                record_error(a.err, kErrTimeout);
            }
            failed = true;
        };

        int s = 0, use = 0, t = 0, c = c_lo;                     // item i: stage and its use, tile and chunk
        int tj = 0, cj = c_lo;                                   // item i - 1: tile and chunk
        for (int i = 0; i <= items && !failed; ++i) {
            if (i < items) {
                // ---------------- convert item i into A[i & 1]
                const int p = i & 1;
                const int64_t row0 = r_begin + static_cast<int64_t>(t) * kTcM;
                const int n = static_cast<int>(min(static_cast<int64_t>(kTcM), r_end - row0));
                const bool valid = rho < n;
                // this warp's groups gi0, gi0 + 1, ... (nblk of them): kTcGPW a
                // part, or one a part when the item holds four groups or fewer
                // (a Q8_0 row's last half item), so that all parts share it
                const int ngi = min(8, a.G - 8 * c);
                const int gi0 = ngi <= 4 ? h : kTcGPW * h;
                const int nblk = ngi <= 4 ? (h < ngi ? 1 : 0) : max(0, min(kTcGPW, ngi - kTcGPW * h));
                bool ok = !*abort_flag && mbar_wait_sleep(sb + kBarFull + 8u * s, use & 1, a.wait_ns);
                ok = __all_sync(0xFFFFFFFFu, ok);
                if (!ok) {
                    fail();
                    break;
                }
                const uint8_t *stg = sm + a.off_stage + s * a.stage_bytes;
                const uint32_t acol = tl + 128u * p + static_cast<uint32_t>(16 * gi0);
#pragma unroll
                for (int b = 0; b < B; ++b) ocur[b] = 0.f;
                if constexpr (FMT == kFmtQ4K) {
                    static_assert(kTcGPW == 2, "a Q4_K converter warp takes one 32-byte qs chunk");
                    const uint8_t *slot = stg + rho * a.row_stride;
                    const uint4 hd = *reinterpret_cast<const uint4 *>(slot);
                    const uint4 q0 = *reinterpret_cast<const uint4 *>(slot + 16 + 32 * h);
                    const uint4 q1 = *reinterpret_cast<const uint4 *>(slot + 32 + 32 * h);
                    // 6-bit scales and mins of sub-blocks 2h (low nibbles) and 2h+1 (high)
                    const uint32_t sc4 = h < 2 ? (hd.y & 0x3F3F3F3Fu)
                                               : ((hd.w & 0x0F0F0F0Fu) | ((hd.y >> 2) & 0x30303030u));
                    const uint32_t m4 = h < 2 ? (hd.z & 0x3F3F3F3Fu)
                                              : (((hd.w >> 4) & 0x0F0F0F0Fu) | ((hd.z >> 2) & 0x30303030u));
                    const float d = half_bits_to_float(hd.x), dmin = half_bits_to_float(hd.x >> 16);
                    const int sh = 16 * (h & 1);                 // byte (2h) & 3 of the four
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        scur[e] = d * static_cast<float>((sc4 >> (sh + 8 * e)) & 0xFFu);
                        scur[2 + e] = dmin * static_cast<float>((m4 >> (sh + 8 * e)) & 0xFFu);
                    }
                    // outliers of this warp's groups: their exact terms, read
                    // from the stage before it is handed back
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int g = 8 * c + 2 * h + e;
                        const uint2 fl = *reinterpret_cast<const uint2 *>(ftab + 8 * g);
                        if ((fl.x | fl.y) != 0u && valid) {
#pragma unroll
                            for (int b = 0; b < B; ++b) {
                                const uint32_t fw = b < 4 ? fl.x : fl.y;
                                const int fb = static_cast<int>((fw >> (8 * (b & 3))) & 0xFFu);
                                if (fb) {
                                    const int col = fb - 1;
                                    const int qv = (slot[16 + 32 * h + col] >> (4 * e)) & 15;
                                    const float wv = fmaf(scur[e], static_cast<float>(qv), -scur[2 + e]);
                                    ocur[b] += wv * otab[g * 8 + b];
                                }
                            }
                        }
                    }
                    __syncwarp();
                    mbar_arrive_if(sb + kBarEmpty + 8u * s, lane == 0);   // the stage may be refilled
                    q4k_tc_store_a(q0, q1, acol);
                } else {
                    // this row's chunk: 288 bytes from the 16-byte boundary
                    // below it, the first 144 in box 2*par, the rest in box
                    // 2*par+1, its data o bytes in
                    const int par = rho & 1, m = rho >> 1;
                    const uint8_t *sp0 = stg + (2 * par) * kQ8Half + 144 * m;
                    const uint8_t *sp1 = sp0 + kQ8Half;
                    const int o = par ? a.ph1 : a.ph0;
                    auto at = [&](int off) { return off < 144 ? sp0 + off : sp1 + (off - 144); };
                    // outliers first (the blocks' d from the stage)
#pragma unroll
                    for (int jj = 0; jj < kTcGPW; ++jj) {
                        const int g = 8 * c + gi0 + jj;
                        if (jj < nblk) {
                            const uint2 fl = *reinterpret_cast<const uint2 *>(ftab + 8 * g);
                            if ((fl.x | fl.y) != 0u && valid) {
                                const int bo = o + 34 * (gi0 + jj);
                                const float dj = half_bits_to_float(static_cast<uint32_t>(*at(bo)) |
                                                                    (static_cast<uint32_t>(*at(bo + 1)) << 8));
#pragma unroll
                                for (int b = 0; b < B; ++b) {
                                    const uint32_t fw = b < 4 ? fl.x : fl.y;
                                    const int fb = static_cast<int>((fw >> (8 * (b & 3))) & 0xFFu);
                                    if (fb) {
                                        const int col = fb - 1;
                                        const float wv = dj * static_cast<float>(static_cast<int8_t>(*at(bo + 2 + col)));
                                        ocur[b] += wv * otab[g * 8 + b];
                                    }
                                }
                            }
                        }
                    }
                    // one block at a time (fewer registers live); the rows of a
                    // warp share one parity, so each block's phase is the same
                    // for all its lanes, and the branch holds register work and
                    // shared-memory reads only
#pragma unroll
                    for (int jj = 0; jj < kTcGPW; ++jj) {
                        float dq = 0.f;
                        uint32_t r[16];
                        if (jj < nblk) {                         // the same for the warp
                            const int bo = o + 34 * (gi0 + jj);
                            const int ph = bo & 15;
                            const int w0 = bo - ph;
                            switch (ph) {
                            case 0: q80_tc_convert<0>(sp0, sp1, w0, r, dq); break;
                            case 2: q80_tc_convert<2>(sp0, sp1, w0, r, dq); break;
                            case 4: q80_tc_convert<4>(sp0, sp1, w0, r, dq); break;
                            case 6: q80_tc_convert<6>(sp0, sp1, w0, r, dq); break;
                            case 8: q80_tc_convert<8>(sp0, sp1, w0, r, dq); break;
                            case 10: q80_tc_convert<10>(sp0, sp1, w0, r, dq); break;
                            case 12: q80_tc_convert<12>(sp0, sp1, w0, r, dq); break;
                            default: q80_tc_convert<14>(sp0, sp1, w0, r, dq); break;
                            }
                        }
                        scur[jj] = dq;
                        if (jj + 1 == kTcGPW) {
                            __syncwarp();
                            mbar_arrive_if(sb + kBarEmpty + 8u * s, lane == 0);   // the stage may be refilled
                        }
                        if (jj < nblk) tmem_st_32x32b_x16(acol + 16u * jj, r);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                mbar_arrive_if(sb + kBarAFull + 8u * p, lane == 0);      // A[p] holds item i
            }
            if (i > 0) {
                // ---------------- epilogue of item j = i - 1
                const int j = i - 1, p = j & 1;
                const int t = tj, c = cj;
                const int ngi = min(8, a.G - 8 * c);
                const int gi0 = ngi <= 4 ? h : kTcGPW * h;
                const int nblk = ngi <= 4 ? (h < ngi ? 1 : 0) : max(0, min(kTcGPW, ngi - kTcGPW * h));
                bool ok = !*abort_flag && mbar_wait_sleep(sb + kBarMma + 8u * p, (j >> 1) & 1, a.wait_ns);
                ok = __all_sync(0xFFFFFFFFu, ok);
                if (!ok) {
                    fail();
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int jj = 0; jj < kTcGPW; ++jj) {
                    if (jj < nblk) {
                        // one group at a time (fewer registers live): batch
                        // rows in pairs (f32x2), accumulator columns b (hi) and
                        // B + b (lo), per-row scales d*sc / dmin*m, per-(group,
                        // batch row) scales S and sums of x
                        uint32_t dv[16];
                        tmem_ld_32x32b_x16(tl + 256u + 128u * p + 16u * (gi0 + jj), dv);
                        tmem_ld_wait();
                        const int g = 8 * c + gi0 + jj;
                        const uint64_t dsc2 = pack2f(sprev[jj], sprev[jj]);
                        const uint64_t ndm2 = FMT == kFmtQ4K ? pack2f(-sprev[kTcGPW + jj], -sprev[kTcGPW + jj]) : 0ull;
#pragma unroll
                        for (int mm = 0; mm < B / 2; ++mm) {
                            const uint64_t hi2 = pack2(dv[2 * mm], dv[2 * mm + 1]);
                            const uint64_t lo2 = pack2(dv[B + 2 * mm], dv[B + 2 * mm + 1]);
                            const uint64_t s2 = *reinterpret_cast<const uint64_t *>(stab + 8 * g + 2 * mm);
                            uint64_t a2 = pack2f(acc[2 * mm], acc[2 * mm + 1]);
                            a2 = fma_f32x2(dsc2, mul_f32x2(add_f32x2(hi2, lo2), s2), a2);
                            if constexpr (FMT == kFmtQ4K)
                                a2 = fma_f32x2(ndm2, *reinterpret_cast<const uint64_t *>(xtab + 8 * g + 2 * mm), a2);
                            const float2 r2 = unpack2f(a2);
                            acc[2 * mm] = r2.x;
                            acc[2 * mm + 1] = r2.y;
                        }
                        if constexpr (B & 1) {
                            const float tsum = (__uint_as_float(dv[B - 1]) + __uint_as_float(dv[2 * B - 1])) *
                                               stab[8 * g + B - 1];
                            acc[B - 1] = fmaf(sprev[jj], tsum, acc[B - 1]);
                            if constexpr (FMT == kFmtQ4K)
                                acc[B - 1] = fmaf(-sprev[kTcGPW + jj], xtab[8 * g + B - 1], acc[B - 1]);
                        }
                    }
                }
                tc_fence_before();
#pragma unroll
                for (int b = 0; b < B; ++b) acc[b] += oprev[b];
                if (c == c_hi - 1) {
                    // ---------------- the tile's rows: each warp of a lane quarter
                    // leaves its partial sums; the last of the four to arrive adds
                    // them in the order h = 0..3 and stores the rows (no warp waits).
                    // A tile's arrivals all come before those of the tile two
                    // later (a warp reaches that one only after every warp has
                    // converted the item after this tile's last), so two buffers
                    // and counters by tile parity suffice; with two or more items
                    // a tile, before those of the next tile too (one buffer).
                    float *xch = reinterpret_cast<float *>(sm + a.off_xch) + (NC == 1 ? (t & 1) * (kTcCW * kTcM * B) : 0);
                    uint32_t *cnt = reinterpret_cast<uint32_t *>(sm + kXCount) + 4 * (t & 1) + qd;
                    const int64_t row0 = r_begin + static_cast<int64_t>(t) * kTcM;
                    const int n = static_cast<int>(min(static_cast<int64_t>(kTcM), r_end - row0));
#pragma unroll
                    for (int b = 0; b < B; ++b) xch[(h * kTcM + L) * B + b] = acc[b];
                    __syncwarp();
                    __threadfence_block();
                    uint32_t prev = 0;
                    if (lane == 0) prev = atomicAdd(cnt, 1u);
                    prev = __shfl_sync(0xFFFFFFFFu, prev, 0);
                    if ((prev & (kTcCW - 1)) == kTcCW - 1) {
                        __threadfence_block();
                        float yv[B];
#pragma unroll
                        for (int b = 0; b < B; ++b) {
                            float v = xch[L * B + b];
#pragma unroll
                            for (int hh = 1; hh < kTcCW; ++hh) v += xch[(hh * kTcM + L) * B + b];
                            yv[b] = v;
                        }
                        if (ks && rank) {
                            // K split, odd CTA: its row sums of the tile go to buffer
                            // t & 1 of the even CTA (once the even CTA has read the
                            // tile two before out of it)
                            const uint32_t kb = static_cast<uint32_t>(t & 1);
                            bool ok = t < 2 || mbar_wait_poll(sb + kKsEmpty + 8u * kb, ((t >> 1) - 1) & 1, a.wait_ns);
                            ok = __all_sync(0xFFFFFFFFu, ok);
                            if (!ok) {
                                fail();
                            } else {
                                const uint32_t dst = mapa_shared(
                                    sb + static_cast<uint32_t>(a.off_ksx) + ((kb * kTcM + rho) * 8u) * 4u, 0);
#pragma unroll
                                for (int b = 0; b < B; ++b)
                                    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(dst + 4u * b), "f"(yv[b])
                                                 : "memory");
                                __syncwarp();
                                if (lane == 0) {
                                    asm volatile("fence.acq_rel.cluster;" ::: "memory");
                                    mbar_arrive_remote(mapa_shared(sb + kKsFull + 8u * kb, 0));
                                }
                            }
                        } else {
                            bool ok = true;
                            if (ks) {
                                // K split, even CTA: add the odd CTA's sums of the second
                                // half of K, then free the buffer
                                const uint32_t kb = static_cast<uint32_t>(t & 1);
                                ok = mbar_wait_poll(sb + kKsFull + 8u * kb, (t >> 1) & 1, a.wait_ns);
                                ok = __all_sync(0xFFFFFFFFu, ok);
                                if (!ok) {
                                    fail();
                                } else {
                                    const float *src =
                                        reinterpret_cast<const float *>(sm + a.off_ksx) + (kb * kTcM + rho) * 8;
#pragma unroll
                                    for (int b = 0; b < B; ++b) yv[b] += src[b];
                                    __syncwarp();
                                    if (lane == 0) mbar_arrive_remote(mapa_shared(sb + kKsEmpty + 8u * kb, 1));
                                }
                            }
                            if (ok && rho < n) {
#pragma unroll
                                for (int b = 0; b < B; ++b) a.y[b * a.ldy + row0 + rho] = yv[b];
                            }
                        }
                    }
#pragma unroll
                    for (int b = 0; b < B; ++b) acc[b] = 0.f;
                }
            }
#pragma unroll
            for (int b = 0; b < B; ++b) oprev[b] = ocur[b];
#pragma unroll
            for (int jj = 0; jj < 2 * kTcGPW; ++jj) sprev[jj] = scur[jj];
            tj = t;
            cj = c;
            if (++s == NS) { s = 0; ++use; }
            if (++c == c_hi) { c = c_lo; ++t; }
        }
    }

    // every tensor-memory access of the CTA is done before it is freed (K
    // split: and neither CTA leaves while the other may still write to it)
    tc_fence_before();
    if constexpr (ks)
        cluster_sync();
    else
        __syncthreads();
    if (warp == kTcIssuer) {
        tc_fence_after();
        tmem_dealloc_1(tmem, kTcCols);
    }
}

template <int FMT, int B, bool KS>
cudaError_t gemv_tc_launch_ks(const CUtensorMap &tm0, const CUtensorMap &tm1, const GemvTcArgs &a, int grid,
                              int smem, cudaStream_t st, bool pdl)
{
    auto kern = gemv_tc_kernel<FMT, B, KS>;
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
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (KS) {
        attr[na].id = cudaLaunchAttributeClusterDimension;     // K split: CTA pairs
        attr[na].val.clusterDim.x = 2;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    e = cudaLaunchKernelEx(&cfg, kern, tm0, tm1, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int FMT, int B>
cudaError_t gemv_tc_launch_one(const CUtensorMap &tm0, const CUtensorMap &tm1, const GemvTcArgs &a, int grid,
                               int smem, cudaStream_t st, bool pdl)
{
    return a.ks ? gemv_tc_launch_ks<FMT, B, true>(tm0, tm1, a, grid, smem, st, pdl)
                : gemv_tc_launch_ks<FMT, B, false>(tm0, tm1, a, grid, smem, st, pdl);
}

template <int FMT>
cudaError_t gemv_tc_launch_fmt(int batch, const CUtensorMap &tm0, const CUtensorMap &tm1, const GemvTcArgs &a,
                               int grid, int smem, cudaStream_t st, bool pdl)
{
    switch (batch) {
    case 2: return gemv_tc_launch_one<FMT, 2>(tm0, tm1, a, grid, smem, st, pdl);
    case 3: return gemv_tc_launch_one<FMT, 3>(tm0, tm1, a, grid, smem, st, pdl);
    case 4: return gemv_tc_launch_one<FMT, 4>(tm0, tm1, a, grid, smem, st, pdl);
    case 5: return gemv_tc_launch_one<FMT, 5>(tm0, tm1, a, grid, smem, st, pdl);
    case 6: return gemv_tc_launch_one<FMT, 6>(tm0, tm1, a, grid, smem, st, pdl);
    case 7: return gemv_tc_launch_one<FMT, 7>(tm0, tm1, a, grid, smem, st, pdl);
    case 8: return gemv_tc_launch_one<FMT, 8>(tm0, tm1, a, grid, smem, st, pdl);
    default: return cudaErrorInvalidValue;
    }
}

int64_t round_up_tc(int64_t v, int64_t m) { return ((v + m - 1) / m) * m; }

}  // namespace

// Plan of the tensor-core GEMV for a device with `sms` SMs and `smem_optin`
// bytes of shared memory a block.  Whether a call takes this path depends on
// the format and K only (and the device), never on the rows: Q8_0 needs K a
// multiple of 128 (rows then start on the same 16-byte phase within each
// warp's rows, which the conversion is compiled for), and the activations'
// B operand (32 bytes a column) plus two stages must fit.
bool gemv_tc_plan_for(int fmt, int64_t rows, int64_t K, int sms, int smem_optin, GemvTcPlan *p)
{
    if (fmt != kFmtQ80 && fmt != kFmtQ4K) return false;
    if (rows <= 0 || rows > (1LL << 31) - 1 || K <= 0 || sms <= 0 || smem_optin <= 0) return false;
    if (fmt == kFmtQ80 && K % 128 != 0) return false;
    const int64_t Kp = fmt == kFmtQ4K ? round_up_tc(K, 256) : K;
    if (Kp > (1 << 16)) return false;
    const int G = static_cast<int>(Kp / 32);
    const int NC = static_cast<int>((Kp + kTcKC - 1) / kTcKC);
    const int chunk_bytes = fmt == kFmtQ4K ? 144 : 272;
    const int row_stride = 144;                                    // 16-byte units odd: conflict-free row reads
    const int stage_bytes = fmt == kFmtQ4K ? kTcM * 144 : 4 * kQ8Half;
    // K split over a cluster of two CTAs when a tile has an even number of
    // items, 8 or more: each CTA then converts half of every tile of the
    // cluster's rows and stages its half of x (the B operand holds that
    // half).  It depends on K only, so the order of a row's additions (the
    // two halves' sums, then their sum) does too.
    const int ks = (NC % 2 == 0 && NC >= 8) ? 1 : 0;
    const int64_t off_bop = kTcBarBytes;
    const int64_t off_scale = off_bop + 32 * (ks ? Kp / 2 : Kp);
    const int64_t off_xsum = off_scale + 32LL * G;
    const int64_t off_out = off_xsum + (fmt == kFmtQ4K ? 32LL * G : 0);
    const int64_t off_flag = off_out + 32LL * G;
    const int64_t off_xch = round_up_tc(off_flag + 8LL * G, 16);
    // the partial sums of a tile: 4 warps x 128 rows x up to 8 batch rows
    // (two buffers when a tile is one item)
    // (K split: the odd CTA's row sums of a tile, 2 buffers x 128 rows x 8)
    const int64_t off_ksx = round_up_tc(off_xch + (NC == 1 ? 2 : 1) * static_cast<int64_t>(kTcCW) * kTcM * 8 * 4, 16);
    const int64_t off_stage = round_up_tc(off_ksx + (ks ? 2LL * kTcM * 8 * 4 : 0), 128);
    const int64_t budget = static_cast<int64_t>(smem_optin) - 1024;   // alignment slack of the base
    int64_t ns = (budget - off_stage) / stage_bytes;
    if (ns > kTcMaxStages) ns = kTcMaxStages;
    if (ns < 2) return false;
    p->G = G;
    p->NC = NC;
    p->chunk_bytes = chunk_bytes;
    p->row_stride = row_stride;
    p->stage_bytes = stage_bytes;
    p->NS = static_cast<int>(ns);
    p->off_bop = static_cast<int>(off_bop);
    p->off_scale = static_cast<int>(off_scale);
    p->off_xsum = static_cast<int>(off_xsum);
    p->off_out = static_cast<int>(off_out);
    p->off_flag = static_cast<int>(off_flag);
    p->off_xch = static_cast<int>(off_xch);
    p->off_stage = static_cast<int>(off_stage);
    p->off_ksx = static_cast<int>(off_ksx);
    p->ks = ks;
    p->smem = static_cast<int>(off_stage + ns * stage_bytes + 1024);
    // (K split: one CTA pair for every 2 SMs, never more pairs than rows)
    p->grid = ks ? 2 * static_cast<int>(rows < sms / 2 ? rows : sms / 2) : static_cast<int>(rows < sms ? rows : sms);
    p->row_bytes = fmt == kFmtQ4K ? (Kp / 256) * 144 : (K / 32) * 34;
    return true;
}

bool gemv_tc_plan(int fmt, int64_t rows, int64_t K, GemvTcPlan *p)
{
    int sms = 0, smem = 0;
    if (!device_limits(&sms, &smem)) return false;
    return gemv_tc_plan_for(fmt, rows, K, sms, smem, p);
}

cudaError_t gemv_tc_launch(int fmt, const uint8_t *w_rows, int64_t rows, int64_t K, const float *x, int batch,
                           float *y, int64_t ldy, cudaStream_t st, const GemvTcPlan &p, int *err, uint64_t wait_ns,
                           bool pdl, int64_t skip_item)
{
    GemvTcArgs a;
    a.w = w_rows;
    a.x = x;
    a.y = y;
    a.rows = rows;
    a.K = K;
    a.ldy = ldy;
    a.row_bytes = p.row_bytes;
    a.G = p.G;
    a.NC = p.NC;
    a.skip_item = skip_item;
    a.chunk_bytes = p.chunk_bytes;
    a.row_stride = p.row_stride;
    a.stage_bytes = p.stage_bytes;
    a.NS = p.NS;
    a.off_bop = p.off_bop;
    a.off_scale = p.off_scale;
    a.off_xsum = p.off_xsum;
    a.off_out = p.off_out;
    a.off_flag = p.off_flag;
    a.off_xch = p.off_xch;
    a.off_stage = p.off_stage;
    a.ks = p.ks;
    a.off_ksx = p.off_ksx;
    a.wait_ns = wait_ns;
    a.err = err;
    // The rows come by TMA.  Q4_K: one map over the call's rows (144-byte
    // super-blocks keep them 16-byte aligned), one box of 128 rows x 144
    // bytes an item.  Q8_0 (34-byte blocks, rows of K/32*34 bytes, a multiple
    // of 8, from any 2-byte aligned start): one map over the rows of even
    // index and one over those of odd index, each with a row pitch of two
    // rows (a multiple of 16), its base at the 16-byte boundary at or below
    // its first row and its width ending at the row's last byte (what lies
    // beyond reads as zeros); boxes of 64 rows x 144 bytes, two a parity.
    gemm::EncodeTiledFn enc = gemm::encode_fn();
    if (!enc) return cudaErrorNotSupported;
    CUtensorMap tm[2];
    std::memset(tm, 0, sizeof(tm));
    a.ph0 = a.ph1 = 0;
    auto encode = [&](CUtensorMap *m, const uint8_t *base, uint64_t width, uint64_t height, uint64_t pitch,
                      uint32_t box_w, uint32_t box_h) {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(width), static_cast<cuuint64_t>(height)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(pitch)};
        const cuuint32_t box[2] = {box_w, box_h};
        const cuuint32_t estr[2] = {1, 1};
        return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    if (fmt == kFmtQ4K) {
        if (!encode(&tm[0], w_rows, p.row_bytes, rows, p.row_bytes, 144, kTcM)) return cudaErrorInvalidValue;
        tm[1] = tm[0];
        return gemv_tc_launch_fmt<kFmtQ4K>(batch, tm[0], tm[1], a, p.grid, p.smem, st, pdl);
    }
    if (fmt == kFmtQ80) {
        for (int par = 0; par < 2; ++par) {
            const uintptr_t first = reinterpret_cast<uintptr_t>(w_rows) + static_cast<uintptr_t>(par * p.row_bytes);
            const int ph = static_cast<int>(first & 15u);
            const int64_t height = par ? rows / 2 : (rows + 1) / 2;
            if (par) a.ph1 = ph; else a.ph0 = ph;
            if (height == 0) {                      // a single row: no rows of odd index
                tm[1] = tm[0];
                continue;
            }
            if (!encode(&tm[par], reinterpret_cast<const uint8_t *>(first - ph), ph + p.row_bytes, height,
                        2 * p.row_bytes, 144, kTcM / 2))
                return cudaErrorInvalidValue;
        }
        return gemv_tc_launch_fmt<kFmtQ80>(batch, tm[0], tm[1], a, p.grid, p.smem, st, pdl);
    }
    return cudaErrorInvalidValue;
}

}  // namespace qk
