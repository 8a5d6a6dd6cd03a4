// qk_gemm.cu -- prefill GEMM with GGUF Q4_K or Q8_0 weights on the tcgen05
// tensor cores (sm_103a):  Y[m][n] = sum_k bf16(x[m][k]) * bf16(w[n][k]),
// f32 accumulation, where w (Q4_K: d*sc*q - dmin*m; Q8_0: d*q) is computed in
// fp32 and rounded to bf16 (round to nearest even) in shared memory, once per
// weight.
//
// This is the prefill counterpart of the decode matvec: the chunked prefill
// multiplies a whole chunk of positions at once, so a chunk reads each weight
// only once (nurllama 0.18.1 API reference, model.nu), and the loom port runs
// prefill through GEMMs that dequantise the weight format in the kernel
// (loom-port-llm SKILL.md, "What the starter generates", gen_gemm.py).
//
// Kernel shape: a cluster of two CTAs (a CTA pair) per 256 weight rows x up
// to 512 tokens; one tcgen05.mma.cta_group::2 covers M = 256 weight rows
// (128 in each CTA's shared memory) x N = 256 tokens (128 in each CTA's
// shared memory) x K = 16, and each CTA's tensor memory accumulates its own
// 128 rows x 512 tokens (512 f32 columns).  In each CTA:
//  * warp 0 issues the TMA copies of each 64-column K chunk: the raw weight
//    bytes of its 128 rows (Q4_K: two tensor maps over the rows, the 16-byte
//    header d, dmin, scales and the chunk's 32 quant bytes; Q8_0 with 16-byte
//    row strides: the aligned 80 bytes holding the chunk's two blocks; other
//    Q8_0 rows are read by the dequantising threads themselves) and its
//    128-token slices of the bf16 activations (a tensor map with the 128-byte
//    swizzle, one box per token block);
//  * warp 1 owns the tensor memory; in the even CTA one thread issues the
//    pair's MMAs and commits (multicast to both CTAs' mbarriers), in the odd
//    CTA one thread forwards "stage ready" (its own activations landed and
//    weights dequantised) to the even CTA;
//  * warps 2-9 dequantise each chunk of the 128 rows into the K-major
//    128-byte-swizzled bf16 layout the MMA reads, then run the epilogue:
//    tcgen05.ld of 32 lanes x 32 columns into a 4 KB [token][row] tile in
//    shared memory and one TMA store (acc: an f32 add-reduce) per tile when
//    Y's rows are 16-byte aligned, else direct stores.
// Three or four stages (see Shape) synchronise through mbarriers; every wait
// is bounded, a wait that runs out aborts the CTA cleanly (copies drained,
// MMAs completed, tensor memory freed) and records the device error word,
// and both CTAs meet at a cluster barrier before the tensor memory is freed.
#include <algorithm>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "qk_device.cuh"
#include "qk_internal.h"
#include "qk_tc.cuh"

namespace qk {

namespace gemm {

constexpr int kBM = 128;                 // weight rows per CTA (half of the pair's MMA M = 256)
constexpr int kBN = 256;                 // tokens per MMA (MMA N), kBN/2 in each CTA
constexpr int kBNc = kBN / 2;            // tokens of one CTA's slice of a token block
constexpr int kBK = 64;                  // K columns per stage (one 128-byte swizzle row)
constexpr int kRawHdr = kBM * 16;       // Q4_K: the 16-byte header (d, dmin, scales) of 128 rows
constexpr int kRawChunk = kBM * 48;      // Q4_K per chunk: headers + the 32 quant bytes of 128 rows
constexpr int kQ8Box = 80;               // Q8_0 by TMA: the 16-byte-aligned 80 bytes holding a chunk's 2 blocks
constexpr int kFmtQ80T = 3;              // Q8_0 with 16-byte row strides (K a multiple of 256): weights by TMA
constexpr int kDeq = 256;                // dequantising threads: two per weight row
constexpr int kThreads = 64 + kDeq;
constexpr uint32_t kTmemCols = 512;

// Modes: Y = X W^T (store), Y += X W^T (acc), or H = silu(X Wg^T) * (X Wu^T)
// (swiglu: a CTA's 128-row weight tile holds the gate rows of 64 outputs in
// rows 0..63 and their up rows in rows 64..127).
constexpr int kStore = 0, kAcc = 1, kSwiglu = 2;

template <int FMT, int MODE>
struct Shape {
    static constexpr int halves = 2;                          // token blocks of kBN per CTA pass
    static constexpr int tiles = 1;                           // weight tiles per K chunk
    static constexpr int b_half = kBNc * kBK * 2;            // 16 KB: a CTA's slice of one token block
    static constexpr int b_stage = halves * b_half;
    static constexpr int a_tile = kBM * kBK * 2;             // 16 KB
    static constexpr int a_stage = tiles * a_tile;
    // raw weight bytes of a chunk (Q8_0 from a row stride that is not a
    // multiple of 16 bytes: none, the dequantising threads read them directly)
    static constexpr int raw_stage = FMT == kFmtQ80 ? 0 : tiles * (FMT == kFmtQ80T ? kBM * kQ8Box : kRawChunk);
    static constexpr int stages = FMT == kFmtQ80T ? 3 : 4;
    static constexpr int off_b = 0;
    static constexpr int off_a = off_b + stages * b_stage;
    static constexpr int off_raw = off_a + stages * a_stage;
    static constexpr int off_bar = off_raw + stages * raw_stage;
    static constexpr int smem = off_bar + (MODE == kSwiglu ? 512 : 256) + 1024;   // + alignment slack
};

// barrier slots (8 bytes each) after the barrier offset, four per stage kind:
// XFull (this CTA's activation copies of the stage landed), AFull (this
// CTA's dequantising warps wrote the stage's weights; they have read its raw
// bytes), Empty (the pair's MMAs of the stage completed), Peer (even CTA: the
// odd CTA's stage is complete), RFull (this CTA's raw weight bytes of the
// stage landed: Q4_K, and Q8_0 by TMA)
constexpr int kBarXFull = 0, kBarAFull = 4, kBarEmpty = 8, kBarPeer = 12, kBarAcc = 16, kBarDone = 17,
              kBarRFull = 18;
constexpr int kOffTmemSlot = 184, kOffAbort = 188;
// swiglu epilogue: per exchange pair p (0..3) the full and empty barriers of
// its two streams, slots kBarXch + 4p + {0: A full, 1: A empty, 2: B full, 3: B empty}
constexpr int kBarXch = 24;

struct Args {
    float *y;
    int64_t N, K, M, ldy;
    int row0[2];       // tensor-map row of output row 0 for the weight tile (swiglu: gate, up)
    const uint8_t *wq8[2];  // Q8_0: first byte of output row 0 of each weight tile (read directly)
    int64_t row_bytes;      // Q8_0: bytes of one weight row
    int nb;                 // Q8_0: blocks of 32 per row
    int n_tiles;            // pair tiles (2*kBM output rows; swiglu: kBM)
    int tok_pass;           // tokens a pair takes in one pass: 2*kBN, or kBN (one block)
    int nk;            // number of 64-column K chunks
    int skip_chunk;    // test hook: CTA 0 never loads the activations of this chunk (-1: none)
    int tma_y;         // 1: the output is written through the tensor map of Y (16-byte aligned rows)
    uint64_t wait_ns;
    int *err;
};

__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, uint64_t limit, volatile int *abort_flag,
                                              int *err, bool poll = false)
{
    if (*abort_flag) return false;
    if (poll ? mbar_wait_poll(bar, parity, limit) : mbar_wait(bar, parity, limit)) return true;
    *abort_flag = 1;
    record_error(err, kErrTimeout);
    return false;
}

template <int FMT, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
gemm_q4k_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_y, const Args a)
{
    constexpr bool kQ8 = FMT == kFmtQ80;        // Q8_0: weights read directly by the dequantising threads
    constexpr bool kQ8T = FMT == kFmtQ80T;      // Q8_0: weights by TMA
    using L = Shape<FMT, MODE>;
    constexpr int kHalves = L::halves, kTiles = L::tiles, kStages = L::stages;
    constexpr int kOffB = L::off_b, kOffA = L::off_a, kOffRaw = L::off_raw, kOffBar = L::off_bar;
    constexpr int kBStage = L::b_stage, kAStage = L::a_stage, kRawStage = L::raw_stage;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base_u32 = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t *base = smem_raw + (base_u32 - smem_u32(smem_raw));
    const uint32_t bar0 = base_u32 + kOffBar;
    auto bar = [&](int i) { return bar0 + 8u * i; };
    volatile int *abort_flag = reinterpret_cast<volatile int *>(base + kOffBar + kOffAbort);
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(base + kOffBar + kOffTmemSlot);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();     // 0: the CTA that issues the pair's MMAs
    const int pair = blockIdx.x >> 1;
    const int n_tile = pair % a.n_tiles;
    const int m_block = pair / a.n_tiles;
    // this CTA's first output row (swiglu: its 64 rows' gate rows, then their up rows)
    constexpr int kRowsCta = MODE == kSwiglu ? kBM / 2 : kBM;
    const int n0 = n_tile * (2 * kRowsCta) + static_cast<int>(rank) * kRowsCta;
    // (written so, the store GEMM at N = 14336 keeps the speed it had before
    // the one-block pass existed; m_block * tok_pass measured 2% slower)
    const bool one_block = a.tok_pass == kBN;
    const int m0 = m_block * (kBN * kHalves) / (one_block ? 2 : 1);
    const int nh = (kHalves == 2 && !one_block && (a.M - m0) > kBN) ? 2 : 1;   // token blocks of kBN in this pass
    const int nk = a.nk;
    // The pair takes its K chunks in the order k0, k0 + 1, ... (mod nk), k0
    // set by its weight tile: pairs running at the same time read different
    // activation chunks instead of all the same lines of L2 at once.  The
    // order depends on the output rows' 256-row block only (a swiglu pair
    // covers half of one), so the same rows give the same bits in every mode.
    const int k0 = static_cast<int>((static_cast<int64_t>(MODE == kSwiglu ? n_tile >> 1 : n_tile) * 37) % nk);
    auto phys = [&](int k) { const int p = k + k0; return p >= nk ? p - nk : p; };

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar(kBarXFull + s), 1);
            mbar_init(bar(kBarRFull + s), 1);
            mbar_init(bar(kBarAFull + s), kDeq / 32);   // one arrival per dequantising warp
            mbar_init(bar(kBarEmpty + s), 1);
            mbar_init(bar(kBarPeer + s), 1);
        }
        mbar_init(bar(kBarAcc), 1);
        mbar_init(bar(kBarDone), 1);
        if (MODE == kSwiglu)
            for (int i = 0; i < 16; ++i) mbar_init(bar(kBarXch + i), 1);
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tm_x);
        if (!kQ8) tma_prefetch_desc(&tm_w);
        if (!kQ8 && !kQ8T) tma_prefetch_desc(&tm_q);
    }
    if (warp == 1) {
        tmem_alloc_pair(base_u32 + kOffBar + kOffTmemSlot, kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();          // both CTAs' mbarriers initialised, tensor memory allocated
    tc_fence_after();
    const uint32_t taddr = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        // per chunk: this CTA's 128-token slices of the activations and, for
        // Q4_K, the headers and the chunk's 32 quant bytes of its 128 rows
        if (lane == 0) {
            const uint64_t pol_w = l2_evict_first_policy();
            const uint64_t pol_x = l2_evict_last_policy();
            auto raw_copies = [&](int kc, int s, uint32_t full) {
                // (swiglu: two boxes of 64 rows, the gate rows then the up rows)
                constexpr int kParts = MODE == kSwiglu ? 2 : 1;
                if constexpr (kQ8T) {
                    // blocks 2kc, 2kc+1 span bytes 68kc .. 68kc+67 of a row
                    for (int i = 0; i < kParts; ++i)
                        tma_load_2d(base_u32 + kOffRaw + s * kRawStage + i * (kRowsCta * kQ8Box), &tm_w,
                                    (68 * kc) & ~15, a.row0[i] + n0, full, pol_w);
                } else if constexpr (!kQ8) {
                    const int kb = kc >> 2, c = kc & 3;
                    const uint32_t raw = base_u32 + kOffRaw + s * kRawStage;
                    for (int i = 0; i < kParts; ++i) {
                        tma_load_2d(raw + i * (kRowsCta * 16), &tm_w, kb * 144, a.row0[i] + n0, full, pol_w);
                        tma_load_2d(raw + kRawHdr + i * (kRowsCta * 32), &tm_q, kb * 144 + 16 + 32 * c,
                                    a.row0[i] + n0, full, pol_w);
                    }
                }
            };
            // Two cursors.  Raw weight bytes of chunk kr go into raw slot
            // kr % kStages once the dequantising warps have read the chunk
            // kStages back (its AFull); they do not depend on the kernel
            // before this one, so the first kStages go out before the wait for
            // it.  The activations of chunk kb go into stage kb % kStages once
            // the pair's MMAs of the chunk kStages back completed (Empty).  So
            // a chunk's raw bytes are in place well before its stage frees, and
            // the dequantisation overlaps the activation copy.  No cycle: raw
            // kr needs the dequantisation of kr - kStages, which needs raw
            // kr - kStages and the MMAs of kr - 2 kStages, whose activations
            // (kb > kr - kStages) are out already.
            int kr = 0, kb = 0;
            if constexpr (L::raw_stage > 0) {
                for (; kr < nk && kr < kStages; ++kr) {
                    mbar_arrive_expect_tx(bar(kBarRFull + kr), static_cast<uint32_t>(L::raw_stage));
                    raw_copies(phys(kr), kr, bar(kBarRFull + kr));
                }
            } else {
                kr = nk;
            }
            asm volatile("griddepcontrol.wait;" ::: "memory");
            uint64_t idle_since = 0;
            while ((kb < nk || kr < nk) && !*abort_flag) {
                bool did = false;
                if (kb < nk && (kb < kStages || mbar_test(bar(kBarEmpty + kb % kStages), ((kb / kStages) - 1) & 1))) {
                    const int s = kb % kStages;
                    if (!(kb == a.skip_chunk && blockIdx.x == 0)) {
                        // both CTAs' activation copies are counted on the even
                        // CTA's XFull (the odd CTA's through the pair form of the
                        // load), so the issuer sees them without a forwarded signal
                        const uint32_t full = bar(kBarXFull + s);
                        if (rank == 0) {
                            mbar_arrive_expect_tx(full, static_cast<uint32_t>(2 * nh * L::b_half));
                            for (int h = 0; h < nh; ++h)
                                tma_load_2d(base_u32 + kOffB + s * kBStage + h * L::b_half, &tm_x, phys(kb) * kBK,
                                            m0 + h * kBN, full, pol_x);
                        } else {
                            const uint32_t full0 = mapa_shared(full, 0);
                            for (int h = 0; h < nh; ++h)
                                tma_load_2d_peer(base_u32 + kOffB + s * kBStage + h * L::b_half, &tm_x, phys(kb) * kBK,
                                                 m0 + h * kBN + kBNc, full0, pol_x);
                        }
                    }
                    ++kb;
                    did = true;
                }
                if (kr < nk && kr < kb + kStages &&
                    mbar_test(bar(kBarAFull + kr % kStages), ((kr / kStages) - 1) & 1)) {
                    const int s = kr % kStages;
                    mbar_arrive_expect_tx(bar(kBarRFull + s), static_cast<uint32_t>(L::raw_stage));
                    raw_copies(phys(kr), s, bar(kBarRFull + s));
                    ++kr;
                    did = true;
                }
                if (did) {
                    idle_since = 0;
                } else {
                    // bounded: no progress for the wait limit aborts the CTA
                    const uint64_t now = globaltimer_ns();
                    if (idle_since == 0) {
                        idle_since = now;
                    } else if (now - idle_since > a.wait_ns) {
                        *abort_flag = 1;
                        record_error(a.err, kErrTimeout);
                    }
                }
            }
            // let every copy issued land before the CTA can exit (the even
            // CTA's XFull counts the odd CTA's activation copies too, and the
            // odd CTA leaves only after the closing cluster barrier)
            if (rank == 0)
                for (int t = kb - kStages; t < kb; ++t) {
                    if (t < 0 || (t == a.skip_chunk && blockIdx.x == 0)) continue;
                    mbar_wait(bar(kBarXFull + t % kStages), (t / kStages) & 1, a.wait_ns);
                }
            if constexpr (L::raw_stage > 0)
                for (int t = kr - kStages; t < kr; ++t)
                    if (t >= 0) mbar_wait(bar(kBarRFull + t % kStages), (t / kStages) & 1, a.wait_ns);
        }
        // the other lanes wait here, blocked, until lane 0 is done: the warp
        // reaches the cluster barrier below converged, and lane 0 does not
        // share its issue slots with lanes spinning in that barrier
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            // -------------------------------------------------------- MMA issuer (even CTA)
            constexpr uint32_t idesc = idesc_bf16_f32(2 * kBM, kBN);
            bool any = false, ready = false;
            for (int kc = 0; kc < nk; ++kc) {
                const int s = kc % kStages;
                const uint32_t par = (kc / kStages) & 1;
                // polled: the issuing thread must not sleep past the phase
                if (!ready) {
                    if (!wait_or_abort(bar(kBarAFull + s), par, a.wait_ns, abort_flag, a.err, true)) break;
                    if (!wait_or_abort(bar(kBarXFull + s), par, a.wait_ns, abort_flag, a.err, true)) break;
                    if (!wait_or_abort(bar(kBarPeer + s), par, a.wait_ns, abort_flag, a.err, true)) break;
                }
                ready = false;
                tc_fence_after();
                const uint32_t a_base = base_u32 + kOffA + s * kAStage;
                const uint32_t b_base = base_u32 + kOffB + s * kBStage;
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk) {
#pragma unroll
                    for (int i = 0; i < kTiles; ++i) {
                        const uint64_t ad = smem_desc_sw128_kmajor(a_base + i * L::a_tile + 32u * kk);
                        for (int h = 0; h < nh; ++h) {
                            // accumulator columns: token block h (store/acc) or weight tile i (swiglu)
                            const uint64_t bd = smem_desc_sw128_kmajor(b_base + h * L::b_half + 32u * kk);
                            tc_mma_bf16_pair(taddr + static_cast<uint32_t>((h + i) * kBN), ad, bd, idesc,
                                             (kc | kk) != 0);
                        }
                    }
                    if (kk == 0 && kc + 1 < nk) {
                        // while this chunk's MMAs are queued: is the next stage
                        // complete already?  Then its MMAs follow without a gap
                        const int s1 = (kc + 1) % kStages;
                        const uint32_t par1 = ((kc + 1) / kStages) & 1;
                        ready = mbar_test(bar(kBarAFull + s1), par1) && mbar_test(bar(kBarXFull + s1), par1) &&
                                mbar_test(bar(kBarPeer + s1), par1);
                    }
                }
                any = true;
                tc_commit_pair(bar(kBarEmpty + s), 0x3);   // stage s reusable in both CTAs once these complete
            }
            if (!*abort_flag) tc_commit_pair(bar(kBarAcc), 0x3);
            if (any) {
                // no MMA may still read shared memory or write tensor memory
                // when the tensor memory is freed below
                tc_commit_pair(bar(kBarDone), 0x1);
                mbar_wait(bar(kBarDone), 0, a.wait_ns);
            }
        } else if (lane == 0) {
            // -------------------------------------------------------- stage-ready forwarder (odd CTA)
            // the stage's weights are written (AFull); its activation copy
            // is counted on the even CTA's XFull directly
            const uint32_t peer0 = mapa_shared(bar(kBarPeer), 0);
            for (int kc = 0; kc < nk; ++kc) {
                const int s = kc % kStages;
                if (!wait_or_abort(bar(kBarAFull + s), (kc / kStages) & 1, a.wait_ns, abort_flag, a.err, true)) break;
                mbar_arrive_remote(peer0 + 8u * s);
            }
        }
        __syncwarp();            // (as for warp 0: converged before the cluster barrier)
    } else {
        // ------------------------------------------------------------ dequantise + epilogue
        // thread -> weight row t of the tile and half `sel` of each 64-column
        // chunk: Q4_K sub-block 2c + sel (the low or the high nibbles of the
        // chunk's 32 bytes), Q8_0 block 2kc + sel
        const int t = (tid - 64) & (kBM - 1);
        const int sel = (tid - 64) >> 7;
        if constexpr (!kQ8 && !kQ8T) {
            for (int kc = 0; kc < nk; ++kc) {
                const int s = kc % kStages;
                const int c = phys(kc) & 3;
                // the chunk's raw bytes landed, and the stage's weights of
                // kStages chunks back are no longer read (their MMAs completed)
                bool ok = wait_or_abort(bar(kBarRFull + s), (kc / kStages) & 1, a.wait_ns, abort_flag, a.err);
                if (ok && kc >= kStages)
                    ok = wait_or_abort(bar(kBarEmpty + s), ((kc / kStages) - 1) & 1, a.wait_ns, abort_flag, a.err);
                if (!__all_sync(0xFFFFFFFFu, ok)) break;       // the warp goes on together or not at all
#pragma unroll
                for (int i = 0; i < kTiles; ++i) {
                    const uint8_t *raw = base + kOffRaw + s * kRawStage + i * kRawChunk;
                    const uint4 hd = *reinterpret_cast<const uint4 *>(raw + t * 16);
                    const float d = half_bits_to_float(hd.x);
                    const float dmin = half_bits_to_float(hd.x >> 16);
                    // 6-bit scale and min of sub-block j = 2c + sel
                    const int j = 2 * c + sel;
                    uint32_t scv, mv;
                    if (j < 4) {
                        scv = (hd.y >> (8 * j)) & 63u;
                        mv = (hd.z >> (8 * j)) & 63u;
                    } else {
                        const int k = j - 4;
                        scv = ((hd.w >> (8 * k)) & 15u) | (((hd.y >> (8 * k)) >> 6 & 3u) << 4);
                        mv = ((hd.w >> (8 * k + 4)) & 15u) | (((hd.z >> (8 * k)) >> 6 & 3u) << 4);
                    }
                    const float ds = d * static_cast<float>(scv), dm = dmin * static_cast<float>(mv);
                    // a nibble at bit position p (0 or 8) of a word becomes the exact
                    // float 2^23 + q 2^p (one LOP3); fma(ds 2^-p, ., -ds 2^-p 2^23) = ds q
                    // exactly, and one subtraction of dm rounds w = ds q - dm once, the
                    // same as fma(q, ds, -dm)
                    const int sh = 4 * sel;                      // nibble offset in a byte
                    const float s0 = ds, s1 = ds * (1.0f / 256.0f);  // fields at bits 0 and 8 after the shift
                    const uint64_t sc01 = pack2f(s0, s1);
                    const uint64_t of01 = pack2f(s0 * -kTwo23, s1 * -kTwo23);
                    const uint64_t ndm = pack2f(-dm, -dm);
                    const uint4 *qs = reinterpret_cast<const uint4 *>(raw + kRawHdr + t * 32);
                    const uint32_t a_row = base_u32 + kOffA + s * kAStage + i * L::a_tile + t * 128;
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {                  // bytes 16*hf .. 16*hf+15 of the sub-block
                        const uint4 qv = qs[hf];
                        const uint32_t w4[4] = {qv.x, qv.y, qv.z, qv.w};
                        uint32_t packed[8];
#pragma unroll
                        for (int wi = 0; wi < 4; ++wi) {
                            // the word's 4 nibbles (bytes 0..3, offset sh): bytes 0, 1 from the
                            // word at bits sh, sh+8; bytes 2, 3 from the word >> 16 likewise
                            const uint32_t v = w4[wi] >> sh, v2 = w4[wi] >> (16 + sh);
                            const uint64_t f01 = pack2(magic_field<0xFu>(v), magic_field<0xF00u>(v));
                            const uint64_t f23 = pack2(magic_field<0xFu>(v2), magic_field<0xF00u>(v2));
                            const float2 w01 = unpack2f(add_f32x2(fma_f32x2(f01, sc01, of01), ndm));
                            const float2 w23 = unpack2f(add_f32x2(fma_f32x2(f23, sc01, of01), ndm));
                            const __nv_bfloat162 p01 = __floats2bfloat162_rn(w01.x, w01.y);
                            const __nv_bfloat162 p23 = __floats2bfloat162_rn(w23.x, w23.y);
                            packed[2 * wi] = *reinterpret_cast<const uint32_t *>(&p01);
                            packed[2 * wi + 1] = *reinterpret_cast<const uint32_t *>(&p23);
                        }
                        // two 16-byte chunks (8 columns each) of the swizzled row
#pragma unroll
                        for (int h8 = 0; h8 < 2; ++h8) {
                            const int chunk = 4 * sel + 2 * hf + h8;            // logical 16-byte chunk 0..7
                            const uint32_t dst = a_row + ((static_cast<uint32_t>(chunk) ^ (t & 7u)) << 4);
                            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(packed[4 * h8]),
                                         "r"(packed[4 * h8 + 1]), "r"(packed[4 * h8 + 2]), "r"(packed[4 * h8 + 3])
                                         : "memory");
                        }
                    }
                }
                // every lane's stores are made visible to the tensor cores, then
                // one lane arrives for the warp
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(kBarAFull + s));
            }
        } else if constexpr (kQ8T) {
            // Q8_0 by TMA: block 2kc + sel of this thread's row sits at byte
            // (68kc & 15) + 34 sel of the row's 80-byte slot; the nine aligned
            // words around it are realigned as in the direct path
            for (int kc = 0; kc < nk; ++kc) {
                const int s = kc % kStages;
                // raw bytes landed; the stage's weights of kStages chunks back no longer read
                bool ok = wait_or_abort(bar(kBarRFull + s), (kc / kStages) & 1, a.wait_ns, abort_flag, a.err);
                if (ok && kc >= kStages)
                    ok = wait_or_abort(bar(kBarEmpty + s), ((kc / kStages) - 1) & 1, a.wait_ns, abort_flag, a.err);
                if (!__all_sync(0xFFFFFFFFu, ok)) break;       // the warp goes on together or not at all
                const uint32_t pos = static_cast<uint32_t>((68 * phys(kc)) & 15) + 34u * static_cast<uint32_t>(sel);
                const uint32_t off = pos & 3u;                  // 0 or 2
#pragma unroll
                for (int i = 0; i < kTiles; ++i) {
                    const uint32_t *wp = reinterpret_cast<const uint32_t *>(
                        base + kOffRaw + s * kRawStage + i * (kBM * kQ8Box) + t * kQ8Box + (pos & ~3u));
                    uint32_t cur[9];
#pragma unroll
                    for (int k = 0; k < 9; ++k) cur[k] = wp[k];
                    const uint32_t a_row = base_u32 + kOffA + s * kAStage + i * L::a_tile + t * 128;
                    const float d = half_bits_to_float(cur[0] >> (8 * off));
                    const uint32_t psel = off ? 0x7654u : 0x5432u;
                    uint32_t packed[16];
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        // quants 4k..4k+3 of the block (bytes 2+4k.. past its start)
                        const uint32_t v = __byte_perm(cur[k], cur[k + 1], psel);
                        const float q0 = static_cast<float>(static_cast<int8_t>(v & 0xFFu));
                        const float q1 = static_cast<float>(static_cast<int8_t>((v >> 8) & 0xFFu));
                        const float q2 = static_cast<float>(static_cast<int8_t>((v >> 16) & 0xFFu));
                        const float q3 = static_cast<float>(static_cast<int8_t>(v >> 24));
                        const __nv_bfloat162 p01 = __floats2bfloat162_rn(d * q0, d * q1);
                        const __nv_bfloat162 p23 = __floats2bfloat162_rn(d * q2, d * q3);
                        packed[2 * k] = *reinterpret_cast<const uint32_t *>(&p01);
                        packed[2 * k + 1] = *reinterpret_cast<const uint32_t *>(&p23);
                    }
#pragma unroll
                    for (int h8 = 0; h8 < 4; ++h8) {
                        const int chunk = 4 * sel + h8;                     // logical 16-byte chunk 0..7
                        const uint32_t dst = a_row + ((static_cast<uint32_t>(chunk) ^ (t & 7u)) << 4);
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(packed[4 * h8]),
                                     "r"(packed[4 * h8 + 1]), "r"(packed[4 * h8 + 2]), "r"(packed[4 * h8 + 3])
                                     : "memory");
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(kBarAFull + s));
            }
        } else {
            // Q8_0: block 2kc + sel of this thread's row of each tile (rows past N
            // repeat the last row, unstored), read as the nine aligned words
            // around the 34-byte block, one chunk ahead
            // (swiglu: rows 0..63 of the tile are gate rows, 64..127 their up rows)
            const int tr = MODE == kSwiglu ? (t & (kRowsCta - 1)) : t;
            const uint8_t *wrow = (MODE == kSwiglu && t >= kRowsCta) ? a.wq8[1] : a.wq8[0];
            const int64_t nr = min(static_cast<int64_t>(n0 + tr), a.N - 1);
            uint32_t nxt[kTiles][9], nof[kTiles];
            auto fetch = [&](int kc, uint32_t (&wv)[kTiles][9], uint32_t (&of)[kTiles]) {
                const int j = 2 * kc + sel;
#pragma unroll
                for (int i = 0; i < kTiles; ++i) {
                    if (j < a.nb) {
                        const uintptr_t ad = reinterpret_cast<uintptr_t>(wrow + nr * a.row_bytes + 34 * j);
                        const uint32_t *wp = reinterpret_cast<const uint32_t *>(ad & ~static_cast<uintptr_t>(3));
#pragma unroll
                        for (int k = 0; k < 9; ++k) wv[i][k] = __ldg(wp + k);
                        of[i] = static_cast<uint32_t>(ad & 3u);      // 0 or 2: blocks are 2-byte aligned
                    } else {
#pragma unroll
                        for (int k = 0; k < 9; ++k) wv[i][k] = 0u;
                        of[i] = 0u;
                    }
                }
            };
            fetch(phys(0), nxt, nof);
            for (int kc = 0; kc < nk; ++kc) {
                const int s = kc % kStages;
                uint32_t cur[kTiles][9], cof[kTiles];
#pragma unroll
                for (int i = 0; i < kTiles; ++i) {
                    cof[i] = nof[i];
#pragma unroll
                    for (int k = 0; k < 9; ++k) cur[i][k] = nxt[i][k];
                }
                if (kc + 1 < nk) fetch(phys(kc + 1), nxt, nof);
                // the stage's weights of kStages chunks back are no longer read
                // (their MMAs completed)
                bool ok = true;
                if (kc >= kStages)
                    ok = wait_or_abort(bar(kBarEmpty + s), ((kc / kStages) - 1) & 1, a.wait_ns, abort_flag, a.err);
                if (!__all_sync(0xFFFFFFFFu, ok)) break;       // the warp goes on together or not at all
#pragma unroll
                for (int i = 0; i < kTiles; ++i) {
                    const uint32_t a_row = base_u32 + kOffA + s * kAStage + i * L::a_tile + t * 128;
                    const uint32_t off = cof[i];
                    const float d = half_bits_to_float(cur[i][0] >> (8 * off));
                    const uint32_t psel = off ? 0x7654u : 0x5432u;
                    uint32_t packed[16];
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        // quants 4k..4k+3 of the block (bytes 2+4k.. past its start)
                        const uint32_t v = __byte_perm(cur[i][k], cur[i][k + 1], psel);
                        const float q0 = static_cast<float>(static_cast<int8_t>(v & 0xFFu));
                        const float q1 = static_cast<float>(static_cast<int8_t>((v >> 8) & 0xFFu));
                        const float q2 = static_cast<float>(static_cast<int8_t>((v >> 16) & 0xFFu));
                        const float q3 = static_cast<float>(static_cast<int8_t>(v >> 24));
                        const __nv_bfloat162 p01 = __floats2bfloat162_rn(d * q0, d * q1);
                        const __nv_bfloat162 p23 = __floats2bfloat162_rn(d * q2, d * q3);
                        packed[2 * k] = *reinterpret_cast<const uint32_t *>(&p01);
                        packed[2 * k + 1] = *reinterpret_cast<const uint32_t *>(&p23);
                    }
#pragma unroll
                    for (int h8 = 0; h8 < 4; ++h8) {
                        const int chunk = 4 * sel + h8;                     // logical 16-byte chunk 0..7
                        const uint32_t dst = a_row + ((static_cast<uint32_t>(chunk) ^ (t & 7u)) << 4);
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(packed[4 * h8]),
                                     "r"(packed[4 * h8 + 1]), "r"(packed[4 * h8 + 2]), "r"(packed[4 * h8 + 3])
                                     : "memory");
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(kBarAFull + s));
            }
        }
        // epilogue: tensor memory -> registers -> Y (store, acc) or H (swiglu)
        // warp-uniform: tcgen05.ld below is a whole-warp instruction
        if (__all_sync(0xFFFFFFFFu, wait_or_abort(bar(kBarAcc), 0, a.wait_ns, abort_flag, a.err))) {
            tc_fence_after();
            // warp w may read TMEM lanes 32*(w%4) ..; the two warps of each lane
            // quarter take one half of the accumulator columns each
            const int q = warp & 3;
            const uint32_t lane_base = taddr + (static_cast<uint32_t>(32 * q) << 16);
            const int cols = nh * kBN;
            const int part = (warp - 2) >> 2;
            const int n = n0 + 32 * q + lane;             // store, acc: this lane's output row
            if constexpr (MODE == kSwiglu) {
                // The gate rows of outputs n0 + 32 fq .. n0 + 32 fq + 31 sit in
                // lane quarter fq, their up rows in quarter fq + 2.  The two
                // warps of a part and an fq swap alternate 32-token chunks through
                // shared memory (the up warp sends the even chunks on stream A,
                // the gate warp the odd ones on stream B, one 4 KB buffer each
                // with a full and an empty barrier), and each warp finishes the
                // chunks it receives: silu(g) * u, stored.
                const int fq = q & 1;
                const bool upw = q >= 2;
                const int px = 2 * part + fq;
                const uint32_t xbuf = base_u32 + 65536u + static_cast<uint32_t>(px) * 8192u;   // A, then B
                const uint32_t xbar = bar(kBarXch + 4 * px);    // A full, A empty, B full, B empty
                const int nsw = n0 + 32 * fq + lane;            // this lane's output row
                const int jbeg = part * (cols / 2);
                const uint32_t buf0 = base_u32 + static_cast<uint32_t>(warp - 2) * 8192u;   // as below
                int nv = 0;                                     // chunks of this part with tokens below M
                if (n0 + 32 * fq < a.N)
                    for (int j0 = jbeg; j0 < jbeg + cols / 2 && m0 + j0 < a.M; j0 += 32) ++nv;
                uint32_t nb = 0;
                for (int c2 = 0; c2 < nv; c2 += 2) {
                    const uint32_t ph = static_cast<uint32_t>(c2 >> 1);
                    const int cs = upw ? c2 : c2 + 1;           // the chunk this warp sends
                    if (cs < nv) {
                        const uint32_t sfull = xbar + (upw ? 0u : 16u), sbuf = xbuf + (upw ? 0u : 4096u);
                        bool ok = true;
                        if (ph > 0) ok = wait_or_abort(sfull + 8u, (ph - 1) & 1u, a.wait_ns, abort_flag, a.err);
                        if (!__all_sync(0xFFFFFFFFu, ok)) break;
                        uint32_t v[32];
                        tmem_ld_32x32b_x32(lane_base + static_cast<uint32_t>(jbeg + 32 * cs), v);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            asm volatile("st.shared.b32 [%0], %1;" ::"r"(sbuf + static_cast<uint32_t>(i * 32 + lane) * 4u),
                                         "r"(v[i])
                                         : "memory");
                        __syncwarp();
                        if (lane == 0) mbar_arrive(sfull);
                    }
                    const int cr = upw ? c2 + 1 : c2;           // the chunk this warp finishes
                    if (cr < nv) {
                        const uint32_t rfull = xbar + (upw ? 16u : 0u), rbuf = xbuf + (upw ? 4096u : 0u);
                        const bool ok = wait_or_abort(rfull, ph & 1u, a.wait_ns, abort_flag, a.err);
                        if (!__all_sync(0xFFFFFFFFu, ok)) break;
                        uint32_t v[32], o[32];
                        tmem_ld_32x32b_x32(lane_base + static_cast<uint32_t>(jbeg + 32 * cr), v);
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            asm volatile("ld.shared.b32 %0, [%1];"
                                         : "=r"(o[i])
                                         : "r"(rbuf + static_cast<uint32_t>(i * 32 + lane) * 4u)
                                         : "memory");
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const float g = __uint_as_float(upw ? o[i] : v[i]);
                            const float u = __uint_as_float(upw ? v[i] : o[i]);
                            v[i] = __float_as_uint(silu(g) * u);
                        }
                        __syncwarp();
                        if (lane == 0) mbar_arrive(rfull + 8u);   // the buffer may be refilled
                        const int j0 = jbeg + 32 * cr;
                        if (a.tma_y) {
                            if (lane == 0) bulk_wait_group_read<1>();   // this tile's buffer is read out
                            __syncwarp();
                            const uint32_t buf = buf0 + nb * 4096u;
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                asm volatile("st.shared.b32 [%0], %1;" ::"r"(buf + static_cast<uint32_t>(i * 32 + lane) * 4u),
                                             "r"(v[i])
                                             : "memory");
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                tma_store_2d<false>(&tm_y, buf, n0 + 32 * fq, m0 + j0);
                                bulk_commit_group();
                            }
                            nb ^= 1u;
                        } else if (nsw < a.N) {
                            // rows not 16-byte aligned: direct stores
#pragma unroll
                            for (int i = 0; i < 32; ++i) {
                                const int64_t m = m0 + j0 + i;
                                if (m < a.M) a.y[m * a.ldy + nsw] = __uint_as_float(v[i]);
                            }
                        }
                    }
                }
                if (a.tma_y && lane == 0) bulk_wait_group_all();
            } else if (a.tma_y) {
                // each 32 rows x 32 tokens go through a 4 KB shared-memory tile
                // ([token][row], two per warp, the stages' space is free now)
                // and one TMA store (acc: f32 add-reduce) of the tile
                const uint32_t buf0 = base_u32 + static_cast<uint32_t>(warp - 2) * 8192u;
                const bool rows_in = n0 + 32 * q < a.N;
                uint32_t nb = 0;
                for (int j0 = part * (cols / 2); j0 < (part + 1) * (cols / 2); j0 += 32) {
                    if (!rows_in || m0 + j0 >= a.M) break;        // warp-uniform
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(lane_base + static_cast<uint32_t>(j0), v);
                    tmem_ld_wait();
                    if (lane == 0) bulk_wait_group_read<1>();     // this tile's buffer is read out
                    __syncwarp();
                    const uint32_t buf = buf0 + nb * 4096u;
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        asm volatile("st.shared.b32 [%0], %1;" ::"r"(buf + static_cast<uint32_t>(i * 32 + lane) * 4u),
                                     "r"(v[i])
                                     : "memory");
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d<MODE == kAcc>(&tm_y, buf, n0 + 32 * q, m0 + j0);
                        bulk_commit_group();
                    }
                    nb ^= 1u;
                }
                if (lane == 0) bulk_wait_group_all();
            } else {
                // rows not 16-byte aligned: direct stores, one token of 32 rows
                // a warp instruction
                for (int j0 = part * (cols / 2); j0 < (part + 1) * (cols / 2); j0 += 32) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(lane_base + static_cast<uint32_t>(j0), v);
                    tmem_ld_wait();
                    if (n < a.N) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const int64_t m = m0 + j0 + i;
                            if (m < a.M) {
                                float *yp = a.y + m * a.ldy + n;
                                *yp = MODE == kAcc ? *yp + __uint_as_float(v[i]) : __uint_as_float(v[i]);
                            }
                        }
                    }
                }
            }
        }
    }
    tc_fence_before();
    cluster_sync();          // no CTA of the pair leaves while the other may still use its memory
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(taddr, kTmemCols);
    }
}

// X fp32 [M][K] -> Xb bf16 [M][K8], round to nearest even; columns K..K8-1 zero.
__global__ void x_to_bf16_kernel(const float *__restrict__ x, __nv_bfloat16 *__restrict__ xb, int64_t M, int64_t K,
                                 int64_t K8)
{
    // the GEMM launched after it may start its prologue and weight copies now
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t total = M * K8;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t m = i / K8, k = i - m * K8;
        xb[i] = k < K ? __float2bfloat16_rn(x[m * K + k]) : __float2bfloat16_rn(0.0f);
    }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

}  // namespace gemm

int64_t gemm_k8(int64_t K) { return (K + 7) / 8 * 8; }

size_t gemm_workspace_bytes(int64_t M, int64_t K) { return static_cast<size_t>(M * gemm_k8(K) * 2 + 256); }

namespace {

template <int FMT, int MODE>
cudaError_t launch_mode(const CUtensorMap &tm_x, const CUtensorMap &tm_w, const CUtensorMap &tm_q,
                        const CUtensorMap &tm_y, const gemm::Args &a, int64_t grid, cudaStream_t st)
{
    using namespace gemm;
    constexpr int smem = Shape<FMT, MODE>::smem;
    static int granted[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && granted[dev] == 0) {
        e = cudaFuncSetAttribute(gemm_q4k_kernel<FMT, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        granted[dev] = 1;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;     // CTA pairs
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // programmatic dependent launch after the x -> bf16 pre-pass: only the
    // activation copies wait for it (griddepcontrol.wait in the producer)
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, gemm_q4k_kernel<FMT, MODE>, tm_x, tm_w, tm_q, tm_y, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

cudaError_t gemm_launch(int fmt, const uint8_t *w_rows, int64_t N, int64_t K, const float *x, int64_t M, float *y,
                        int64_t ldy, void *workspace, cudaStream_t st, int *err, uint64_t wait_ns, int skip_chunk,
                        bool *encode_failed, int mode, int64_t up_rows)
{
    using namespace gemm;
    *encode_failed = false;
    const bool q8 = fmt == kFmtQ80;
    const int64_t K8 = gemm_k8(K);
    const int64_t row_bytes = q8 ? ((K + 31) / 32) * 34 : ((K + 255) / 256) * 144;
    __nv_bfloat16 *xb = static_cast<__nv_bfloat16 *>(workspace);
    {
        const int64_t total = M * K8;
        int64_t blocks = (total + 255) / 256;
        if (blocks > 4096) blocks = 4096;
        x_to_bf16_kernel<<<static_cast<int>(blocks), 256, 0, st>>>(x, xb, M, K, K8);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    EncodeTiledFn enc = encode_fn();
    if (!enc) {
        *encode_failed = true;
        return cudaErrorNotSupported;
    }
    CUtensorMap tm_x, tm_w;
    {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K8), static_cast<cuuint64_t>(M)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K8 * 2)};
        const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(kBNc)};
        const cuuint32_t estr[2] = {1, 1};
        if (enc(&tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, xb, dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
            *encode_failed = true;
            return cudaErrorInvalidValue;
        }
    }
    // the weight map spans the rows of every tile: [0, N) and, for swiglu,
    // the up rows [up_rows, up_rows + N) relative to w_rows
    const int64_t lo = mode == kSwiglu ? std::min<int64_t>(0, up_rows) : 0;
    const int64_t hi = mode == kSwiglu ? std::max<int64_t>(N, up_rows + N) : N;
    // two maps over the Q4_K rows: the 16-byte headers and the 32 quant
    // bytes of one 64-column chunk, 128 rows a box (swiglu: 64, the gate
    // and the up rows of a tile come as two boxes; x offsets are multiples
    // of 16 bytes: 144 kb and 144 kb + 16 + 32 c)
    const int box_rows = mode == kSwiglu ? kBM / 2 : kBM;
    CUtensorMap tm_q;
    // Q8_0 rows of a multiple of 16 bytes (K a multiple of 256) from a
    // 16-byte aligned tensor come by TMA, 128 rows (swiglu: 64) x 80 bytes a
    // box; other Q8_0 rows are read directly
    const bool q8_tma = q8 && row_bytes % 16 == 0 && (reinterpret_cast<uintptr_t>(w_rows + lo * row_bytes) & 15u) == 0;
    if (q8_tma) {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(hi - lo)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
        const cuuint32_t estr[2] = {1, 1};
        const cuuint32_t box[2] = {static_cast<cuuint32_t>(kQ8Box), static_cast<cuuint32_t>(box_rows)};
        if (enc(&tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(w_rows + lo * row_bytes), dims, strides,
                box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
            *encode_failed = true;
            return cudaErrorInvalidValue;
        }
        tm_q = tm_x;
    } else if (q8) {
        tm_w = tm_x;       // Q8_0 weights are read directly: the maps are not used
        tm_q = tm_x;
    } else {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(hi - lo)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
        const cuuint32_t estr[2] = {1, 1};
        for (int m = 0; m < 2; ++m) {
            const cuuint32_t box[2] = {m ? 32u : 16u, static_cast<cuuint32_t>(box_rows)};
            if (enc(m ? &tm_q : &tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(w_rows + lo * row_bytes),
                    dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
                *encode_failed = true;
                return cudaErrorInvalidValue;
            }
        }
    }
    // the output through a tensor map of 32 x 32 boxes when its rows allow
    // (16-byte aligned base and row stride); else the kernel stores directly
    CUtensorMap tm_y = tm_x;
    bool tma_y = false;
    if ((reinterpret_cast<uintptr_t>(y) & 15u) == 0 && (ldy % 4) == 0) {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ldy) * 4u};
        const cuuint32_t box[2] = {32u, 32u};
        const cuuint32_t estr[2] = {1, 1};
        tma_y = enc(&tm_y, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, y, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
        if (!tma_y) tm_y = tm_x;
    }
    Args a;
    a.tma_y = tma_y ? 1 : 0;
    a.y = y;
    a.N = N;
    a.K = K;
    a.M = M;
    a.ldy = ldy;
    a.row0[0] = static_cast<int>(-lo);
    a.row0[1] = static_cast<int>(up_rows - lo);
    a.wq8[0] = w_rows;
    a.wq8[1] = w_rows + up_rows * row_bytes;
    a.row_bytes = row_bytes;
    a.nb = static_cast<int>((K + 31) / 32);
    const int64_t rows_pair = mode == kSwiglu ? kBM : 2 * kBM;   // output rows of a CTA pair
    a.n_tiles = static_cast<int>((N + rows_pair - 1) / rows_pair);
    a.nk = static_cast<int>((K8 + kBK - 1) / kBK);
    a.skip_chunk = skip_chunk;
    a.wait_ns = wait_ns;
    a.err = err;
    // Tokens a pair takes in one pass: 2 kBN; or one block of kBN when the
    // weight tiles are few, so that twice the pairs (each tile's weights
    // dequantised once per token block) still run at once, one pair to two
    // SMs.  Every output sums its K chunks in the same order either way.
    int sms = 0, smem_optin = 0;
    const bool have_sms = device_limits(&sms, &smem_optin);
    const int64_t m_half = (M + kBN - 1) / kBN;
    a.tok_pass = (have_sms && M > kBN && a.n_tiles * m_half <= sms / 2) ? kBN : 2 * kBN;
    const int64_t m_blocks = (M + a.tok_pass - 1) / a.tok_pass;
    const int64_t grid = 2 * a.n_tiles * m_blocks;          // CTA pairs
    if (q8_tma) {
        if (mode == kSwiglu) return launch_mode<kFmtQ80T, kSwiglu>(tm_x, tm_w, tm_q, tm_y, a, grid, st);
        if (mode == kAcc) return launch_mode<kFmtQ80T, kAcc>(tm_x, tm_w, tm_q, tm_y, a, grid, st);
        return launch_mode<kFmtQ80T, kStore>(tm_x, tm_w, tm_q, tm_y, a, grid, st);
    }
    if (q8) {
        if (mode == kSwiglu) return launch_mode<kFmtQ80, kSwiglu>(tm_x, tm_w, tm_q, tm_y, a, grid, st);
        if (mode == kAcc) return launch_mode<kFmtQ80, kAcc>(tm_x, tm_w, tm_q, tm_y, a, grid, st);
        return launch_mode<kFmtQ80, kStore>(tm_x, tm_w, tm_q, tm_y, a, grid, st);
    }
    if (mode == kSwiglu) return launch_mode<kFmtQ4K, kSwiglu>(tm_x, tm_w, tm_q, tm_y, a, grid, st);
    if (mode == kAcc) return launch_mode<kFmtQ4K, kAcc>(tm_x, tm_w, tm_q, tm_y, a, grid, st);
    return launch_mode<kFmtQ4K, kStore>(tm_x, tm_w, tm_q, tm_y, a, grid, st);
}

cudaError_t gemm_q4k_launch(const uint8_t *w_rows, int64_t N, int64_t K, const float *x, int64_t M, float *y,
                            int64_t ldy, void *workspace, cudaStream_t st, int *err, uint64_t wait_ns, int skip_chunk,
                            bool *encode_failed)
{
    return gemm_launch(kFmtQ4K, w_rows, N, K, x, M, y, ldy, workspace, st, err, wait_ns, skip_chunk, encode_failed);
}

}  // namespace qk
