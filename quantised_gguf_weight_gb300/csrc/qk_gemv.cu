// qk_gemv.cu -- launch planning and dispatch of the GEMV kernel
// (qk_gemv_kernel.cuh): team shape, K chunks, stage ring, shared-memory
// layout, grid.
#include <algorithm>
#include <cstdint>
#include <cuda_runtime.h>

#include "qk_gemv_kernel.cuh"
#include "qk_internal.h"

namespace qk {

namespace {

struct DevInfo {
    int sms = 0;
    int smem_optin = 0;
};

DevInfo dev_info()
{
    static DevInfo cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DevInfo{};
    DevInfo &di = cache[dev];
    if (di.sms == 0) {
        int sms = 0, smem = 0;
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        di.smem_optin = smem;
        di.sms = sms;
    }
    return di;
}

int64_t round_up(int64_t v, int64_t m) { return ((v + m - 1) / m) * m; }

// GEMV plan: team width SW, lane units per lane per item (cpl), K chunks,
// consumer warps, stages per warp and the shared-memory layout.
bool gemv_plan_for(int fmt, int64_t rows, int64_t K, int batch, bool pair, int64_t n_assign, const DevInfo &di,
                   GemvPlan *p)
{
    // units of x (UC columns) and of the lane work: Q8_0 blocks; Q4_K 128-column
    // halves of super-blocks, a lane taking whole super-blocks; Q6_K halves of
    // super-blocks, a lane taking one half (UB: bytes a lane unit occupies)
    const int UC = fmt == kFmtQ80 ? 32 : 128;
    const int UB = fmt == kFmtQ80 ? 34 : (fmt == kFmtQ4K ? 144 : 105);
    const int64_t row_bytes = fmt == kFmtQ80 ? ((K + 31) / 32) * 34
                                             : ((K + 255) / 256) * (fmt == kFmtQ4K ? 144 : 210);
    const int64_t U64 = (K + UC - 1) / UC;
    if (U64 > (1 << 20)) return false;
    const int U = static_cast<int>(U64);
    const int LU = fmt == kFmtQ4K ? (U + 1) / 2 : U;
    const int R = gemv_rows(fmt, batch);
    const int CM = gemv_cpl_max(fmt, batch);
    // activation unit slots (Q4_K: half super-blocks h-major, XU/2 slots a
    // half), each with B*UC/4 16-byte slots plus one padding slot
    const int XU = fmt == kFmtQ4K ? 2 * LU : U;
    const int64_t x_bytes = round_up(static_cast<int64_t>(XU) * (static_cast<int64_t>(batch) * (UC / 4) + 1) * 16, 128);
    // Q4_K: sums of x per 32 columns (every batch row); Q6_K: per 16 columns (batch 1)
    const int64_t xsum_bytes = fmt == kFmtQ4K   ? round_up(static_cast<int64_t>(batch) * 4 * XU * 4, 128)
                               : fmt == kFmtQ6K ? (batch == 1 ? round_up(static_cast<int64_t>(8) * XU * 4, 128) : 0)
                                                : 0;
    // batch 1: per 32-column group its scale, and its outlier's value and
    // column (8 bytes)
    const int64_t xscale_bytes = batch == 1 ? round_up(static_cast<int64_t>(UC / 32) * XU * 4, 128) : 0;
    const int64_t xout_bytes = batch == 1 ? round_up(static_cast<int64_t>(UC / 32) * XU * 8, 128) : 0;
    const int64_t off_x = kGemvBarBytes;
    const int64_t off_xsum = off_x + x_bytes;
    const int64_t off_xscale = off_xsum + xsum_bytes;
    const int64_t off_xout = off_xscale + xscale_bytes;
    const int64_t off_stage = off_xout + xout_bytes;
    const int64_t budget = di.smem_optin;
    if (off_stage >= budget) return false;

    int64_t grid = di.sms, cpa = 0;
    if (grid > rows) grid = rows;
    if (n_assign > 0) {
        // experts mode: each CTA takes part of one assignment's rows
        cpa = std::max<int64_t>(1, std::min<int64_t>(rows, di.sms / n_assign));
        grid = n_assign * cpa;
        if (grid > (1LL << 31) - 1) return false;
    }
    int NW = gemv_warps(fmt, batch);
    // The way a row is cut into lanes and K chunks fixes the order of its
    // additions, so it depends on K (and the format and batch) only: the
    // rows of a call get the same bits as the same rows of a larger call.
    // Most busy lanes first; among equals more units a lane, then the wider
    // team (fewer copies).  A row group split into K chunks is copied one row
    // at a time: at most 8 rows an item, and chunks of 2 KB or more are
    // preferred.
    int best_sw = 0, best_nkc = 0, best_cpl = 0;
    double best_util = -1.0;
    for (int sw = 32; sw >= 1; sw >>= 1) {
        const int cpl = std::min(CM, (LU + sw - 1) / sw);
        const int nkc = (LU + sw * cpl - 1) / (sw * cpl);
        const int rows_w = (32 / sw) * R;
        if (nkc > 1 && rows_w > 8) continue;
        if (fmt == kFmtQ6K && nkc > 1 && (sw * cpl) % 2) continue;   // chunks of whole super-blocks
        if (pair && sw == 32 && R % 2) continue;    // a gate row and its up row must share a lane or a team pair
        double util = static_cast<double>(LU) / (static_cast<double>(nkc) * sw * cpl);
        if (nkc > 1 && static_cast<int64_t>(sw) * cpl * UB < 2048) util *= 0.85;
        if (util > best_util + 1e-9 || (util > best_util - 1e-9 && cpl > best_cpl)) {
            best_util = util;
            best_sw = sw;
            best_nkc = nkc;
            best_cpl = cpl;
        }
    }
    if (best_sw == 0) return false;
    const int SW = best_sw, nkc = best_nkc, cpl = best_cpl;
    const int rows_w = (32 / SW) * R;
    const int gr = pair ? rows_w / 2 : rows_w;     // output rows per row group
    int64_t chunk_bytes = 0, row_stride = 0, stage, up_stage_off = 0;
    if (nkc == 1) {
        if (pair) {
            up_stage_off = round_up(gr * row_bytes + 32, 16);
            stage = round_up(up_stage_off + gr * row_bytes + 32, 128);
        } else {
            stage = round_up(rows_w * row_bytes + 32, 128);
        }
    } else {
        chunk_bytes = static_cast<int64_t>(SW) * cpl * UB;
        // a Q8_0 or Q6_K chunk is widened to 16-byte boundaries and its last
        // block read a few bytes past its end (whole aligned words)
        row_stride = fmt == kFmtQ4K ? chunk_bytes : round_up(chunk_bytes + 30, 16) + 16;
        stage = round_up(rows_w * row_stride, 128);
    }
    if (stage > (1 << 20)) return false;
    int64_t stages = (budget - off_stage) / stage;
    if (stages > kGemvMaxStages) stages = kGemvMaxStages;
    if (stages < 1) return false;
    // consumer warps that get row groups (all that have one) and stages per
    // warp: a warp copies an item into registers and hands its stage back
    // before the arithmetic, so one stage a warp already keeps a copy in
    // flight while the warp computes
    const int64_t rows_cta_max = n_assign > 0 ? (rows + cpa - 1) / cpa : (rows + grid - 1) / grid;
    // Batch 1: the 16-warp form (same arithmetic in the same order, more
    // warps in flight) for Q6_K, and for Q4_K when a CTA has more items than
    // the 11 consumer warps of the other form
    const bool wide = batch == 1 && (fmt == kFmtQ6K ||
                                     (fmt == kFmtQ4K && (rows_cta_max + gr - 1) / gr * nkc > NW));
    if (wide) NW = gemv_warps(fmt, batch, true);
    const int64_t ng = (rows_cta_max + gr - 1) / gr;   // row groups of the fullest CTA
    int64_t nw = std::min<int64_t>(NW, ng);
    // Split K over warps: when a CTA has fewer row groups than warps and the
    // rows are cut into K chunks, kw warps share each row group, one residue
    // class of its chunks each.  Every warp keeps one sum per lane and chunk
    // and the group's first warp adds them in chunk order, which is the
    // order of the unsplit path, so the bits do not depend on the split.
    int64_t kw = 1, part_bytes = 0;
    if (nkc > 1 && ng < NW) {
        kw = std::min<int64_t>(nkc, NW / ng);
        if (kw > 1) {
            nw = ng * kw;
            part_bytes = round_up(ng * nkc * 32 * R * batch * 4, 128);
            stages = (budget - off_stage - part_bytes) / stage;
            if (stages > kGemvMaxStages) stages = kGemvMaxStages;
            if (stages < nw) {                       // not enough stages: no split
                kw = 1;
                nw = std::min<int64_t>(NW, ng);
                part_bytes = 0;
                stages = std::min<int64_t>(kGemvMaxStages, (budget - off_stage) / stage);
            }
        }
    }
    nw = std::min(nw, stages);
    const int64_t m = stages / nw;
    stages = nw * m;
    p->U = U;
    p->XU = XU;
    p->SW = SW;
    p->R = R;
    p->stages = static_cast<int>(stages);
    p->stage_bytes = static_cast<int>(stage);
    p->off_x = static_cast<int>(off_x);
    p->off_xsum = static_cast<int>(off_xsum);
    p->off_xscale = static_cast<int>(off_xscale);
    p->off_xout = static_cast<int>(off_xout);
    p->off_part = static_cast<int>(off_stage);
    p->off_stage = static_cast<int>(off_stage + part_bytes);
    p->kw = static_cast<int>(kw);
    p->smem = static_cast<int>(off_stage + part_bytes + stages * stage);
    p->grid = static_cast<int>(grid);
    p->nw = static_cast<int>(nw);
    p->m = static_cast<int>(m);
    p->LU = LU;
    p->cpl = cpl;
    p->nkc = nkc;
    p->rows_w = rows_w;
    p->pair = pair ? 1 : 0;
    p->cpa = static_cast<int>(cpa);
    p->wide = wide ? 1 : 0;
    p->up_stage_off = static_cast<int>(up_stage_off);
    p->chunk_bytes = static_cast<int>(chunk_bytes);
    p->row_stride = static_cast<int>(row_stride);
    p->row_bytes = row_bytes;
    return true;
}

}  // namespace

bool device_limits(int *sms, int *smem_optin)
{
    const DevInfo di = dev_info();
    if (di.sms <= 0) return false;
    *sms = di.sms;
    *smem_optin = di.smem_optin;
    return true;
}

// Launch plan of a GEMV call; returns false if it cannot fit in shared memory.
bool gemv_plan(int fmt, int64_t rows, int64_t K, int batch, bool pair, GemvPlan *p, int64_t n_assign)
{
    const DevInfo di = dev_info();
    if (di.sms <= 0) return false;
    return gemv_plan_for(fmt, rows, K, batch, pair, n_assign, di, p);
}

// The plan for a device with `sms` SMs and `smem_optin` bytes of shared
// memory per block (host only: lets the planner be checked without a GPU).
bool gemv_plan_host(int fmt, int64_t rows, int64_t K, int batch, bool pair, int64_t n_assign, int sms,
                    int smem_optin, GemvPlan *p)
{
    if (sms <= 0 || smem_optin <= 0) return false;
    DevInfo di;
    di.sms = sms;
    di.smem_optin = smem_optin;
    return gemv_plan_for(fmt, rows, K, batch, pair, n_assign, di, p);
}

cudaError_t gemv_launch(int fmt, const uint8_t *w_rows, int64_t rows, int64_t K, const float *x,
                        int batch, float *y, int64_t ldy, cudaStream_t st, const GemvPlan &p,
                        int *err, uint64_t wait_ns, int64_t skip_item, bool pdl, int64_t up_rows,
                        const int32_t *expid, int64_t n_experts, int xk)
{
    if (p.R != gemv_rows(fmt, batch)) return cudaErrorInvalidValue;
    GemvArgs r;
    r.w = w_rows;
    r.x = x;
    r.y = y;
    r.rows = rows;
    r.K = K;
    r.ldy = ldy;
    r.row_bytes = p.row_bytes;
    r.U = p.U;
    r.LU = p.LU;
    r.XU = p.XU;
    r.SW = p.SW;
    r.lsw = 0;
    while ((1 << r.lsw) < p.SW) ++r.lsw;
    r.cpl = p.cpl;
    r.nkc = p.nkc;
    r.rows_w = p.rows_w;
    r.chunk_bytes = p.chunk_bytes;
    r.row_stride = p.row_stride;
    r.nw = p.nw;
    r.m = p.m;
    r.kw = p.kw;
    r.off_part = p.off_part;
    r.stage_bytes = p.stage_bytes;
    r.off_x = p.off_x;
    r.off_xsum = p.off_xsum;
    r.off_xscale = p.off_xscale;
    r.off_xout = p.off_xout;
    r.off_stage = p.off_stage;
    r.pair = p.pair;
    r.up_rows = up_rows;
    r.up_stage_off = p.up_stage_off;
    r.expid = expid;
    r.n_experts = n_experts;
    r.xk = xk;
    r.cpa = p.cpa;
    r.skip_item = skip_item;
    r.wait_ns = wait_ns;
    r.err = err;
    if (fmt == kFmtQ4K) return gemv_launch_q4k(batch, p.wide != 0, r, p.grid, p.smem, st, pdl);
    if (fmt == kFmtQ6K) return gemv_launch_q6k(batch, p.wide != 0, r, p.grid, p.smem, st, pdl);
    return gemv_launch_q80(batch, r, p.grid, p.smem, st, pdl);
}

}  // namespace qk
