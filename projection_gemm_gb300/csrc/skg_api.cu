// skg_api.cu -- host side of the C ABI declared in include/skg.h.
//
// Plans, the kernel picker, argument checks, the split-K workspace, TMA
// descriptor encoding and kernel launches.  No computation of the projection
// happens on the host; a request the kernels cannot serve is rejected with a
// status, never rerouted.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>

#include "skg.h"
#include "skg_internal.h"

using namespace skg;

namespace {

thread_local std::string g_last_error;

skg_status fail(skg_status st, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

skg_status cuda_fail(cudaError_t e, const char *what)
{
    return fail(SKG_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// ------------------------------------------------------------ picker table
struct TableRow {
    int kind, M, N, K, epi, split, stages, grid, burst, ahead, reducers;
};

const TableRow kTable[] = {
#include "skg_plan_table.inc"
    {0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0}  // sentinel
};

bool is_pow2(int v) { return v > 0 && (v & (v - 1)) == 0; }

int gemv_rows_per_group(int split) { return (kGemvThreads / 32) / split; }

// Ring depth for the M <= 2 kernel: the deepest ring (<= 9 slots) with which
// two CTAs share an SM, else one CTA; 0 if even a 2-slot ring does not fit.
int gemv_default_ring(int M, int K, int split, int *ctas)
{
    for (int c = 2; c >= 1; --c) {
        const int budget = 233472 / c - 1024;   // 228 KB per SM, 1 KB reserved per CTA
        int r = 9;
        while (r >= 3 && gemv_smem_bytes(M, K, split, r) > std::min(budget, kGemvMaxSmem))
            --r;
        if (r >= 3) {
            *ctas = c;
            return r;
        }
    }
    *ctas = 1;
    return gemv_smem_bytes(M, K, split, 2) <= kGemvMaxSmem ? 2 : 0;
}

void fill_gemv(skg_plan_desc *d, int split, int ring, int grid, int num_sms)
{
    const int want_batch = d->tma_burst;          // bulk-copy form: strips per copy asked for
    d->kernel_kind = SKG_KERNEL_GEMV;
    d->split_k = split;
    d->m_pad = d->M;
    d->workspace_bytes = 0;
    d->tma_burst = 0;
    d->threads = kGemvThreads;
    if (split == 1 && ring == 3) {
        // one balanced wave: CTAs own row runs, warps equal runs of chunks
        const int batch = want_batch == 4 || want_batch == 8 ? want_batch : gemv_bulk_default_batch(d->M, d->K);
        d->split_k = 1;
        d->stages = 3;
        d->tma_burst = batch;
        d->threads = kGemvThreads;
        d->grid = grid > 0 ? std::min(grid, d->N) : gemv_span_grid(d->M, d->N, d->K, batch, num_sms);
        d->tile_n = (d->N + d->grid - 1) / d->grid;
        d->smem_bytes = gemv_span_smem_bytes(d->M, d->K, batch, d->tile_n);
        return;
    }
    if (split == 1 && ring >= 2) {
        // the whole-row kernel with its weight batches moved by the copy
        // engine; tma_burst = strips per bulk copy
        const int batch = want_batch == 4 || want_batch == 8 ? want_batch : gemv_bulk_default_batch(d->M, d->K);
        fill_gemv(d, 1, 0, grid, num_sms);
        d->stages = 2;
        d->tma_burst = batch;
        d->smem_bytes = gemv_bulk_smem_bytes(d->M, d->K, batch);
        return;
    }
    if (split == 1) {
        // whole rows per warp: tile_n = rows per CTA = 8 warps x rows per warp
        const int warps = kGemvThreads / 32;
        int rpw = 1;
        if (grid > 0)
            rpw = std::max(1, (d->N + warps * grid - 1) / (warps * grid));
        d->tile_n = warps * rpw;
        d->stages = 0;
        d->smem_bytes = gemv_smem_bytes(d->M, d->K, 1, 0);
        d->grid = (d->N + d->tile_n - 1) / d->tile_n;
        return;
    }
    d->tile_n = gemv_rows_per_group(split);
    int ctas = 1;
    const int r0 = gemv_default_ring(d->M, d->K, split, &ctas);
    d->stages = ring > 0 ? ring : r0;
    d->tma_burst = 0;
    d->threads = kGemvThreads;
    d->smem_bytes = gemv_smem_bytes(d->M, d->K, split, d->stages);
    const int groups = (d->N + d->tile_n - 1) / d->tile_n;
    if (grid <= 0)
        grid = std::max(1, num_sms) * ctas;
    d->grid = std::min(grid, groups);
    d->workspace_bytes = 0;
}

void fill_tc(skg_plan_desc *d, int split, int stages, int burst)
{
    d->kernel_kind = SKG_KERNEL_SPLITK_TC;
    d->split_k = split;
    d->tile_n = kTileN;
    d->m_pad = (d->M + 15) / 16 * 16;
    const int smax = tc_max_stages(d->m_pad, 232448);
    d->stages = stages <= 0 ? std::min(kTcDefaultStages, smax) : std::max(2, std::min(stages, smax));
    d->threads = kTcThreads;
    d->smem_bytes = tc_smem_bytes(d->m_pad, d->stages);
    d->tma_burst = std::max(1, std::min(burst, d->stages));
    const int n_tiles = (d->N + kTileN - 1) / kTileN;
    d->grid = n_tiles * split;
    d->workspace_bytes = tc_partial_bytes(d->M, d->N, split) + static_cast<size_t>(n_tiles) * sizeof(unsigned int);
}

const TableRow *table_lookup(int kind, int M, int N, int K, int epi)
{
    const TableRow *best = nullptr;
    double best_d = 1e30;
    for (const TableRow *r = kTable; r->kind != 0; ++r) {
        if (r->kind != kind || r->N != N || r->K != K || r->epi != epi)
            continue;
        const double dist = std::fabs(std::log2(static_cast<double>(r->M)) - std::log2(static_cast<double>(M)));
        if (dist < best_d) {
            best_d = dist;
            best = r;
        }
    }
    return best;
}

// A GEMV plan with warps sharing rows (split > 1) runs one wave of the CTAs
// the SMs hold at its ring depth, unless its table row fixes the grid: the
// host-only query can only estimate that occupancy, the plan measures it.
bool gemv_grid_from_occupancy(const skg_plan_desc &d)
{
    if (d.kernel_kind != SKG_KERNEL_GEMV || d.split_k <= 1)
        return false;
    if (!d.from_table)
        return true;
    const TableRow *row = table_lookup(SKG_KERNEL_GEMV, d.M, d.N, d.K, d.epilogue);
    return !row || row->grid <= 0;
}

bool table_has_exact(int kind, int M, int N, int K, int epi)
{
    for (const TableRow *r = kTable; r->kind != 0; ++r)
        if (r->kind == kind && r->M == M && r->N == N && r->K == K && r->epi == epi)
            return true;
    return false;
}

// Reducers per tile where neither the table nor the caller sets them,
// measured on GB300: from M = 16 four reducers beat one wherever a tile's
// split is 4 or 8 and the tiles are few (<= 56); with more tiles, or
// shorter splits, the waits cost more than the shorter reduction saves.
int default_reducers(int M, int split, int n_tiles)
{
    return (M >= 16 && split >= 4 && n_tiles <= 56) ? 4 : 1;
}

// force_kind 0: the picker chooses the kernel kind.
skg_status query(int M, int N, int K, int epi, int num_sms, size_t l2_bytes, skg_plan_desc *d,
                 int force_kind = 0)
{
    if (!d)
        return fail(SKG_ERR_INVALID_ARG, "skg_plan_query: out is NULL");
    std::memset(d, 0, sizeof *d);
    if (M < 1 || M > 64)
        return fail(SKG_ERR_UNSUPPORTED, "M=%d outside 1..64 (decode batch)", M);
    if (N < 1)
        return fail(SKG_ERR_INVALID_ARG, "N=%d must be >= 1", N);
    if (K < 8 || K % 8 != 0)
        return fail(SKG_ERR_UNSUPPORTED, "K=%d must be a positive multiple of 8 (16-byte rows)", K);
    if (epi != SKG_EPI_BF16 && epi != SKG_EPI_BF16_RESIDUAL && epi != SKG_EPI_FP32)
        return fail(SKG_ERR_INVALID_ARG, "unknown epilogue %d", epi);
    if (static_cast<long long>(M) * N >= (1ll << 31) || static_cast<long long>(N) * K >= (1ll << 40))
        return fail(SKG_ERR_UNSUPPORTED, "problem too large");
    if (num_sms < 1)
        num_sms = 1;
    d->M = M;
    d->N = N;
    d->K = K;
    d->epilogue = epi;
    d->pdl = 1;
    const size_t wbytes = static_cast<size_t>(N) * K * 2;
    d->prefetch_bytes = std::min(wbytes, static_cast<size_t>(0.5 * static_cast<double>(l2_bytes))) & ~static_cast<size_t>(15);

    // [TS]: the kernel kind follows the batch size -- except where the
    // measured table holds a tensor-core row for exactly this M <= 2 shape
    // (the tuner writes one only where that kernel beat every GEMV form).
    int kind = (M <= 2) ? SKG_KERNEL_GEMV : SKG_KERNEL_SPLITK_TC;
    if (force_kind != 0) {
        if (force_kind != SKG_KERNEL_GEMV && force_kind != SKG_KERNEL_SPLITK_TC)
            return fail(SKG_ERR_INVALID_ARG, "unknown kernel kind %d", force_kind);
        if (force_kind == SKG_KERNEL_GEMV && M > 2)
            return fail(SKG_ERR_UNSUPPORTED, "the GEMV kernel takes M <= 2 (M=%d)", M);
        kind = force_kind;
    } else if (M <= 2 && table_has_exact(SKG_KERNEL_SPLITK_TC, M, N, K, epi)) {
        kind = SKG_KERNEL_SPLITK_TC;
    } else if (M <= 2 && gemv_smem_bytes(M, K, 1, 0) > kGemvMaxSmem) {
        kind = SKG_KERNEL_SPLITK_TC;   // x does not fit the GEMV's shared memory: the split-K kernel streams it
    } else if (M == 2 && N >= 2048 && !table_has_exact(SKG_KERNEL_GEMV, M, N, K, epi)) {
        // measured on GB300 (9 shapes outside the table, N = 2048-28672):
        // at two tokens the split-K kernel beats every GEMV form by 0-35%
        kind = SKG_KERNEL_SPLITK_TC;
    }
    if (kind == SKG_KERNEL_GEMV && gemv_smem_bytes(M, K, 1, 0) > kGemvMaxSmem)
        return fail(SKG_ERR_UNSUPPORTED, "K=%d too large for the M<=2 kernel (x is staged in shared memory)", K);
    const TableRow *row = table_lookup(kind, M, N, K, epi);
    if (kind == SKG_KERNEL_GEMV) {
        int split, grid = 0, ring = 0;
        if (row) {
            split = row->split;
            grid = row->grid;
            ring = row->stages;
            d->tma_burst = row->burst;   // split 1 with bulk-copied batches: strips per copy
            d->l2_ahead = row->ahead;
            d->from_table = 1;
        } else if (N >= 1024) {
            split = 1;   // enough rows for one warp per row
            // measured: bulk-copied batches beat 16-byte loads at M = 1 and 2;
            // at M = 1 one balanced wave beats whole rows per warp where rows
            // are long (K >= 5120) and not too many (N < 16384), whole rows
            // per warp elsewhere (up to 1.4x at K <= 4096)
            if (gemv_bulk_ok(M, K, gemv_bulk_default_batch(M, K)))
                ring = (M == 1 && K >= 5120 && N < 16384) ? 3 : 2;
            else
                d->l2_ahead = 1;   // measured: the next 8-strip batch into L2 while this one loads
        } else {
            // short N: warps share rows; the smallest split whose per-warp K
            // slice fits 4-strip ring slots, then finer while N is short
            split = 2;
            while (split < 8 && gemv_strips_per_warp(K, split) > 4)
                split *= 2;
            while (split < 8 && static_cast<long long>(N) * split < 48ll * num_sms)
                split *= 2;
        }
        if (split > 1 && (gemv_strips_per_warp(K, split) > 16 || gemv_smem_bytes(M, K, split, 2) > kGemvMaxSmem))
            split = 1;   // K too long for the shared rows' ring
        fill_gemv(d, split, ring, grid, num_sms);
        if (split > 1 && d->stages < 2)
            return fail(SKG_ERR_UNSUPPORTED, "M=%d K=%d does not fit the M<=2 kernel's shared memory", M, K);
    } else {
        int split, stages = 0, burst = 1;
        const int n_tiles = (N + kTileN - 1) / kTileN;
        if (row) {
            split = row->split;
            stages = row->stages;
            burst = row->burst;
            d->l2_ahead = row->ahead;
            d->from_table = 1;
        } else {
            // Measured on GB300 (the tuned rows and 48 shapes outside the
            // table, back-to-back launches): the fastest launches split K as
            // finely as one wave of CTAs at the ring's occupancy holds (at
            // most 8 ways, no finer than the chunks K has), with a short ring:
            // m_pad 16 takes 4 stages (3 CTAs per SM) or 6 (2 per SM), m_pad
            // 32 3 stages (3 per SM) or 4 (2 per SM) -- the deeper ring
            // wherever 2 CTAs per SM hold the same split in one wave -- and
            // m_pad 48 and 64 4 stages (2 per SM).  One CTA per SM with a
            // deep ring and grids beyond one wave both lose.
            const int mp = (M + 15) / 16 * 16;
            const int present = chunks_present((K + kBlockK - 1) / kBlockK);
            auto split_for = [&](int per_sm) {
                int sp = 2;
                while (sp < 8 && static_cast<long long>(n_tiles) * sp * 2 <= static_cast<long long>(num_sms) * per_sm &&
                       sp * 2 <= present)
                    sp *= 2;
                return sp;
            };
            const int s3 = split_for(3), s2 = split_for(2);
            const bool deep = mp > 32 || (s2 == s3 && static_cast<long long>(n_tiles) * s2 <= 2ll * num_sms);
            split = deep ? s2 : s3;
            stages = mp == 16 ? (deep ? 6 : 4) : (mp == 32 ? (deep ? 4 : 3) : 4);
            d->l2_ahead = 2;   // measured: 2 tiles after the ring into L2 before the wait
        }
        d->reducers = (row && row->reducers > 0) ? row->reducers : default_reducers(M, split, n_tiles);
        fill_tc(d, split, stages, burst);
    }
    return SKG_OK;
}

// --------------------------------------------------------- TMA descriptors
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2-D bf16 row-major [rows, cols] with a box of [box_rows, 64], 128B swizzle,
// zero fill outside the tensor.
skg_status encode_2d(CUtensorMap *m, const void *base, int rows, int cols, int box_rows)
{
    EncodeTiledFn enc = get_encode();
    if (!enc)
        return fail(SKG_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBlockK), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
                           box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(SKG_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d) for [%d,%d]", (int)r, rows, cols);
    return SKG_OK;
}

constexpr int kMapCache = 4;

struct MapCache {
    const void *ptr[kMapCache] = {};
    CUtensorMap map[kMapCache];
    int next = 0;

    skg_status get(const void *base, int rows, int cols, int box_rows, const CUtensorMap **out)
    {
        for (int i = 0; i < kMapCache; ++i) {
            if (ptr[i] == base) {
                *out = &map[i];
                return SKG_OK;
            }
        }
        const int slot = next;
        next = (next + 1) % kMapCache;
        ptr[slot] = nullptr;
        skg_status st = encode_2d(&map[slot], base, rows, cols, box_rows);
        if (st != SKG_OK)
            return st;
        ptr[slot] = base;
        *out = &map[slot];
        return SKG_OK;
    }
    void clear() { std::fill(ptr, ptr + kMapCache, nullptr); }
};

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// The reducers per tile a launch may use: at most the plan's R and the
// split (splits of 16 reduce in one CTA), and none but the last arrival
// while the grid, tiles x split, is more than one wave of the CTAs the SMs
// hold at once (`slots`; a waiter would wait for CTAs of a later wave,
// measured 25% slower on a two-wave launch).  Within one wave the waiting
// CTAs, tiles x (R - 1), are fewer than the slots, so every CTA a waiter
// waits for -- one that never waits -- always has an SM.
int safe_reducers(int want, int n_tiles, int split, int slots)
{
    if (split > 8 || static_cast<long long>(n_tiles) * split > slots)
        return 1;
    return std::max(1, std::min(want, split));
}

} // namespace

namespace skg {

skg_status set_error(skg_status st, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

skg_status prepare_splitk_launch(int M, int N, int K, int epi, const void *x, const void *W,
                                 const void *residual, const void *y, size_t scratch_bytes,
                                 int max_tiles, CUtensorMap *tmW, CUtensorMap *tmX, TcParams *t,
                                 int *m_pad, int *grid)
{
    if (!x || !W || !y)
        return fail(SKG_ERR_INVALID_ARG, "x, W and y must be non-NULL");
    if (M <= 2 && M >= 1)
        return fail(SKG_ERR_UNSUPPORTED, "M=%d runs the small-matrix kernel, which needs no scratch: use skg_run", M);
    int dev = 0, sms = 0, l2 = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "device query");
    skg_plan_desc d;
    skg_status st = query(M, N, K, epi, sms, static_cast<size_t>(l2), &d);
    if (st != SKG_OK)
        return st;
    const bool want_res = epi == SKG_EPI_BF16_RESIDUAL;
    if (want_res != (residual != nullptr))
        return fail(SKG_ERR_INVALID_ARG, want_res ? "this epilogue needs a residual" : "this epilogue takes no residual");
    if (!aligned(x, 16) || !aligned(W, 16))
        return fail(SKG_ERR_ALIGNMENT, "x and W must be 16-byte aligned");
    if (!aligned(y, epi == SKG_EPI_FP32 ? 4 : 2) || (residual && !aligned(residual, 2)))
        return fail(SKG_ERR_ALIGNMENT, "y / residual miss their element alignment");
    const int n_tiles = (N + kTileN - 1) / kTileN;
    if (n_tiles > max_tiles)
        return fail(SKG_ERR_UNSUPPORTED, "N=%d needs %d arrival counters; the static scratch has %d", N, n_tiles,
                    max_tiles);
    if (tc_partial_bytes(M, N, d.split_k) > scratch_bytes)
        return fail(SKG_ERR_UNSUPPORTED, "M=%d N=%d needs %zu bytes of partials at split %d; the static scratch holds %zu",
                    M, N, tc_partial_bytes(M, N, d.split_k), d.split_k, scratch_bytes);
    st = encode_2d(tmW, W, N, K, kTileN);
    if (st != SKG_OK)
        return st;
    st = encode_2d(tmX, x, M, K, d.m_pad);
    if (st != SKG_OK)
        return st;
    *t = TcParams{};
    t->res = static_cast<const uint16_t *>(residual);
    t->y = const_cast<void *>(y);
    t->M = M;
    t->N = N;
    t->K = K;
    t->split = d.split_k;
    t->nkb = (K + kBlockK - 1) / kBlockK;
    t->n_tiles = n_tiles;
    t->stages = d.stages;
    t->burst = d.tma_burst;
    t->ahead = d.l2_ahead;
    t->epilogue = epi;
    t->timeout_ns = kDefaultTimeoutNs;
    int occ = 1;
    e = tc_occupancy(d.m_pad, d.stages, &occ);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
    t->reducers = safe_reducers(d.reducers, n_tiles, d.split_k, sms * std::max(1, occ));
    t->chunk_base = 0;
    t->chunk_count = kChunks;
    *m_pad = d.m_pad;
    *grid = d.grid;
    return SKG_OK;
}

} // namespace skg

struct skg_plan_s {
    skg_plan_desc d;
    int device = 0;
    int num_sms = 0;
    size_t l2_bytes = 0;
    double prefetch_fraction = 0.5;
    void *ws = nullptr;               // [S][tiles][M][128] fp32 partials, then counters
    size_t ws_cap = 0;
    std::vector<void *> retired;      // outgrown workspaces: a captured graph may still use them
    int want_reducers = 0;            // requested reducers per tile (table, default or skg_plan_set_reducers)
    bool reducers_set = false;        // want_reducers came from skg_plan_set_reducers
    int occ_m_pad = 0, occ_stages = 0; // shape of the split-K launch tc_ctas_per_sm was measured for
    int tc_ctas_per_sm = 1;
    const void *next_w = nullptr;     // prefetched into L2 by this plan's launches
    size_t next_bytes = 0;
    int gemv_ctas_per_sm = 0;         // measured occupancy of the GEMV kernel
    unsigned int *err_host = nullptr; // mapped pinned word
    unsigned int *err_dev = nullptr;
    cudaStream_t last_stream = nullptr;
    MapCache wmaps, xmaps;
    int k_rank = 0, k_ranks = 1;      // K shard: canonical chunks [16 r / R, 16 (r + 1) / R)
};

// A group: several projections of the same M in one persistent launch.
struct skg_group_s {
    int n = 0, M = 0, m_pad = 0, device = 0, num_sms = 0, stages = 0, grid = 0, units = 0;
    int N[kGroupMax] = {}, K[kGroupMax] = {}, epi[kGroupMax] = {}, dep[kGroupMax] = {};
    int split[kGroupMax] = {}, n_tiles[kGroupMax] = {}, ahead[kGroupMax] = {}, reducers[kGroupMax] = {};
    size_t ws_off[kGroupMax] = {}, ctr_off[kGroupMax] = {}, done_off = 0, ws_bytes = 0;
    void *ws = nullptr;               // partials and counters of every projection, then done[]
    unsigned int *err_host = nullptr; // mapped pinned word
    unsigned int *err_dev = nullptr;
    cudaStream_t last_stream = nullptr;
    MapCache wmaps[kGroupMax], xmaps[kGroupMax];
};

namespace {

skg_status ensure_workspace(skg_plan_s *p)
{
    const size_t need = p->d.workspace_bytes;
    if (need == 0 || need <= p->ws_cap) {
        if (need && p->ws) {
            // counters must start at zero for a new split
            const size_t n_tiles = (p->d.N + kTileN - 1) / kTileN;
            const size_t part = need - n_tiles * sizeof(unsigned int);
            cudaError_t e = cudaMemset(static_cast<char *>(p->ws) + part, 0, n_tiles * sizeof(unsigned int));
            if (e != cudaSuccess)
                return cuda_fail(e, "cudaMemset(counters)");
        }
        return SKG_OK;
    }
    if (p->ws) {
        // Not freed here: a CUDA graph captured earlier may still launch with
        // this pointer.  Released by skg_plan_destroy.
        p->retired.push_back(p->ws);
        p->ws = nullptr;
        p->ws_cap = 0;
    }
    cudaError_t e = cudaMalloc(&p->ws, need);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaMalloc(split-K workspace)");
    e = cudaMemset(p->ws, 0, need);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaMemset(split-K workspace)");
    p->ws_cap = need;
    return SKG_OK;
}

void refresh_prefetch_bytes(skg_plan_s *p)
{
    const size_t wbytes = static_cast<size_t>(p->d.N) * (p->d.K / p->k_ranks) * 2;   // the W (shard) it runs on
    const double want = p->prefetch_fraction * static_cast<double>(p->l2_bytes);
    p->d.prefetch_bytes = std::min(wbytes, static_cast<size_t>(want)) & ~static_cast<size_t>(15);
}

} // namespace

extern "C" {

int skg_version(void) { return SKG_VERSION; }

const char *skg_last_error(void) { return g_last_error.c_str(); }

skg_status skg_plan_query(int M, int N, int K, int epilogue, int num_sms, size_t l2_bytes,
                          skg_plan_desc *out)
{
    return query(M, N, K, epilogue, num_sms, l2_bytes, out);
}

// After any change of a plan's launch shape: the reducers per tile its
// launches use (the requested count within the bound of safe_reducers, for
// this shape's occupancy), then the workspace for the shape.
skg_status finish_update(skg_plan_t p)
{
    if (p->d.kernel_kind == SKG_KERNEL_SPLITK_TC) {
        if (p->occ_m_pad != p->d.m_pad || p->occ_stages != p->d.stages) {
            int occ = 1;
            const cudaError_t e = tc_occupancy(p->d.m_pad, p->d.stages, &occ);
            if (e != cudaSuccess)
                return cuda_fail(e, "split-K occupancy");
            p->occ_m_pad = p->d.m_pad;
            p->occ_stages = p->d.stages;
            p->tc_ctas_per_sm = std::max(1, occ);
        }
        const int n_tiles = (p->d.N + kTileN - 1) / kTileN;
        p->d.reducers = safe_reducers(p->want_reducers, n_tiles, p->d.split_k, p->num_sms * p->tc_ctas_per_sm);
    } else {
        p->d.reducers = 0;
    }
    return ensure_workspace(p);
}

skg_status skg_plan(int M, int N, int K, int epilogue, skg_plan_t *out)
{
    if (!out)
        return fail(SKG_ERR_INVALID_ARG, "skg_plan: out is NULL");
    *out = nullptr;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    int major = 0, minor = 0, sms = 0, l2 = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    e = cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaDeviceGetAttribute");
    if (major != 10 || minor != 3)
        return fail(SKG_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a only",
                    dev, major, minor);
    skg_plan_desc d;
    skg_status st = query(M, N, K, epilogue, sms, static_cast<size_t>(l2), &d);
    if (st != SKG_OK)
        return st;
    skg_plan_s *p = new (std::nothrow) skg_plan_s();
    if (!p)
        return fail(SKG_ERR_CUDA, "out of host memory");
    p->d = d;
    p->device = dev;
    p->num_sms = sms;
    p->l2_bytes = static_cast<size_t>(l2);
    refresh_prefetch_bytes(p);
    if (p->d.kernel_kind == SKG_KERNEL_GEMV) {
        e = gemv_occupancy(M, K, p->d.split_k, p->d.stages, &p->gemv_ctas_per_sm);
        if (e != cudaSuccess) {
            delete p;
            return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
        }
        if (p->gemv_ctas_per_sm < 1) {
            delete p;
            return fail(SKG_ERR_UNSUPPORTED, "the M<=2 kernel cannot be resident with this shape");
        }
        if (gemv_grid_from_occupancy(p->d))
            fill_gemv(&p->d, p->d.split_k, p->d.stages, sms * p->gemv_ctas_per_sm, sms);
    }
    e = cudaHostAlloc(reinterpret_cast<void **>(&p->err_host), sizeof(unsigned int), cudaHostAllocMapped);
    if (e != cudaSuccess) {
        delete p;
        return cuda_fail(e, "cudaHostAlloc(error word)");
    }
    *p->err_host = 0;
    e = cudaHostGetDevicePointer(reinterpret_cast<void **>(&p->err_dev), p->err_host, 0);
    if (e != cudaSuccess) {
        cudaFreeHost(p->err_host);
        delete p;
        return cuda_fail(e, "cudaHostGetDevicePointer(error word)");
    }
    p->want_reducers = p->d.reducers;
    st = finish_update(p);
    if (st != SKG_OK) {
        skg_plan_destroy(p);
        return st;
    }
    *out = p;
    return SKG_OK;
}

skg_status skg_plan_force(skg_plan_t p, int split_k, int stages, int grid, int tma_burst)
{
    if (!p)
        return fail(SKG_ERR_INVALID_ARG, "skg_plan_force: plan is NULL");
    skg_plan_desc d = p->d;
    if (split_k != 0) {
        if (!is_pow2(split_k) || kChunks % split_k != 0)
            return fail(SKG_ERR_INVALID_ARG, "split_k=%d must be a power of 2 dividing %d", split_k, kChunks);
        if (d.kernel_kind == SKG_KERNEL_GEMV && split_k > 1 && gemv_strips_per_warp(d.K, split_k) > 16)
            return fail(SKG_ERR_UNSUPPORTED, "split_k=%d leaves more than 16 strips per warp at K=%d", split_k, d.K);
        if (d.kernel_kind == SKG_KERNEL_SPLITK_TC && split_k < 2)
            return fail(SKG_ERR_UNSUPPORTED, "the tensor-core kernel needs split_k >= 2");
        if (d.kernel_kind == SKG_KERNEL_GEMV && split_k > 8)
            return fail(SKG_ERR_UNSUPPORTED, "the GEMV kernel supports split_k <= 8");
        if (split_k > kChunks / p->k_ranks)
            return fail(SKG_ERR_UNSUPPORTED, "split_k=%d exceeds the %d chunks of this plan's K shard", split_k,
                        kChunks / p->k_ranks);
    }
    const int split = split_k ? split_k : d.split_k;
    const bool gemv_rows = d.kernel_kind == SKG_KERNEL_GEMV && split == 1;
    if (stages != 0 && (stages < (gemv_rows ? 1 : 2) ||
                        stages > (gemv_rows ? 3 : (d.kernel_kind == SKG_KERNEL_GEMV ? 9 : 16))))
        return fail(SKG_ERR_INVALID_ARG, "stages=%d invalid for this plan", stages);
    if (tma_burst != 0 && (d.kernel_kind == SKG_KERNEL_SPLITK_TC ? tma_burst < 1
                                                                 : !(gemv_rows && (tma_burst == 4 || tma_burst == 8))))
        return fail(SKG_ERR_INVALID_ARG, "tma_burst=%d invalid for this plan", tma_burst);
    if (grid != 0 && (d.kernel_kind != SKG_KERNEL_GEMV || grid < 1))
        return fail(SKG_ERR_INVALID_ARG, "grid=%d invalid for this plan", grid);
    if (gemv_rows) {
        // stages 1: weights straight into registers; >= 2: the copy-engine
        // ring with that many slots; 0: keep the current form
        const int ring = stages == 1 ? 0 : (stages >= 2 ? stages : (d.split_k == 1 ? d.stages : 0));
        const int batch = tma_burst ? tma_burst : (d.stages >= 2 ? d.tma_burst : gemv_bulk_default_batch(d.M, d.K));
        if (tma_burst && ring < 2)
            return fail(SKG_ERR_INVALID_ARG, "tma_burst applies to the bulk-copy form (stages 2) only");
        if (ring >= 2 && !gemv_bulk_ok(d.M, d.K, batch))
            return fail(SKG_ERR_UNSUPPORTED, "the bulk-copy form needs K %% 256 == 0 and room for %d-strip batches "
                        "(M=%d K=%d)", batch, d.M, d.K);
        if (ring == 3 && grid && (d.N + std::min(grid, d.N) - 1) / std::min(grid, d.N) > kGemvSpanMaxRows)
            return fail(SKG_ERR_UNSUPPORTED, "the one-wave form takes at most %d rows per CTA (N=%d, grid=%d)",
                        kGemvSpanMaxRows, d.N, grid);
        d.tma_burst = ring >= 2 ? batch : 0;
        fill_gemv(&d, 1, ring, grid, p->num_sms);
        if (ring == 3 && d.smem_bytes > kGemvMaxSmem)
            return fail(SKG_ERR_UNSUPPORTED, "the one-wave form does not fit shared memory at M=%d K=%d", d.M, d.K);
    } else if (d.kernel_kind == SKG_KERNEL_GEMV) {
        int ctas = 1;
        int ring = stages ? stages : ((split_k || d.stages < 2) ? gemv_default_ring(d.M, d.K, split, &ctas) : d.stages);
        if (ring < 2 || gemv_smem_bytes(d.M, d.K, split, ring) > kGemvMaxSmem)
            return fail(SKG_ERR_UNSUPPORTED, "a %d-slot ring does not fit shared memory at split %d", ring, split);
        int g = grid ? grid : d.grid;
        if ((split_k || stages || d.split_k == 1) && !grid) {
            int occ = 1;
            cudaError_t e = gemv_occupancy(d.M, d.K, split, ring, &occ);
            if (e != cudaSuccess)
                return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
            if (occ < 1)
                return fail(SKG_ERR_UNSUPPORTED, "this GEMV configuration cannot be resident");
            p->gemv_ctas_per_sm = occ;
            g = p->num_sms * occ;
        }
        fill_gemv(&d, split, ring, g, p->num_sms);
    } else {
        const int st = stages ? stages : d.stages;
        if (st > tc_max_stages(d.m_pad, 232448))
            return fail(SKG_ERR_UNSUPPORTED, "stages=%d does not fit in shared memory", st);
        const int b = tma_burst ? tma_burst : d.tma_burst;
        if (b > st)
            return fail(SKG_ERR_INVALID_ARG, "tma_burst=%d exceeds stages=%d", b, st);
        fill_tc(&d, split, st, b);
    }
    d.from_table = 0;
    p->d = d;
    if (!p->reducers_set && d.kernel_kind == SKG_KERNEL_SPLITK_TC)
        p->want_reducers = default_reducers(d.M, d.split_k, (d.N + kTileN - 1) / kTileN);   // the forced shape's default
    p->wmaps.clear();
    p->xmaps.clear();
    return finish_update(p);
}

skg_status skg_plan_force_kernel(skg_plan_t p, int kind)
{
    if (!p)
        return fail(SKG_ERR_INVALID_ARG, "skg_plan_force_kernel: plan is NULL");
    if (p->k_ranks > 1 && kind == SKG_KERNEL_GEMV)
        return fail(SKG_ERR_UNSUPPORTED, "a K-sharded plan runs the split-K kernel");
    skg_plan_desc d;
    skg_status st = query(p->d.M, p->d.N, p->d.K, p->d.epilogue, p->num_sms, p->l2_bytes, &d, kind);
    if (st != SKG_OK)
        return st;
    d.pdl = p->d.pdl;
    int ctas = p->gemv_ctas_per_sm;
    if (d.kernel_kind == SKG_KERNEL_GEMV) {
        const cudaError_t e = gemv_occupancy(d.M, d.K, d.split_k, d.stages, &ctas);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
        if (ctas < 1)
            return fail(SKG_ERR_UNSUPPORTED, "the M<=2 kernel cannot be resident with this shape");
        if (gemv_grid_from_occupancy(d))
            fill_gemv(&d, d.split_k, d.stages, p->num_sms * ctas, p->num_sms);
    }
    p->gemv_ctas_per_sm = ctas;
    if (p->k_ranks > 1 && d.split_k > kChunks / p->k_ranks)
        fill_tc(&d, kChunks / p->k_ranks, d.stages, d.tma_burst);
    p->d = d;
    p->want_reducers = d.reducers;   // re-planned: the new shape's default
    p->reducers_set = false;
    p->wmaps.clear();
    p->xmaps.clear();
    return finish_update(p);
}

skg_status skg_plan_set_k_shard(skg_plan_t p, int rank, int ranks)
{
    if (!p)
        return fail(SKG_ERR_INVALID_ARG, "skg_plan_set_k_shard: plan is NULL");
    if (ranks != 1 && ranks != 2 && ranks != 4 && ranks != 8)
        return fail(SKG_ERR_INVALID_ARG, "ranks=%d must be 1, 2, 4 or 8", ranks);
    if (rank < 0 || rank >= ranks)
        return fail(SKG_ERR_INVALID_ARG, "rank=%d outside 0..%d", rank, ranks - 1);
    if (ranks > 1) {
        if (p->d.epilogue != SKG_EPI_FP32)
            return fail(SKG_ERR_UNSUPPORTED, "a K shard leaves an fp32 partial: the plan's epilogue must be fp32");
        if (p->d.K % (kChunks * kBlockK) != 0)
            return fail(SKG_ERR_UNSUPPORTED, "K=%d: sharding needs K %% %d == 0 (whole, equal canonical chunks)",
                        p->d.K, kChunks * kBlockK);
    }
    skg_plan_desc d = p->d;
    const bool replan = ranks > 1 && d.kernel_kind != SKG_KERNEL_SPLITK_TC;
    if (replan) {
        const skg_status st = query(d.M, d.N, d.K, d.epilogue, p->num_sms, p->l2_bytes, &d, SKG_KERNEL_SPLITK_TC);
        if (st != SKG_OK)
            return st;
        d.pdl = p->d.pdl;
    }
    if (d.kernel_kind == SKG_KERNEL_SPLITK_TC && d.split_k > kChunks / ranks)
        fill_tc(&d, kChunks / ranks, d.stages, d.tma_burst);   // a rank's CTAs split its chunks
    p->d = d;
    if (replan) {
        p->want_reducers = d.reducers;
        p->reducers_set = false;
    }
    p->k_rank = rank;
    p->k_ranks = ranks;
    refresh_prefetch_bytes(p);
    p->wmaps.clear();
    p->xmaps.clear();
    return finish_update(p);
}

skg_status skg_combine_partials(int M, int N, int ranks, const float *const *partials, const void *residual,
                                void *y, int epilogue, void *stream)
{
    if (M < 1 || M > 64 || N < 1)
        return fail(SKG_ERR_INVALID_ARG, "skg_combine_partials: M=%d N=%d", M, N);
    if (ranks != 1 && ranks != 2 && ranks != 4 && ranks != 8)
        return fail(SKG_ERR_INVALID_ARG, "skg_combine_partials: ranks=%d must be 1, 2, 4 or 8", ranks);
    if (!partials || !y)
        return fail(SKG_ERR_INVALID_ARG, "skg_combine_partials: partials and y must be non-NULL");
    if (epilogue != SKG_EPI_BF16 && epilogue != SKG_EPI_BF16_RESIDUAL && epilogue != SKG_EPI_FP32)
        return fail(SKG_ERR_INVALID_ARG, "unknown epilogue %d", epilogue);
    if ((epilogue == SKG_EPI_BF16_RESIDUAL) != (residual != nullptr))
        return fail(SKG_ERR_INVALID_ARG, "skg_combine_partials: residual must be given iff the epilogue adds one");
    for (int r = 0; r < ranks; ++r)
        if (!partials[r] || !aligned(partials[r], 4))
            return fail(SKG_ERR_INVALID_ARG, "skg_combine_partials: partial %d is NULL or misaligned", r);
    if (!aligned(y, epilogue == SKG_EPI_FP32 ? 4 : 2) || (residual && !aligned(residual, 2)))
        return fail(SKG_ERR_ALIGNMENT, "skg_combine_partials: y / residual miss their element alignment");
    const cudaError_t e = launch_combine(partials, ranks, static_cast<const uint16_t *>(residual), y, M, N, epilogue,
                                         static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "skg_combine_partials launch");
    return SKG_OK;
}

skg_status skg_plan_set_pdl(skg_plan_t p, int enable)
{
    if (!p)
        return fail(SKG_ERR_INVALID_ARG, "skg_plan_set_pdl: plan is NULL");
    p->d.pdl = enable ? 1 : 0;
    return SKG_OK;
}

skg_status skg_plan_set_next_weight(skg_plan_t p, const void *W_next, size_t bytes)
{
    if (!p)
        return fail(SKG_ERR_INVALID_ARG, "skg_plan_set_next_weight: plan is NULL");
    if (W_next && !aligned(W_next, 16))
        return fail(SKG_ERR_ALIGNMENT, "skg_plan_set_next_weight: W_next must be 16-byte aligned");
    p->next_w = W_next;
    p->next_bytes = W_next ? (std::min(bytes, p->l2_bytes) & ~static_cast<size_t>(15)) : 0;
    return SKG_OK;
}

skg_status skg_plan_set_l2_ahead(skg_plan_t p, int ahead)
{
    if (!p)
        return fail(SKG_ERR_INVALID_ARG, "skg_plan_set_l2_ahead: plan is NULL");
    if (ahead < 0 || ahead > 64)
        return fail(SKG_ERR_INVALID_ARG, "ahead=%d outside 0..64", ahead);
    p->d.l2_ahead = ahead;
    return SKG_OK;
}

skg_status skg_plan_set_reducers(skg_plan_t p, int reducers)
{
    if (!p)
        return fail(SKG_ERR_INVALID_ARG, "skg_plan_set_reducers: plan is NULL");
    if (reducers != 1 && reducers != 2 && reducers != 4 && reducers != 8)
        return fail(SKG_ERR_INVALID_ARG, "reducers=%d must be 1, 2, 4 or 8", reducers);
    if (p->d.kernel_kind != SKG_KERNEL_SPLITK_TC)
        return fail(SKG_ERR_UNSUPPORTED, "reducers apply to the split-K kernel only");
    p->want_reducers = reducers;
    p->reducers_set = true;
    return finish_update(p);
}

skg_status skg_plan_set_prefetch_fraction(skg_plan_t p, double fraction)
{
    if (!p)
        return fail(SKG_ERR_INVALID_ARG, "skg_plan_set_prefetch_fraction: plan is NULL");
    if (!(fraction >= 0.0 && fraction <= 1.0))
        return fail(SKG_ERR_INVALID_ARG, "prefetch fraction %g outside [0, 1]", fraction);
    p->prefetch_fraction = fraction;
    refresh_prefetch_bytes(p);
    return SKG_OK;
}

skg_status skg_plan_info(skg_plan_t p, skg_plan_desc *out)
{
    if (!p || !out)
        return fail(SKG_ERR_INVALID_ARG, "skg_plan_info: NULL argument");
    *out = p->d;
    out->ctas_per_sm = p->d.kernel_kind == SKG_KERNEL_SPLITK_TC ? p->tc_ctas_per_sm : p->gemv_ctas_per_sm;
    return SKG_OK;
}

skg_status skg_run(skg_plan_t p, const void *x, const void *W, const void *residual, void *y,
                   void *stream)
{
    if (!p)
        return fail(SKG_ERR_INVALID_ARG, "skg_run: plan is NULL");
    if (!x || !W || !y)
        return fail(SKG_ERR_INVALID_ARG, "skg_run: x, W and y must be non-NULL");
    const skg_plan_desc &d = p->d;
    const bool want_res = d.epilogue == SKG_EPI_BF16_RESIDUAL;
    if (want_res != (residual != nullptr))
        return fail(SKG_ERR_INVALID_ARG, want_res ? "skg_run: this plan's epilogue needs a residual"
                                                  : "skg_run: this plan's epilogue takes no residual");
    if (!aligned(x, 16) || !aligned(W, 16))
        return fail(SKG_ERR_ALIGNMENT, "skg_run: x and W must be 16-byte aligned");
    if (!aligned(y, d.epilogue == SKG_EPI_FP32 ? 4 : 2) || (residual && !aligned(residual, 2)))
        return fail(SKG_ERR_ALIGNMENT, "skg_run: y / residual miss their element alignment");
    if (__atomic_load_n(p->err_host, __ATOMIC_ACQUIRE) != 0) {
        __atomic_store_n(p->err_host, 0u, __ATOMIC_RELEASE);
        return fail(SKG_ERR_DEVICE_TIMEOUT, "an earlier launch of this plan ran out of a bounded wait");
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (d.kernel_kind == SKG_KERNEL_GEMV) {
        GemvParams g;
        g.x = static_cast<const uint4 *>(x);
        g.W = static_cast<const uint4 *>(W);
        g.res = static_cast<const uint16_t *>(residual);
        g.y = y;
        g.err = p->err_dev;
        g.M = d.M;
        g.N = d.N;
        g.K = d.K;
        g.nv = d.K / 8;
        g.split = d.split_k;
        g.rows_per_group = d.tile_n;
        g.groups = (d.N + d.tile_n - 1) / d.tile_n;
        g.ring = d.stages;
        g.rows_per_warp = d.split_k == 1 ? d.tile_n / (kGemvThreads / 32) : 0;
        g.batch_strips = d.tma_burst;
        g.timeout_ns = kDefaultTimeoutNs;
        g.ahead = d.l2_ahead;
        g.next_w = static_cast<const unsigned char *>(p->next_w);
        g.next_bytes = p->next_bytes;
        g.epilogue = d.epilogue;
        e = launch_gemv(g, d.grid, d.pdl != 0, s);
    } else {
        const CUtensorMap *mw = nullptr, *mx = nullptr;
        const int k_cols = d.K / p->k_ranks;          // a K shard holds only its chunks' columns
        skg_status st = p->wmaps.get(W, d.N, k_cols, kTileN, &mw);
        if (st != SKG_OK)
            return st;
        st = p->xmaps.get(x, d.M, k_cols, d.m_pad, &mx);
        if (st != SKG_OK)
            return st;
        const int n_tiles = (d.N + kTileN - 1) / kTileN;
        TcParams t;
        t.res = static_cast<const uint16_t *>(residual);
        t.y = y;
        t.ws = static_cast<float *>(p->ws);
        t.counters = reinterpret_cast<unsigned int *>(static_cast<char *>(p->ws) +
                                                      tc_partial_bytes(d.M, d.N, d.split_k));
        t.err = p->err_dev;
        t.M = d.M;
        t.N = d.N;
        t.K = d.K;
        t.split = d.split_k;
        t.nkb = (d.K + kBlockK - 1) / kBlockK;
        t.n_tiles = n_tiles;
        t.stages = d.stages;
        t.burst = d.tma_burst;
        t.ahead = d.l2_ahead;
        t.next_w = static_cast<const unsigned char *>(p->next_w);
        t.next_bytes = p->next_bytes;
        t.epilogue = d.epilogue;
        t.timeout_ns = kDefaultTimeoutNs;
        t.reducers = d.reducers;      // bounded for this launch shape whenever the shape changed
        t.chunk_count = kChunks / p->k_ranks;
        t.chunk_base = p->k_rank * t.chunk_count;
        e = launch_splitk_tc(*mw, *mx, t, d.m_pad, d.grid, d.pdl != 0, s);
    }
    if (e != cudaSuccess)
        return cuda_fail(e, "skg_run launch");
    p->last_stream = s;
    return SKG_OK;
}

skg_status skg_prefetch_l2(skg_plan_t next, const void *W_next, void *side_stream)
{
    if (!next || !W_next)
        return fail(SKG_ERR_INVALID_ARG, "skg_prefetch_l2: NULL argument");
    if (!aligned(W_next, 16))
        return fail(SKG_ERR_ALIGNMENT, "skg_prefetch_l2: W_next must be 16-byte aligned");
    cudaError_t e = launch_prefetch_l2(W_next, next->d.prefetch_bytes, static_cast<cudaStream_t>(side_stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "skg_prefetch_l2 launch");
    return SKG_OK;
}

skg_status skg_plan_check(skg_plan_t p)
{
    if (!p)
        return fail(SKG_ERR_INVALID_ARG, "skg_plan_check: plan is NULL");
    cudaError_t e = p->last_stream ? cudaStreamSynchronize(p->last_stream) : cudaDeviceSynchronize();
    if (e != cudaSuccess)
        return cuda_fail(e, "skg_plan_check synchronize");
    e = cudaGetLastError();
    if (e != cudaSuccess)
        return cuda_fail(e, "skg_plan_check pending error");
    const unsigned w = __atomic_exchange_n(p->err_host, 0u, __ATOMIC_ACQ_REL);
    if (w != 0) {
        // an aborted split-K run leaves its arrival counters unreset
        ensure_workspace(p);
        return fail(SKG_ERR_DEVICE_TIMEOUT, "a kernel of this plan ran out of a bounded wait (bits 0x%x)", w);
    }
    return SKG_OK;
}

skg_status skg_debug_wait_timeout(skg_plan_t p, unsigned long long timeout_ns, void *stream)
{
    if (timeout_ns == 0 || timeout_ns > 10000000000ull)
        return fail(SKG_ERR_INVALID_ARG, "timeout_ns must be in (0, 10 s]");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned int *err = nullptr;
    if (p) {
        err = p->err_dev;
    } else {
        // no plan: the timeout word of skg_run_noalloc's fixed array
        const skg_status st = noalloc_error_word(&err);
        if (st != SKG_OK)
            return st;
    }
    cudaError_t e = launch_debug_wait(err, timeout_ns, s);
    if (e != cudaSuccess)
        return cuda_fail(e, "skg_debug_wait_timeout launch");
    if (p)
        p->last_stream = s;
    return SKG_OK;
}

skg_status skg_plan_destroy(skg_plan_t p)
{
    if (!p)
        return SKG_OK;
    if (p->ws)
        cudaFree(p->ws);
    for (void *w : p->retired)
        cudaFree(w);
    if (p->err_host)
        cudaFreeHost(p->err_host);
    delete p;
    return SKG_OK;
}

// --------------------------------------------------------------- groups
skg_status skg_group(int n, int M, const int *N, const int *K, const int *epilogue, const int *dep,
                     skg_group_t *out)
{
    if (!out)
        return fail(SKG_ERR_INVALID_ARG, "skg_group: out is NULL");
    *out = nullptr;
    if (n < 1 || n > kGroupMax)
        return fail(SKG_ERR_UNSUPPORTED, "skg_group: n=%d outside 1..%d", n, kGroupMax);
    if (!N || !K || !epilogue)
        return fail(SKG_ERR_INVALID_ARG, "skg_group: N, K and epilogue must be non-NULL");
    if (M < 1 || M > 64)
        return fail(SKG_ERR_UNSUPPORTED, "skg_group: M=%d outside 1..64", M);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    int major = 0, minor = 0, sms = 0, l2 = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    e = cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaDeviceGetAttribute");
    if (major != 10 || minor != 3)
        return fail(SKG_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a only",
                    dev, major, minor);
    skg_group_s *g = new (std::nothrow) skg_group_s();
    if (!g)
        return fail(SKG_ERR_CUDA, "out of host memory");
    g->n = n;
    g->M = M;
    g->m_pad = (M + 15) / 16 * 16;
    g->device = dev;
    g->num_sms = sms;
    size_t off = 0;
    for (int i = 0; i < n; ++i) {
        skg_plan_desc d;
        // the split-K kernel's launch shape for this projection (at M <= 2 too)
        const skg_status st =
            query(M, N[i], K[i], epilogue[i], sms, static_cast<size_t>(l2), &d, SKG_KERNEL_SPLITK_TC);
        if (st != SKG_OK) {
            delete g;
            return st;
        }
        g->N[i] = N[i];
        g->K[i] = K[i];
        g->epi[i] = epilogue[i];
        g->dep[i] = (i > 0 && dep && dep[i]) ? 1 : 0;
        // the picker's split for this projection, at most 8 (any split gives the same bits)
        g->split[i] = std::min(8, d.split_k);
        g->ahead[i] = d.l2_ahead;
        g->reducers[i] = std::min(d.reducers, g->split[i]);
        g->n_tiles[i] = (N[i] + kTileN - 1) / kTileN;
        g->ws_off[i] = off;
        off += (tc_partial_bytes(M, N[i], g->split[i]) + 255) / 256 * 256;
        g->ctr_off[i] = off;
        off += (static_cast<size_t>(g->n_tiles[i]) * sizeof(unsigned int) + 255) / 256 * 256;
        g->units += g->n_tiles[i] * g->split[i];
    }
    g->done_off = off;
    off += kGroupDoneWords * sizeof(unsigned int);
    g->ws_bytes = off;
    const int mp = g->m_pad;
    // The most CTAs per SM that still keep a ring of 4 stages each, and the
    // deepest ring at that count: while one CTA's epilogue reduces a tile the
    // others keep the SM's weight stream going.
    int per_sm = 0;
    for (int s = tc_max_stages(mp, 232448); s >= 4; --s) {
        const int c = group_ctas_per_sm(mp, s);
        if (c > per_sm) {
            per_sm = c;
            g->stages = s;
        }
    }
    if (per_sm < 1) {
        delete g;
        return fail(SKG_ERR_UNSUPPORTED, "skg_group: the group kernel cannot be resident at m_pad %d", mp);
    }
    // one wave: CTAs beyond the SMs' capacity would only start once others
    // finished (correct -- units are handed out in order -- but idle)
    g->grid = std::min(g->units, per_sm * sms);
    // Reducers per tile beyond the last arrival wait for the tile's other
    // units: allowed only where every CTA owns exactly one unit (no
    // dependencies, so CTA c runs unit c, and the grid holds every unit in
    // one wave), as in the one-projection kernel.
    bool has_dep = false;
    for (int i = 1; i < n; ++i)
        has_dep = has_dep || g->dep[i];
    if (has_dep || g->units > g->grid)
        for (int i = 0; i < n; ++i)
            g->reducers[i] = 1;
    e = cudaMalloc(&g->ws, g->ws_bytes);
    if (e == cudaSuccess)
        e = cudaMemset(g->ws, 0, g->ws_bytes);
    if (e == cudaSuccess)
        e = cudaHostAlloc(reinterpret_cast<void **>(&g->err_host), sizeof(unsigned int), cudaHostAllocMapped);
    if (e == cudaSuccess) {
        *g->err_host = 0;
        e = cudaHostGetDevicePointer(reinterpret_cast<void **>(&g->err_dev), g->err_host, 0);
    }
    if (e != cudaSuccess) {
        skg_group_destroy(g);
        return cuda_fail(e, "skg_group allocation");
    }
    *out = g;
    return SKG_OK;
}

skg_status skg_group_info(skg_group_t g, int *grid, int *stages, int *units, int *split)
{
    if (!g)
        return fail(SKG_ERR_INVALID_ARG, "skg_group_info: group is NULL");
    if (grid)
        *grid = g->grid;
    if (stages)
        *stages = g->stages;
    if (units)
        *units = g->units;
    if (split)
        for (int i = 0; i < g->n; ++i)
            split[i] = g->split[i];
    return SKG_OK;
}

skg_status skg_group_run(skg_group_t g, const void *const *x, const void *const *W, const void *const *residual,
                         void *const *y, void *stream)
{
    if (!g)
        return fail(SKG_ERR_INVALID_ARG, "skg_group_run: group is NULL");
    if (!x || !W || !y)
        return fail(SKG_ERR_INVALID_ARG, "skg_group_run: x, W and y arrays must be non-NULL");
    if (const unsigned w = __atomic_load_n(g->err_host, __ATOMIC_ACQUIRE))
        return fail(SKG_ERR_DEVICE_TIMEOUT, "an earlier launch of this group ran out of a bounded wait (bits 0x%x); "
                    "destroy the group", w);
    GroupParams gp;
    memset(&gp, 0, sizeof(gp));
    char *base = static_cast<char *>(g->ws);
    int unit = 0;
    for (int i = 0; i < g->n; ++i) {
        const void *res = residual ? residual[i] : nullptr;
        const bool want_res = g->epi[i] == SKG_EPI_BF16_RESIDUAL;
        if (!x[i] || !W[i] || !y[i])
            return fail(SKG_ERR_INVALID_ARG, "skg_group_run: projection %d: x, W and y must be non-NULL", i);
        if (want_res != (res != nullptr))
            return fail(SKG_ERR_INVALID_ARG, "skg_group_run: projection %d: residual %s", i,
                        want_res ? "missing" : "given to an epilogue without one");
        if (!aligned(x[i], 16) || !aligned(W[i], 16))
            return fail(SKG_ERR_ALIGNMENT, "skg_group_run: projection %d: x and W must be 16-byte aligned", i);
        if (!aligned(y[i], g->epi[i] == SKG_EPI_FP32 ? 4 : 2) || (res && !aligned(res, 2)))
            return fail(SKG_ERR_ALIGNMENT, "skg_group_run: projection %d: y / residual miss their alignment", i);
        const CUtensorMap *mw = nullptr, *mx = nullptr;
        skg_status st = g->wmaps[i].get(W[i], g->N[i], g->K[i], kTileN, &mw);
        if (st != SKG_OK)
            return st;
        st = g->xmaps[i].get(x[i], g->M, g->K[i], g->m_pad, &mx);
        if (st != SKG_OK)
            return st;
        GroupProj &P = gp.proj[i];
        P.tmW = *mw;
        P.tmX = *mx;
        P.res = static_cast<const uint16_t *>(res);
        P.y = y[i];
        P.ws = reinterpret_cast<float *>(base + g->ws_off[i]);
        P.counters = reinterpret_cast<unsigned int *>(base + g->ctr_off[i]);
        P.M = g->M;
        P.N = g->N[i];
        P.K = g->K[i];
        P.nkb = (g->K[i] + kBlockK - 1) / kBlockK;
        P.n_tiles = g->n_tiles[i];
        P.split = g->split[i];
        P.epilogue = g->epi[i];
        P.dep = g->dep[i];
        P.ahead = g->ahead[i];
        P.reducers = std::max(1, g->reducers[i]);
        P.unit_begin = unit;
        unit += g->n_tiles[i] * g->split[i];
    }
    gp.static_first = 1;
    for (int i = 1; i < g->n; ++i)
        if (g->dep[i])
            gp.static_first = 0;
    gp.done = reinterpret_cast<unsigned int *>(base + g->done_off);
    gp.err = g->err_dev;
    gp.n = g->n;
    gp.M = g->M;
    gp.units = g->units;
    gp.stages = g->stages;
    gp.timeout_ns = kDefaultTimeoutNs;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const cudaError_t e = launch_group_tc(gp, g->m_pad, g->grid, true, s);
    if (e != cudaSuccess)
        return cuda_fail(e, "skg_group_run launch");
    g->last_stream = s;
    return SKG_OK;
}

skg_status skg_group_check(skg_group_t g)
{
    if (!g)
        return fail(SKG_ERR_INVALID_ARG, "skg_group_check: group is NULL");
    cudaError_t e = g->last_stream ? cudaStreamSynchronize(g->last_stream) : cudaDeviceSynchronize();
    if (e != cudaSuccess)
        return cuda_fail(e, "skg_group_check synchronize");
    const unsigned w = __atomic_load_n(g->err_host, __ATOMIC_ACQUIRE);
    if (w != 0)
        return fail(SKG_ERR_DEVICE_TIMEOUT, "a launch of this group ran out of a bounded wait (bits 0x%x)", w);
    return SKG_OK;
}

skg_status skg_group_destroy(skg_group_t g)
{
    if (!g)
        return SKG_OK;
    if (g->ws)
        cudaFree(g->ws);
    if (g->err_host)
        cudaFreeHost(g->err_host);
    delete g;
    return SKG_OK;
}

} // extern "C"
