// skg_internal.h -- shared between the host ABI (skg_api.cu) and the kernel
// translation units: launch parameters, the canonical K chunking, and the
// launcher entry points.  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "skg.h"

namespace skg {

constexpr int kChunks = SKG_CANONICAL_CHUNKS;  // leaves of the canonical tree
constexpr int kTileN = 128;                    // W rows per tcgen05 tile (MMA M)
constexpr int kBlockK = 64;                    // k per TMA box: 64 bf16 = 128 B
constexpr int kTcThreads = 320;                // producer, MMA, 8 epilogue warps
constexpr int kTmemColsPerSm = 512;           // tensor memory: 128 lanes x 512 fp32 columns per SM
constexpr int kGemvThreads = 256;              // 8 warps
constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;  // 2 s bounded waits

// Start of canonical chunk c (0 <= c <= kChunks) when `units` (16-byte
// vectors for GEMV, 64-wide k-blocks for the tensor-core kernel) are cut into
// kChunks chunks: the first units % kChunks chunks hold one unit more, so
// any empty chunks are the last ones.
__host__ __device__ __forceinline__ int chunk_begin(int c, int units)
{
    const int q = units / kChunks, r = units % kChunks;
    return c * q + (c < r ? c : r);
}

// Number of non-empty chunks.
__host__ __device__ __forceinline__ int chunks_present(int units)
{
    return units >= kChunks ? kChunks : units;
}

struct GemvParams {
    const uint4 *x;         // [M, K/8] 16-byte vectors
    const uint4 *W;         // [N, K/8]
    const uint16_t *res;    // [M, N] bf16 bits or null
    void *y;                // [M, N] bf16 bits or fp32
    unsigned int *err;      // device-visible error word (mapped host memory)
    int M, N, K;
    int nv;                 // K / 8
    int split;              // warps per output row (1, 2, 4, 8)
    int rows_per_group;     // 8 / split
    int groups;             // ceil(N / rows_per_group)
    int ring;               // split > 1: weight-ring slots per warp (2..9); split 1: the form --
                            // 0 16-byte loads, 2 whole rows with bulk-copied batches, 3 one wave
    int ahead;              // split 1: batches of the row requested into L2 ahead of use
    const unsigned char *next_w;  // the next projection's weight, or null
    size_t next_bytes;      // bytes of next_w the grid asks the L2 for (multiple of 16)
    int rows_per_warp;      // split 1: consecutive rows each warp computes
    int batch_strips;       // split 1, bulk-copied batches: strips per copy (4 or 8)
    int epilogue;           // skg_epilogue
    unsigned long long timeout_ns;  // bounded mbarrier waits (bulk-copy forms)
};

struct TcParams {
    const uint16_t *res;    // [M, N] bf16 bits or null
    void *y;                // [M, N]
    float *ws;              // [S, M, N] fp32 partials (S > 1)
    unsigned int *counters; // [n_tiles] arrival counters, zero between runs
    unsigned int *err;      // device-visible error word
    int M, N, K;
    int split;              // S: CTAs per output tile (2, 4, 8, 16)
    int nkb;                // ceil(K / 64)
    int n_tiles;            // ceil(N / 128)
    int stages;             // shared-memory pipeline depth
    int burst;              // k-blocks the producer requests back to back
    int ahead;              // W tiles requested into L2 this many k-blocks ahead
    const unsigned char *next_w;  // the next projection's weight, or null
    size_t next_bytes;      // bytes of next_w the grid asks the L2 for (multiple of 16)
    int epilogue;
    unsigned long long timeout_ns;
    int reducers;           // R: the last R arrivals of a tile each reduce 1/R of it (1, 2, 4, 8)
    int chunk_base;         // first canonical K chunk of this launch (0 unless K is sharded)
    int chunk_count;        // canonical chunks of this launch (16 unless K is sharded)
};

// Several projections of the same M in one persistent split-K launch.
constexpr int kGroupMax = 8;
struct GroupProj {              // aligned as CUtensorMap
    CUtensorMap tmW;        // W [N, K], box 64 x 128
    CUtensorMap tmX;        // x [M, K], box 64 x m_pad
    const uint16_t *res;    // [M, N] bf16 bits or null
    void *y;                // [M, N]
    float *ws;              // fp32 partials, tile-major [split][tiles][M][128]
    unsigned int *counters; // [n_tiles] arrival counters, zero between runs
    int M, N, K, nkb, n_tiles, split, epilogue;
    int dep;                // 1: x read only after the previous projection of the group is complete
    int ahead;              // W k-blocks past the ring prefetched to L2 before a wait for x
    int unit_begin;         // first work unit (tile, split) of this projection
    int reducers;           // R: the last R arrivals of a tile each reduce 1/R of it (R > 1 only when every
                            // CTA owns one unit and the group has no dependencies)
};

constexpr int kGroupDoneExit = kGroupMax;
constexpr int kGroupDoneNext = kGroupMax + 1;
constexpr int kGroupDoneWords = kGroupMax + 2;
constexpr int kGroupUnitQueue = 16;   // unit ids in flight from the producer to the MMA and epilogue
int group_smem_bytes(int m_pad, int stages);

struct GroupParams {
    GroupProj proj[kGroupMax];
    unsigned int *done;     // [j < kGroupMax] tiles finished per projection, [kGroupDoneExit] CTAs
                            // finished, [kGroupDoneNext] units handed out
    unsigned int *err;
    int n, M, units, stages;
    int static_first;       // 1 (no dependencies): CTA c's first unit is unit c, the counter hands out the rest
    unsigned long long timeout_ns;
};

// The grid's share of an L2 prefetch of the next projection's weight: CTA
// `cta` of `ctas` asks for its slice of [base, base + bytes), evict-last.
__device__ __forceinline__ void prefetch_next_slice(const unsigned char *base, size_t bytes, unsigned cta,
                                                    unsigned ctas, uint64_t pol)
{
    if (!base || bytes == 0)
        return;
    const size_t chunk = ((bytes + ctas - 1) / ctas + 15) & ~static_cast<size_t>(15);
    const size_t b0 = chunk * cta;
    if (b0 >= bytes)
        return;
    size_t n = bytes - b0 < chunk ? bytes - b0 : chunk;
    for (size_t off = 0; off < n; off += 65536) {
        const size_t k = n - off < 65536 ? n - off : 65536;
        asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;"
                     :: "l"(base + b0 + off), "r"(static_cast<uint32_t>(k)), "l"(pol) : "memory");
    }
}

// Error-word bits written by kernels.
constexpr unsigned kErrTimeoutProducer = 1u << 0;
constexpr unsigned kErrTimeoutMma = 1u << 1;
constexpr unsigned kErrTimeoutEpilogue = 1u << 2;
constexpr unsigned kErrTimeoutDebug = 1u << 3;

// Bytes of fp32 split-K partials: S x ceil(N / 128) tiles x [M][128].
inline size_t tc_partial_bytes(int M, int N, int split)
{
    return static_cast<size_t>(split) * ((N + kTileN - 1) / kTileN) * kTileN * M * sizeof(float);
}

// Shared-memory bytes of the tensor-core kernel for (m_pad, stages).
int tc_smem_bytes(int m_pad, int stages);
int gemv_smem_bytes(int M, int K, int split, int ring);
int gemv_tile_strips(int K, int split);       // ring slot size in strips: 4, 8 or 16
int gemv_fast_jc(int K);                      // >0: the specialised whole-row kernel applies
// Split 1 with the copy engine on the load path (K % 256 == 0 and room for
// one batch slot per warp): selected by ring >= 2; batches of 8 or 4 strips.
bool gemv_bulk_ok(int M, int K, int batch_strips);
int gemv_bulk_smem_bytes(int M, int K, int batch_strips);
int gemv_bulk_default_batch(int M, int K);
// Split 1 in one balanced wave (ring == 3): CTAs own row runs, warps equal chunk runs.
constexpr int kGemvSpanMaxRows = 256;
int gemv_span_smem_bytes(int M, int K, int batch_strips, int rows_per_cta);
int gemv_span_grid(int M, int N, int K, int batch_strips, int num_sms);
constexpr int kGemvMaxSmem = 226 * 1024;      // x (M * K * 2 bytes) + the weight rings (static smem needs the rest)
int tc_max_stages(int m_pad, int smem_limit);
int tc_tmem_cols(int m_pad);                  // TMEM columns one CTA allocates
cudaError_t tc_occupancy(int m_pad, int stages, int *ctas_per_sm);  // split-K CTAs one SM holds
constexpr int kTcDefaultStages = 4;

// Launchers (return the cudaError_t of the launch).
cudaError_t launch_gemv(const GemvParams &p, int grid, bool pdl, cudaStream_t s);
cudaError_t gemv_occupancy(int M, int K, int split, int ring, int *ctas_per_sm);
int gemv_strips_per_warp(int K, int split);   // must be <= 16
cudaError_t launch_splitk_tc(const CUtensorMap &tmW, const CUtensorMap &tmX, const TcParams &p,
                             int m_pad, int grid, bool pdl, cudaStream_t s);
cudaError_t launch_group_tc(const GroupParams &g, int m_pad, int grid, bool pdl, cudaStream_t s);
int group_ctas_per_sm(int m_pad, int stages);   // co-resident CTAs of the group kernel
cudaError_t launch_prefetch_l2(const void *base, size_t bytes, cudaStream_t s);
// y = the R fp32 partials combined in index order by the top levels of the
// canonical tree (+ residual), one rounding; R in {1, 2, 4, 8}.
constexpr int kMaxRanks = 8;
cudaError_t launch_combine(const float *const *partials, int ranks, const uint16_t *res, void *y, int M, int N,
                           int epilogue, cudaStream_t s);
cudaError_t launch_debug_wait(unsigned int *err, unsigned long long timeout_ns, cudaStream_t s);
// Records a failure message for skg_last_error and returns st.
skg_status set_error(skg_status st, const char *fmt, ...);

// Everything one split-K launch needs, worked out on the host without
// allocating: the checks of skg_run, the launch shape the picker chooses on
// the current device (rejected if its partials do not fit scratch_bytes),
// and the two TMA descriptors.  ws, counters and err are left null.
// Device address of the timeout word in skg_run_noalloc's fixed array.
skg_status noalloc_error_word(unsigned int **out);

skg_status prepare_splitk_launch(int M, int N, int K, int epilogue, const void *x, const void *W,
                                 const void *residual, const void *y, size_t scratch_bytes,
                                 int max_tiles, CUtensorMap *tmW, CUtensorMap *tmX, TcParams *t,
                                 int *m_pad, int *grid);

} // namespace skg
