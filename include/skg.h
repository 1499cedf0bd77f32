/*
 * skg.h -- C ABI of the skinny decode projection library (libskg.so).
 *
 * The library computes the projection of low-batch LLM decode,
 *
 *     y[m,n] = sum_k x[m,k] * W[n,k]   (+ residual[m,n])     0 <= m < M <= 64
 *
 * with bfloat16 W, x and residual, fp32 accumulation and a bf16 (or fp32)
 * output, on one NVIDIA GB300 (sm_103a).  Every step runs in the library's
 * own CUDA kernels; there is no CPU path and no fallback to another kernel.
 *
 * Where the operations come from.  The method is described, at paragraph
 * level and without formulas, by "Hyper Optimizing Kimi K3 in vLLM: Moving
 * Fast and Responsibly" (vLLM blog, NVIDIA), read here through its deep-notes
 * page (papercache.org) and its French translation (spke.com, "Hyper
 * optimisation de Kimi K3 dans vLLM : aller vite et responsablement"):
 *   [TS] method details 1 / Partie 1 section 1, "Tune shapes for the
 *        workload": small-matrix kernels at batch 1-2, split-K kernels at
 *        larger batch, each projection tuned to block sizes that fill the GPU.
 *   [OC] method details 2 / Partie 1 section 2, "Overlap computation and
 *        communication": the output projection fused with the attention
 *        residual add.
 *   [PF] method details 4 / Partie 1 section 4, "Prefetching upcoming weights
 *        into cache": small-batch decode is bound by streaming weights from
 *        HBM; a side-stream kernel preloads the next operation's weights.
 *   [VC] background 2 "Validate correctness systematically" / Partie 2
 *        section 3: an activation read was once hoisted above a
 *        synchronisation wait; early loads were restricted to static weights.
 *
 * Conventions shared by every entry point
 *   - Layouts are dense row-major: W is [N,K] (an nn.Linear weight), x is
 *     [M,K], residual and y are [M,N].  bf16 tensors are raw 16-bit patterns.
 *   - Device pointers are CUDA device (or managed) addresses on the current
 *     device.  x and W must be 16-byte aligned (they are read with TMA and
 *     16-byte vector loads); residual and y need their element alignment.
 *   - Streams are cudaStream_t handles passed as void* (NULL = legacy default
 *     stream).  Launches are asynchronous and stream-ordered.
 *   - The caller owns every tensor and stream.  The library owns each plan,
 *     the plan's split-K workspace and counters, and its TMA descriptors.
 *   - Every call returns a status; none throws across the ABI.  On failure,
 *     skg_last_error() returns a message for the calling thread.  A rejected
 *     call launches nothing.
 */
#ifndef SKG_H
#define SKG_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SKG_VERSION 3

/* Symbols of the ABI are exported; everything else in the library is hidden. */
#if defined(__GNUC__)
#define SKG_API __attribute__((visibility("default")))
#else
#define SKG_API
#endif

typedef enum skg_status {
    SKG_OK = 0,
    SKG_ERR_INVALID_ARG = 1,    /* bad size, NULL where a tensor is needed, bad enum */
    SKG_ERR_UNSUPPORTED = 2,    /* legal request outside what the library implements */
    SKG_ERR_ALIGNMENT = 3,      /* a pointer misses its required alignment */
    SKG_ERR_CUDA = 4,           /* a CUDA runtime/driver call failed (message says which) */
    SKG_ERR_DEVICE_TIMEOUT = 5  /* a kernel's bounded wait ran out (see skg_plan_check) */
} skg_status;

typedef enum skg_epilogue {
    SKG_EPI_BF16 = 0,           /* y = bf16(x.W^T) */
    SKG_EPI_BF16_RESIDUAL = 1,  /* y = bf16(x.W^T + residual), one rounding [OC] */
    SKG_EPI_FP32 = 2            /* y = fp32(x.W^T), e.g. router scores */
} skg_epilogue;

typedef enum skg_kernel_kind {
    SKG_KERNEL_GEMV = 1,        /* M <= 2: CUDA-core kernel; weights by 16-byte loads or bulk copies [TS] */
    SKG_KERNEL_SPLITK_TC = 2    /* M > 2: TMA + tcgen05 split-K kernel [TS] */
} skg_kernel_kind;

/* Canonical number of K chunks.  Both kernels cut K into this many chunks
 * (in 16-byte vectors for GEMV, in 64-wide k-blocks for SPLITK_TC), sum each
 * chunk from a fresh fp32 accumulator, and combine the chunk sums with one
 * fixed balanced binary tree.  A split only decides which CTA or warp owns
 * which subtree, so every allowed split gives bit-identical results. */
#define SKG_CANONICAL_CHUNKS 16

/* What a plan will launch.  Filled by skg_plan_query and skg_plan_info. */
typedef struct skg_plan_desc {
    int kernel_kind;        /* skg_kernel_kind */
    int M, N, K, epilogue;
    int split_k;            /* S: CTAs (TC) or warps (GEMV) sharing one output's K range; power of 2 dividing 16 */
    int tile_n;             /* W rows per output tile: 128 (TC) or rows per CTA group (GEMV) */
    int m_pad;              /* MMA N (TC: M rounded up to 16) or M (GEMV) */
    int stages;             /* TC: shared-memory ring stages; GEMV split > 1: weight-ring slots per
                               warp; GEMV split 1: 0 = 16-byte loads into registers, 2 = each warp's
                               weight batches moved by bulk copies through a shared-memory slot,
                               whole rows per warp; 3 = the same in one balanced wave (CTAs own row
                               runs, warps equal runs of chunks, rows combined in shared memory) */
    int tma_burst;          /* TC: k-blocks the TMA producer requests back to back; GEMV split 1
                               with bulk copies: strips (512 bytes each) per copy, 4 or 8 */
    int grid;               /* CTAs launched */
    int threads;            /* threads per CTA */
    int smem_bytes;         /* dynamic shared memory per CTA */
    int from_table;         /* 1 if (M,N,K,epilogue) hit the measured picker table */
    size_t workspace_bytes; /* split-K partials + counters owned by the plan */
    size_t prefetch_bytes;  /* bytes skg_prefetch_l2 touches for this plan's W */
    int pdl;                /* 1: launched with programmatic dependent launch */
    int l2_ahead;           /* weights requested into L2 ahead of use: TC k-blocks after the
                               ring, before the wait for the previous kernel; GEMV (split 1)
                               batches of the row; 0 = none */
    int reducers;           /* TC: the last `reducers` CTAs to finish a tile share its final
                               reduction (1, 2, 4 or 8; a launch uses fewer where the split is
                               smaller, and 1 where its grid is more than one wave); GEMV: 0 */
    int ctas_per_sm;        /* CTAs one SM holds at once: TC, from the kernel's registers, shared
                               memory, threads and TMEM columns at this launch shape; GEMV, the
                               count the plan sizes one-wave grids from.  Filled by skg_plan_info;
                               0 from skg_plan_query */
} skg_plan_desc;

typedef struct skg_plan_s *skg_plan_t;

/*
 * skg_plan_query -- the kernel choice and launch shape for (M,N,K,epilogue)
 * on a GPU with num_sms SMs and l2_bytes of L2, without touching any GPU.
 * [TS]: M <= 2 -> SKG_KERNEL_GEMV, M > 2 -> SKG_KERNEL_SPLITK_TC, except that
 * an M <= 2 shape runs the tensor-core kernel where the table of measured
 * timings holds a tensor-core row for exactly that (M,N,K,epilogue) (written
 * only where it was faster on GB300), where K is too long for the GEMV to
 * stage x in shared memory (M = 1: K > 115,200), or at M = 2 from N = 2048
 * unless the table holds a GEMV row for exactly that shape; inside each kind
 * the split and pipeline depth come from that table (nearest M for a listed
 * (N,K,epilogue)), else from a rule measured on GB300 (split-K: the finest
 * split, at most 8, whose grid is one wave at the ring's occupancy).
 * Constraints: 1 <= M <= 64, N >= 1, K >= 8 and K % 8 == 0, epilogue valid.
 * Errors: SKG_ERR_INVALID_ARG (sizes, enum, NULL out), SKG_ERR_UNSUPPORTED.
 */
SKG_API skg_status skg_plan_query(int M, int N, int K, int epilogue, int num_sms,
                          size_t l2_bytes, skg_plan_desc *out);

/*
 * skg_plan -- build a plan for (M,N,K,epilogue) on the current CUDA device.
 * Picks the kernel as skg_plan_query does and allocates a mapped host word for
 * device-side error reports; a tensor-core plan also allocates its split-K
 * workspace, S x ceil(N/128) x M x 128 fp32 partials plus one zeroed
 * counter per 128-row tile.  The plan must be
 * freed with skg_plan_destroy.  One skg_run of a plan may be in flight at a
 * time (the workspace is shared); concurrent streams need separate plans.
 * Errors: as skg_plan_query, plus SKG_ERR_CUDA.  *out is NULL on failure.
 */
SKG_API skg_status skg_plan(int M, int N, int K, int epilogue, skg_plan_t *out);

/*
 * skg_plan_force -- override of the picker inside the plan's kernel kind
 * (used by tests and by the tuning sweep): split_k (power of 2 dividing 16;
 * TC needs 2..16, GEMV 1..8); for TC, stages (2..16, limited by shared
 * memory) and tma_burst (1..stages); for GEMV, grid (CTAs, >= 1), and at
 * split 1 the load path: stages 1 = 16-byte loads into registers, stages 2 =
 * bulk copies of tma_burst (4 or 8) strips per warp batch, stages 3 = the
 * same batches in one balanced wave (grid <= N, at most 256 rows per CTA)
 * (K % 256 == 0 only; SKG_ERR_UNSUPPORTED otherwise); at split > 1, stages =
 * ring slots (2..9).  A 0 keeps the current value; a field that does not apply must be 0.
 * If the workspace must grow, a new one is allocated and the old one is kept
 * until skg_plan_destroy, because a CUDA graph that captured skg_run of this
 * plan earlier still launches with the captured split, descriptors and
 * workspace.  Used by tests to run every allowed split.  Errors: SKG_ERR_INVALID_ARG, SKG_ERR_UNSUPPORTED, SKG_ERR_CUDA.
 */
SKG_API skg_status skg_plan_force(skg_plan_t plan, int split_k, int stages, int grid,
                                  int tma_burst);

/*
 * skg_plan_force_kernel -- run the plan on the given kernel kind
 * (SKG_KERNEL_GEMV: M <= 2 only; SKG_KERNEL_SPLITK_TC: any M), its launch
 * shape re-picked as skg_plan_query picks it for that kind; earlier
 * skg_plan_force overrides are dropped, the PDL setting is kept.  The two
 * kinds accumulate in different orders, so their results may differ in the
 * last bits (each within the same error bound).  Workspace as skg_plan_force.
 * Used by the tuner and the tests.  Errors: SKG_ERR_INVALID_ARG (NULL plan,
 * unknown kind), SKG_ERR_UNSUPPORTED (GEMV at M > 2, a shape the kind cannot
 * run), SKG_ERR_CUDA.
 */
SKG_API skg_status skg_plan_force_kernel(skg_plan_t plan, int kind);

/*
 * skg_plan_set_k_shard -- [OC] row-parallel projection: the plan computes
 * rank `rank` of `ranks` (1, 2, 4 or 8) of a K split across ranks.  Rank r
 * owns canonical chunks [16r/R, 16(r+1)/R) of K, i.e. columns [rK/R,
 * (r+1)K/R) (K % 1024 == 0 when ranks > 1).  After this call skg_run takes
 * x as that shard [M, K/R] and W as [N, K/R] (dense, row stride K/R) and
 * leaves in y (fp32 [M, N]: the plan's epilogue must be SKG_EPI_FP32) the
 * value of the rank's subtree of the canonical tree, so that
 * skg_combine_partials over the R ranks gives exactly the bits of one
 * launch of the split-K kernel over the whole K.  The plan switches to the
 * split-K kernel if needed and splits a rank's chunks at most 16/R ways;
 * skg_prefetch_l2 then covers the shard.  ranks == 1 restores the whole K.
 * Errors: SKG_ERR_INVALID_ARG, SKG_ERR_UNSUPPORTED (epilogue, K), SKG_ERR_CUDA.
 */
SKG_API skg_status skg_plan_set_k_shard(skg_plan_t plan, int rank, int ranks);

/*
 * skg_combine_partials -- the cross-rank step of a row-parallel projection
 * [OC]: y[m,n] = the R rank partials (fp32 [M, N] each; `partials` is a host
 * array of R device pointers) combined in rank order by the top levels of
 * the canonical tree, + residual (bf16 [M, N], given iff epilogue is
 * SKG_EPI_BF16_RESIDUAL) in fp32, rounded once to bf16 (stored as fp32 for
 * SKG_EPI_FP32).  The caller brings the partials to this device first (an
 * all-gather, or peer pointers).  ranks: 1, 2, 4 or 8.  One kernel on
 * `stream`; allocates nothing.
 * Errors: SKG_ERR_INVALID_ARG, SKG_ERR_ALIGNMENT, SKG_ERR_CUDA.
 */
SKG_API skg_status skg_combine_partials(int M, int N, int ranks, const float *const *partials,
                                        const void *residual, void *y, int epilogue, void *stream);

/*
 * skg_plan_set_pdl -- 1 (default): launch with programmatic dependent launch,
 * so a kernel's prologue and its first WEIGHT loads overlap the previous
 * kernel in the stream; x and residual are read, and y written, only after
 * griddepcontrol.wait [VC].  0: plain stream-ordered launch.
 */
SKG_API skg_status skg_plan_set_pdl(skg_plan_t plan, int enable);

/*
 * skg_run -- y = x.W^T (+ residual) on `stream`, one kernel launch.
 *   x        device, bf16 [M,K], 16-byte aligned; read-only
 *   W        device, bf16 [N,K], 16-byte aligned; read-only (static weight)
 *   residual device, bf16 [M,N], or NULL; non-NULL iff the plan's epilogue
 *            is SKG_EPI_BF16_RESIDUAL [OC]
 *   y        device, [M,N], bf16 (fp32 for SKG_EPI_FP32); must not overlap
 *            the inputs
 * Allocates nothing.  Results are bit-identical across runs and across every
 * allowed split of the plan (see SKG_CANONICAL_CHUNKS).
 * Errors: SKG_ERR_INVALID_ARG (NULL plan/tensor, residual mismatch),
 * SKG_ERR_ALIGNMENT, SKG_ERR_DEVICE_TIMEOUT (reported by an earlier launch of
 * this plan), SKG_ERR_CUDA (descriptor encode or launch failure).
 */
SKG_API skg_status skg_run(skg_plan_t plan, const void *x, const void *W,
                   const void *residual, void *y, void *stream);

/*
 * skg_prefetch_l2 -- [PF] on `side_stream`, ask the L2 to fetch the first
 * min(2*N*K, f * L2size) bytes of W_next, the weight of the plan `next`, so
 * that next's skg_run finds them cached.  f = 0.5 unless changed with
 * skg_plan_set_prefetch_fraction; the L2 size is queried from the device
 * when the plan is built.  The kernel only issues bulk L2 prefetches (no
 * data is written); it may run concurrently with any kernel.
 * Errors: SKG_ERR_INVALID_ARG, SKG_ERR_ALIGNMENT (W_next), SKG_ERR_CUDA.
 */
SKG_API skg_status skg_prefetch_l2(skg_plan_t next, const void *W_next, void *side_stream);

/*
 * skg_plan_set_l2_ahead -- [PF] applied inside a kernel, without shared
 * memory or registers.  TC: before waiting for the previous kernel in the
 * stream, each CTA also requests the `ahead` weight tiles (128 x 64
 * k-blocks) that follow its ring into L2, so the previous kernel's tail
 * keeps HBM busy with this launch's weights.  GEMV split 1 with 16-byte
 * loads (stages 0) or in one wave (stages 3): each batch is also requested
 * into L2 `ahead` batches before it is loaded (the first ones before the
 * wait).  0..64; 0 turns it off.  The GEMV ring kernel (split > 1) and the
 * whole-row bulk-copy form (stages 2) ignore it.
 */
SKG_API skg_status skg_plan_set_l2_ahead(skg_plan_t plan, int ahead);

/*
 * skg_plan_set_reducers -- [TS] the split-K kernel's final reduction of a
 * 128-row tile (its S partial sums combined by the top levels of the
 * canonical tree, the residual added, one rounding) is done by the last R
 * CTAs of the tile to finish, each taking 1/R of the tile's outputs; all but
 * the last wait, with the plan's bounded wait, for the others.  R = 1, 2, 4
 * or 8.  The output bits do not depend on R.  A launch uses min(R, split_k),
 * and 1 at split 16 or while its grid is more than one wave of the CTAs the
 * SMs hold at once (within one wave the waiting CTAs always leave the CTAs
 * they wait for a place); the plan's description reports that count for its
 * current launch shape.  Errors: SKG_ERR_INVALID_ARG (R),
 * SKG_ERR_UNSUPPORTED (a GEMV plan), SKG_ERR_CUDA.
 */
SKG_API skg_status skg_plan_set_reducers(skg_plan_t plan, int reducers);

/*
 * skg_plan_set_next_weight -- [PF] inside the launch instead of on a side
 * stream: every later skg_run of this plan also asks the L2 (evict-last) for
 * the first `bytes` of W_next, the weight of the projection that runs next,
 * each CTA taking its slice once it has requested all of its own weight
 * tiles -- so the next launch finds its first tiles cached and this launch's
 * tail keeps HBM busy.  No extra kernel, stream or dependency is involved.
 * bytes is rounded down to a multiple of 16 and capped at the L2 size;
 * W_next must be 16-byte aligned and stay allocated while the plan runs.
 * W_next == NULL or bytes == 0 turns it off.
 */
SKG_API skg_status skg_plan_set_next_weight(skg_plan_t plan, const void *W_next, size_t bytes);

/* Fraction f in [0, 1] of the L2 that skg_prefetch_l2 fills for this plan. */
SKG_API skg_status skg_plan_set_prefetch_fraction(skg_plan_t plan, double fraction);

/* Copy the plan's launch description into *out. */
SKG_API skg_status skg_plan_info(skg_plan_t plan, skg_plan_desc *out);

/*
 * skg_plan_check -- synchronise the plan's last stream and report whether
 * any of its kernels ran out of a bounded wait since the last check
 * (SKG_ERR_DEVICE_TIMEOUT; the report is then cleared) or a CUDA error is
 * pending (SKG_ERR_CUDA).
 */
SKG_API skg_status skg_plan_check(skg_plan_t plan);

/* Free the plan, its workspace and descriptors (after its work finished). */
SKG_API skg_status skg_plan_destroy(skg_plan_t plan);

/*
 * skg_debug_wait_timeout -- failure-detection self test: launch one CTA that
 * waits on a shared-memory barrier that nothing ever arrives at, bounded by
 * timeout_ns of %globaltimer; on expiry the kernel records the timeout in
 * the plan's error word and returns normally, leaving the context usable.
 * A following skg_plan_check returns SKG_ERR_DEVICE_TIMEOUT.  With plan
 * NULL the timeout is recorded in the word of skg_run_noalloc's fixed array
 * instead, and skg_noalloc_check reports it.
 */
SKG_API skg_status skg_debug_wait_timeout(skg_plan_t plan, unsigned long long timeout_ns,
                                  void *stream);

/*
 * skg_run_noalloc -- the split-K projection (M = 3..64) for callers that may
 * not allocate device memory: runtimes that own the whole device-memory
 * budget, code that must not enter the CUDA allocator, or hosts that cannot
 * create plans (skg_plan allocates).  It takes no plan, allocates nothing, and
 * keeps the kernel's fp32 partials, arrival counters and timeout word in a
 * fixed 16 MiB array inside the library that every GPU loading the library
 * holds until the process exits.  The pages describe no such entry point; it
 * exists only for these callers.
 *   M, N, K, epilogue, x, W, residual, y, stream: as for skg_plan + skg_run.
 *   Limits: M must be 3..64 (M <= 2 needs no scratch: use skg_run); the
 *   partials at the picker's split, split * ceil(N/128) * 128 * M * 4 bytes,
 *   must fit 16 MiB - 64 KiB - 256 bytes, else SKG_ERR_UNSUPPORTED (at
 *   M = 64 that admits N up to 32512, where the picker splits K in 2).
 *   The first call on each device resolves the array's device address
 *   (cudaGetSymbolAddress) and keeps it for the life of the process: make
 *   that first call before any stream capture, and do not reset the device
 *   (cudaDeviceReset) after it.
 *   Every call clears the counters (cudaMemsetAsync on `stream`) and then
 *   launches one kernel, with the same L2 look-ahead as the plan path;
 *   results are bit-identical to skg_run's.  All calls share the one array,
 *   so calls that overlap on the GPU (other streams, or other threads) race:
 *   serialise them.  A bounded wait that runs out stops the kernel, leaves y
 *   incomplete and sets the array's timeout word, which skg_noalloc_check
 *   reports.
 * Errors: as skg_run, except that an earlier timeout is reported only by
 * skg_noalloc_check.
 */
SKG_API skg_status skg_run_noalloc(int M, int N, int K, int epilogue, const void *x, const void *W,
                                   const void *residual, void *y, void *stream);

/*
 * skg_noalloc_check -- synchronise `stream`, then report whether any kernel
 * launched by skg_run_noalloc on the current device ran out of a bounded
 * wait since the last check (SKG_ERR_DEVICE_TIMEOUT: the output of that call
 * is incomplete; the word is then cleared), or a CUDA error is pending
 * (SKG_ERR_CUDA).  Allocates nothing (a 4-byte device-to-host copy and, after
 * a timeout, a 4-byte clear).
 */
SKG_API skg_status skg_noalloc_check(void *stream);

/* Message of the last failed call on this thread ("" if none). */
SKG_API const char *skg_last_error(void);

/* SKG_VERSION of the loaded library. */
SKG_API int skg_version(void);

/*
 * Groups -- several projections of the same M (1..64) in one persistent
 * split-K launch.  [OC] fuses producer and consumer in one kernel across
 * GPUs; this is the one-GPU form of that idea: the launch's CTAs take the
 * work units (projection, 128-row tile, split) from a counter in projection
 * order (so the launch completes with any part of its grid resident), keep
 * their TMA ring, TMEM and barriers from one unit to the next, and stream
 * the next projection's weights while the previous one is still being
 * reduced, so consecutive projections pay no launch head or tail between
 * them.  Each projection's output has the bits of skg_run on the split-K
 * kernel at the same split (splits above 8 are lowered to 8: any split gives
 * the same bits; at M <= 2 that is the plan after
 * skg_plan_force_kernel(SKG_KERNEL_SPLITK_TC)).
 *
 * skg_group -- plan n (1..8) projections: N[i], K[i] and epilogue[i] as for
 * skg_plan; dep[i] (i >= 1; dep may be NULL for none) = 1: projection i
 * reads its x and residual only after projection i - 1 has written all of
 * its y (an on-device counter, bounded wait) -- set it whenever projection
 * i consumes projection i - 1's output.  Projections without dep read their
 * inputs with no ordering against the rest of the group, so their x,
 * residual and y must not be written by another projection of the group.
 * Projection 0 reads x only after the previous kernel in the stream
 * (programmatic dependent launch, as skg_run).  Allocates the partials and
 * counters of every projection.  Errors: SKG_ERR_INVALID_ARG,
 * SKG_ERR_UNSUPPORTED (n, M or a shape outside the limits), SKG_ERR_CUDA.
 */
typedef struct skg_group_s *skg_group_t;
SKG_API skg_status skg_group(int n, int M, const int *N, const int *K, const int *epilogue, const int *dep,
                             skg_group_t *out);

/*
 * skg_group_run -- enqueue the group on `stream`: x[i] bf16 [M, K[i]], W[i]
 * bf16 [N[i], K[i]], residual[i] bf16 [M, N[i]] or NULL (the residual array
 * itself may be NULL when no epilogue takes one), y[i] [M, N[i]] bf16 (fp32
 * for SKG_EPI_FP32); x[i] and W[i] 16-byte aligned.  Allocates nothing.
 * One run of a group may be in flight at a time.  After a device timeout
 * (SKG_ERR_DEVICE_TIMEOUT from a later run or skg_group_check) the group's
 * counters are inconsistent: destroy it.
 */
SKG_API skg_status skg_group_run(skg_group_t group, const void *const *x, const void *const *W,
                                 const void *const *residual, void *const *y, void *stream);

/* Launch shape: CTAs, ring stages, work units, and each projection's split (n ints). */
SKG_API skg_status skg_group_info(skg_group_t group, int *grid, int *stages, int *units, int *split);

/* Synchronize the group's last stream and report a device timeout, if any. */
SKG_API skg_status skg_group_check(skg_group_t group);

/* Free the group (after its work finished). */
SKG_API skg_status skg_group_destroy(skg_group_t group);

#ifdef __cplusplus
}
#endif

#endif /* SKG_H */
