// skg_splitk_tc.cu -- the split-K tensor-core projection kernel for M > 2.
//
// "Hyper Optimizing Kimi K3 in vLLM: Moving Fast and Responsibly", method
// details 1 "Tune shapes for the workload": at larger batch the projections
// switch to split-K, spreading the reduction dimension over more workers;
// method details 2: the output projection is fused with the residual add.
//
// Design for sm_103a (swap-AB): the 128 W rows of an output tile are the MMA
// M dimension, and the M <= 64 decode tokens, padded to m_pad = 16/32/48/64,
// are the MMA N dimension, so nothing is padded to 128.  Per CTA:
//   warp 0      TMA producer: W tile [128 x 64] (L2 evict-first) and x tile
//               [m_pad x 64] (rows >= M zero-filled by TMA) into a ring of
//               shared-memory stages, 128-byte swizzled;
//   warp 1      TMEM owner and MMA issuer: one thread issues
//               tcgen05.mma.kind::f16 (bf16 x bf16 -> fp32) into one of two
//               TMEM accumulators [128 lanes x m_pad columns];
//   warps 2..9  epilogue: tcgen05.ld the finished accumulator, combine it in
//               registers, and finally run the split reduction and output.
//
// Reduction order (fixed): K is cut into 16 canonical chunks of 64-wide
// k-blocks.  Each chunk is summed by the MMA from a fresh accumulator; chunk
// sums are combined by one balanced binary tree (empty chunks skipped).  The
// S CTAs of a tile each own an aligned subtree of 16/S chunks and write its
// value to the plan's fp32 workspace; the last CTA to arrive (an atomic
// counter picks it) combines the S values by the top levels of the same
// tree, in index order, adds the residual in fp32, rounds once to bf16 and
// writes y.  With R > 1 reducers per tile, the last R arrivals each wait
// for the others and combine a 1/R share of the tile's outputs the same way.  Every allowed S gives the same
// bits, and the arrival order never changes them.
//
// Ordering rule of the pages (background 2, the activation read hoisted above
// a synchronisation wait): under programmatic dependent launch only W tiles
// are requested before griddepcontrol.wait; x, residual, workspace, counters
// and y are touched only after it.
//
// Every wait is bounded (%globaltimer); on expiry a thread records the
// timeout in the plan's error word, raises the CTA's abort flag, drains its
// own asynchronous copies / MMAs, and the CTA frees its TMEM and returns.
#include <cuda_bf16.h>

#include <algorithm>
#include <mutex>

#include "skg_internal.h"
#include "skg_ptx.cuh"

namespace skg {
namespace {

#include "skg_tc_common.cuh"

// A reducer that is not the tile's last arrival: poll the tile's counter
// (acquire, GPU scope) until all `target` arrivals are in, for at most
// timeout_ns, or until another role of the CTA gave up.  Every CTA arrives
// before it waits, so a waiter waits only for CTAs that never wait; the host
// allows R > 1 reducers per tile only while the whole grid is one wave of
// the CTAs the SMs hold at once, so the waiters, tiles x (R - 1), are fewer
// than the slots and a CTA waited for always finds one.
__device__ __forceinline__ bool wait_arrivals(const unsigned *ctr, unsigned target, uint64_t timeout_ns,
                                              volatile int *abort)
{
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        unsigned v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
        if ((v & 0xFFFFu) >= target)
            return true;
        if (*abort || globaltimer_ns() - t0 > timeout_ns)
            return false;
        __nanosleep(32);
    }
}

// Several CTAs share an SM (a short ring each): <= 102 registers per thread
// for m_pad 48/64 (2 CTAs per SM), <= 68 for m_pad 16/32 (3 CTAs per SM).
template <int MPAD>
__global__ void __launch_bounds__(kTcThreads, (MPAD <= 32) ? 3 : 2)
splitk_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                 const TcParams p)
{
    using Sh = TcShape<MPAD>;
    constexpr int NC = Sh::kNC;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);

    const int S = p.stages;
    uint8_t *sW = smem;
    uint8_t *sX = smem + S * kWBytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(sX + S * Sh::kXBytes);
    uint64_t *empty = full + S;
    uint64_t *tfull = empty + S;      // [2]
    uint64_t *tempty = tfull + 2;     // [2]
    uint64_t *drain = tempty + 2;     // [1]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *flags = reinterpret_cast<volatile int *>(tmem_slot + 1);  // [0] abort, [1] last

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = blockIdx.x % p.n_tiles;
    const int split = blockIdx.x / p.n_tiles;
    // This launch covers canonical chunks [chunk_base, chunk_base +
    // chunk_count) of K (all 16 unless K is sharded across ranks, when x and
    // W hold only those chunks' columns): CTA `split` owns an aligned subtree
    // of L of them.
    const int L = p.chunk_count / p.split;
    const int leaf0 = p.chunk_base + split * L;
    const int total_present = min(chunks_present(p.nkb), p.chunk_base + p.chunk_count);
    const int present = max(0, min(L, total_present - leaf0));
    const int kb_begin = chunk_begin(leaf0, p.nkb) - chunk_begin(p.chunk_base, p.nkb);   // in the shard
    const int nk = chunk_begin(leaf0 + present, p.nkb) - chunk_begin(leaf0, p.nkb);

    if (threadIdx.x == 0) {
        tma_prefetch_desc(&tmW);
        tma_prefetch_desc(&tmX);
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], kEpiThreads / 32);
        }
        mbar_init(drain, 1);
        flags[0] = 0;
        flags[1] = 0;
        fence_mbar_init();
    }
    // The producer starts as soon as the barriers exist; the MMA and
    // epilogue warps meet again (named barrier 2) once warp 1 has allocated
    // TMEM.  A CTA that starts late, as the previous kernel's CTAs leave,
    // so requests its first weight tiles without waiting for the allocation
    // (measured on GB300: the batch sweep's step 136.4 -> 134.0 us).
    __syncthreads();
    pdl_launch_dependents();
    uint32_t tmem_base = 0;
    if (warp != 0) {
        if (warp == 1) {
            tmem_alloc(tmem_slot, Sh::kTmemCols);
            tmem_relinquish();
        }
        tc_fence_before();
        asm volatile("bar.sync 2, 288;" ::: "memory");   // warps 1..9
        tc_fence_after();
        tmem_base = *tmem_slot;
    }

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0 && nk > 0) {
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_x = policy_evict_last();
            const int pre = nk < S ? nk : S;
            for (int i = 0; i < pre; ++i) {
                mbar_arrive_expect_tx(&full[i], kWBytes + Sh::kXBytes);
                tma_load_2d(sW + i * kWBytes, &tmW, &full[i], (kb_begin + i) * kBlockK,
                            tile * kTileN, pol_w);
            }
            // While the previous kernel finishes, the `ahead` W tiles after the
            // ring are requested into L2 too (weights only: allowed before the
            // wait below), so its tail keeps HBM busy with this launch's bytes.
            for (int i = pre; i < nk && i < pre + p.ahead; ++i)
                tma_prefetch_l2_2d(&tmW, (kb_begin + i) * kBlockK, tile * kTileN);
            pdl_wait();  // activations only from here on
            for (int i = 0; i < pre; ++i)
                tma_load_2d(sX + i * Sh::kXBytes, &tmX, &full[i], (kb_begin + i) * kBlockK, 0, pol_x);
            int issued = pre;
            // Steady state: wait until `burst` consecutive ring slots are free,
            // then request their k-blocks back to back, so the bytes of each
            // W row arrive at the memory system together.
            const int burst = p.burst < 1 ? 1 : (p.burst > S ? S : p.burst);
            bool ok = true;
            for (int i = pre; i < nk && ok; i += burst) {
                const int nb = (nk - i) < burst ? (nk - i) : burst;
                for (int j = 0; j < nb; ++j) {
                    const int s = (i + j) % S;
                    const uint32_t ph = ((i + j) / S) & 1;
                    if (!mbar_wait(&empty[s], ph ^ 1, p.timeout_ns, &flags[0])) {
                        record_failure(p, &flags[0], kErrTimeoutProducer);
                        ok = false;
                        break;
                    }
                }
                if (!ok)
                    break;
                for (int j = 0; j < nb; ++j) {
                    const int s = (i + j) % S;
                    mbar_arrive_expect_tx(&full[s], kWBytes + Sh::kXBytes);
                    tma_load_2d(sW + s * kWBytes, &tmW, &full[s], (kb_begin + i + j) * kBlockK,
                                tile * kTileN, pol_w);
                    tma_load_2d(sX + s * Sh::kXBytes, &tmX, &full[s], (kb_begin + i + j) * kBlockK, 0, pol_x);
                }
                issued = i + nb;
            }
            // Every weight tile of this CTA is requested: use the rest of the
            // launch to ask the L2 for this CTA's slice of the next
            // projection's weight.
            prefetch_next_slice(p.next_w, p.next_bytes, blockIdx.x, gridDim.x, policy_evict_last());
            if (flags[0]) {
                // Abort: let every copy this thread issued land before exit.
                for (int s = 0; s < S && s < issued; ++s) {
                    const int last = s + S * ((issued - 1 - s) / S);
                    volatile int never = 0;
                    mbar_wait(&full[s], (last / S) & 1, p.timeout_ns, &never);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0 && present > 0) {
            bool ok = true;
            int i = 0;
            for (int pl = 0; pl < present && ok; ++pl) {
                const int b = pl & 1;
                const uint32_t u = static_cast<uint32_t>(pl >> 1);
                if (!mbar_wait(&tempty[b], (u & 1) ^ 1, p.timeout_ns, &flags[0])) {
                    record_failure(p, &flags[0], kErrTimeoutMma);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + static_cast<uint32_t>(b * MPAD);
                const int kb0 = chunk_begin(leaf0 + pl, p.nkb);
                const int kb1 = chunk_begin(leaf0 + pl + 1, p.nkb);
                for (int kb = kb0; kb < kb1; ++kb, ++i) {
                    const int s = i % S;
                    const uint32_t ph = (i / S) & 1;
                    if (!mbar_wait(&full[s], ph, p.timeout_ns, &flags[0])) {
                        record_failure(p, &flags[0], kErrTimeoutMma);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = smem_desc_kmajor_sw128(smem_u32(sW + s * kWBytes));
                    const uint64_t bd = smem_desc_kmajor_sw128(smem_u32(sX + s * Sh::kXBytes));
#pragma unroll
                    for (int kk = 0; kk < kBlockK / 16; ++kk)
                        tc_mma_bf16(d, ad + 2 * kk, bd + 2 * kk, Sh::kIdesc,
                                    (kb > kb0 || kk > 0) ? 1u : 0u);
                    tc_commit(&empty[s]);
                }
                if (ok)
                    tc_commit(&tfull[b]);
            }
            if (!ok) {
                // Abort: wait for the MMAs already issued before TMEM is freed.
                tc_commit(drain);
                volatile int never = 0;
                mbar_wait(drain, 0, p.timeout_ns, &never);
            }
        }
    } else {
        // ------------------------------------------------ epilogue
        pdl_wait();  // residual, workspace, counters and y only from here on
        const int ew = warp - 2;
        const int quarter = warp & 3;   // TMEM lanes this warp may access
        const int half = ew >> 2;       // which half of the m_pad columns
        const int row = quarter * 32 + lane;
        const int n = tile * kTileN + row;
        // this thread's columns: accumulator buffer b, and tree levels 1, 2
        const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                   static_cast<uint32_t>(half * NC);
        const uint32_t lvl1 = lane_base + 2 * MPAD;
        const uint32_t lvl2 = lane_base + 3 * MPAD;
        float st0[NC], cur[NC];
        bool ok = true;
        // Canonical tree over this CTA's chunks, as a binary counter: chunk
        // pl closes the blocks of 2, 4 and 8 chunks that end with it.  Level
        // 0 waits in registers, levels 1 and 2 in spare TMEM columns.  After
        // the last chunk cur holds the block of the lowest set bit of
        // `present`; only blocks that a later chunk still needs are stored.
        for (int pl = 0; pl < present; ++pl) {
            const int b = pl & 1;
            const uint32_t u = static_cast<uint32_t>(pl >> 1);
            if (!mbar_wait(&tfull[b], u & 1, p.timeout_ns, &flags[0])) {
                record_failure(p, &flags[0], kErrTimeoutEpilogue);
                ok = false;
                break;
            }
            tc_fence_after();
            tmem_load_cols<NC>(lane_base + static_cast<uint32_t>(b * MPAD), cur);
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&tempty[b]);
            const bool more = pl + 1 < present;
            if (pl & 1) {
#pragma unroll
                for (int c = 0; c < NC; ++c) cur[c] = st0[c] + cur[c];
                if (pl & 2) {
                    tmem_add_cols<NC>(lvl1, cur);
                    if (pl & 4)
                        tmem_add_cols<NC>(lvl2, cur);
                    else if (more)
                        tmem_store_cols<NC>(lvl2, cur);
                } else if (more) {
                    tmem_store_cols<NC>(lvl1, cur);
                }
            } else if (more) {
#pragma unroll
                for (int c = 0; c < NC; ++c) st0[c] = cur[c];
            }
        }
        ok = epi_bar_and(ok && !flags[0]);
        if (ok) {
            // The subtree's value: the stored larger blocks folded onto cur,
            // smallest first (the left operand is the earlier block).
            const int low = present & -present;
            if ((present & 2) && low < 2)
                tmem_add_cols<NC>(lvl1, cur);
            if ((present & 4) && low < 4)
                tmem_add_cols<NC>(lvl2, cur);
            if (present > 0 && n < p.N) {
#pragma unroll
                for (int c = 0; c < NC; ++c) {
                    const int m = half * NC + c;
                    if (m < p.M)
                        p.ws[((static_cast<size_t>(split) * p.n_tiles + tile) * p.M + m) * kTileN + row] = cur[c];
                }
            }
            // Arrive on the tile's counter: the barrier orders every epilogue
            // thread's partial stores before one thread's acq_rel atomic at GPU
            // scope; the last arriver's acquire, passed on by the next
            // barrier, orders its reads of all partials after the stores.
            epi_bar_sync();
            // The last R arrivals of the tile share its reduction: each waits
            // (bounded) until every arrival is in, then reduces its share of
            // the tile's outputs.  Splits of 16 reduce in one CTA.
            const int R = p.split <= 8 ? max(1, min(p.reducers, p.split)) : 1;
            if (ew == 0 && lane == 0) {
                // Low 16 bits of the tile's counter: arrivals; high bits:
                // reducers that have seen every arrival.
                const int old = static_cast<int>(atom_add_acq_rel_gpu(&p.counters[tile], 1u) & 0xFFFFu);
                const int first = p.split - R;
                int role = 0;   // 1 + this CTA's share of the reduction; 0: none
                if (old >= first) {
                    if (old == p.split - 1 ||
                        wait_arrivals(&p.counters[tile], static_cast<unsigned>(p.split), p.timeout_ns, &flags[0]))
                        role = old - first + 1;
                    else
                        record_failure(p, &flags[0], kErrTimeoutEpilogue);
                }
                if (role && R > 1) {
                    // the last reducer to see every arrival returns the
                    // counter to zero: no one polls it any more
                    if ((atom_add_acq_rel_gpu(&p.counters[tile], 1u << 16) >> 16) == static_cast<unsigned>(R - 1))
                        p.counters[tile] = 0;
                } else if (role) {
                    p.counters[tile] = 0;
                }
                flags[1] = role;
            }
            epi_bar_sync();
            const int role = flags[1];
            if (role) {
                const int sp = (total_present - p.chunk_base + L - 1) / L;  // splits holding a value
                const int et = threadIdx.x - 64;
                // work items: 4 rows of one column m; share r of R takes
                // whole columns [r * ceil(M / R), (r + 1) * ceil(M / R))
                const int items = p.M * (kTileN / 4);
                const int share = (p.M + R - 1) / R * (kTileN / 4);
                const int i0 = min(items, (role - 1) * share);
                const int i1 = min(items, role * share);
                constexpr int kL = MPAD <= 32 ? 8 : 16;   // 16-byte loads in flight per thread
                switch (p.split) {
                case 2: reduce_tile_v4<2, kL>(p, tile, sp, et, i0, i1); break;
                case 4: reduce_tile_v4<4, kL>(p, tile, sp, et, i0, i1); break;
                case 8: reduce_tile_v4<8, kL>(p, tile, sp, et, i0, i1); break;
                default:
                    if (n < p.N)
                        reduce_tile<16, NC>(p, tile, row, half, sp);
                    break;
                }
            }
        }
    }

    // Lane 0 of the producer and MMA warps ran their roles alone: reconverge
    // each warp before the CTA barrier, so every warp arrives whole and TMEM
    // is freed only after every role is done.
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, Sh::kTmemCols);
    }
}

// The kernel's shared-memory attributes, set once per device before its
// first launch or occupancy query.
template <int MPAD>
cudaError_t set_tc_attrs()
{
    static int attr_set[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    if (__atomic_load_n(&attr_set[dev], __ATOMIC_ACQUIRE) == 0) {
        e = cudaFuncSetAttribute(splitk_tc_kernel<MPAD>, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
        if (e != cudaSuccess)
            return e;
        e = cudaFuncSetAttribute(splitk_tc_kernel<MPAD>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess)
            return e;
        __atomic_store_n(&attr_set[dev], 1, __ATOMIC_RELEASE);
    }
    return cudaSuccess;
}

// CTAs of one launch shape an SM holds at once, from the kernel's
// registers, shared memory, threads and TMEM columns.  Measured on GB300:
// cudaOccupancyMaxActiveBlocksPerMultiprocessor answers 1 for this kernel at
// every shape, while the profiler's launch statistics show 2 CTAs per SM at
// m_pad 64 (register and shared-memory limits both 2), so the limits are
// taken here one by one.
template <int MPAD>
cudaError_t occupancy_tc(int stages, int *ctas_per_sm)
{
    cudaError_t e = set_tc_attrs<MPAD>();
    if (e != cudaSuccess)
        return e;
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, splitk_tc_kernel<MPAD>);
    if (e != cudaSuccess)
        return e;
    int dev = 0, regs_sm = 0, smem_sm = 0, smem_rsv = 0, threads_sm = 0, blocks_sm = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&smem_rsv, cudaDevAttrReservedSharedMemoryPerBlock, dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&threads_sm, cudaDevAttrMaxThreadsPerMultiProcessor, dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&blocks_sm, cudaDevAttrMaxBlocksPerMultiprocessor, dev);
    if (e != cudaSuccess)
        return e;
    constexpr int kWarps = kTcThreads / 32;
    // registers: allocated per warp in units of 256, each of the SM's four
    // schedulers holding a quarter of the file and of the warps
    const int regs_warp = (fa.numRegs * 32 + 255) / 256 * 256;
    const int by_regs = regs_warp > 0 ? (regs_sm / 4 / regs_warp) * 4 / kWarps : blocks_sm;
    const int by_smem = smem_sm / (tc_smem_bytes(MPAD, stages) + smem_rsv);
    const int by_threads = threads_sm / kTcThreads;
    const int by_tmem = kTmemColsPerSm / static_cast<int>(TcShape<MPAD>::kTmemCols);
    *ctas_per_sm = std::max(0, std::min(std::min(by_regs, by_smem), std::min(std::min(by_threads, by_tmem), blocks_sm)));
    return cudaSuccess;
}

template <int MPAD>
cudaError_t launch_tc(const CUtensorMap &tmW, const CUtensorMap &tmX, const TcParams &p, int grid,
                      bool pdl, cudaStream_t s)
{
    const int smem = tc_smem_bytes(MPAD, p.stages);
    const cudaError_t e = set_tc_attrs<MPAD>();
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, splitk_tc_kernel<MPAD>, tmW, tmX, p);
}

} // namespace

int tc_smem_bytes(int m_pad, int stages)
{
    // 1 KB alignment slack + stages * (W tile + x tile) + barriers and flags
    return 1024 + stages * (static_cast<int>(kWBytes) + m_pad * kBlockK * 2) + 8 * (2 * stages + 5) + 16;
}

int tc_tmem_cols(int m_pad)
{
    int c = 32;
    while (c < 4 * m_pad)
        c *= 2;
    return c;
}

int tc_max_stages(int m_pad, int smem_limit)
{
    int s = 16;
    while (s > 2 && tc_smem_bytes(m_pad, s) > smem_limit)
        --s;
    return s;
}

cudaError_t tc_occupancy(int m_pad, int stages, int *ctas_per_sm)
{
    switch (m_pad) {
    case 16: return occupancy_tc<16>(stages, ctas_per_sm);
    case 32: return occupancy_tc<32>(stages, ctas_per_sm);
    case 48: return occupancy_tc<48>(stages, ctas_per_sm);
    case 64: return occupancy_tc<64>(stages, ctas_per_sm);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_splitk_tc(const CUtensorMap &tmW, const CUtensorMap &tmX, const TcParams &p,
                             int m_pad, int grid, bool pdl, cudaStream_t s)
{
    switch (m_pad) {
    case 16: return launch_tc<16>(tmW, tmX, p, grid, pdl, s);
    case 32: return launch_tc<32>(tmW, tmX, p, grid, pdl, s);
    case 48: return launch_tc<48>(tmW, tmX, p, grid, pdl, s);
    case 64: return launch_tc<64>(tmW, tmX, p, grid, pdl, s);
    default: return cudaErrorInvalidValue;
    }
}

} // namespace skg

// ---------------------------------------------------------------------------
// Scratch-free entry point.
//
// A caller that may not allocate device memory (a runtime that owns the
// whole memory budget, code running where the CUDA allocator must not be
// entered, or a host that cannot create plans because plans allocate) can
// still run the split-K kernel: its fp32 partials, arrival counters and
// timeout word live in the fixed array below, which every GPU that loads
// this library holds until the process exits.
//
// Layout of the array: [0, 256) the timeout word (first 4 bytes) that the
// kernels' bounded waits set and skg_noalloc_check reads and clears;
// [256, 256 + 64 KiB) one arrival counter per 128-row tile; the rest, fp32
// partials [split][tile][M][128].
// ---------------------------------------------------------------------------
namespace skg {
namespace {

constexpr size_t kScratchBytes = static_cast<size_t>(16) << 20;  // 16 MiB
constexpr size_t kScratchErrBytes = 256;
constexpr int kScratchTiles = 16384;                              // counters: N <= 2,097,152
constexpr size_t kScratchCounterBytes = kScratchTiles * sizeof(unsigned int);
constexpr size_t kScratchPartialBytes = kScratchBytes - kScratchErrBytes - kScratchCounterBytes;

static __device__ __align__(256) unsigned char g_splitk_scratch[kScratchBytes];

std::mutex g_scratch_mutex;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of g_splitk_scratch on the current device, looked up once
// per device (the host-side name is only a stand-in for the symbol).  The
// address is kept for the life of the process: a cudaDeviceReset after the
// first call on a device is not supported.
skg_status scratch_address(void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return set_error(SKG_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev >= kMaxDevices)
        return set_error(SKG_ERR_UNSUPPORTED, "device %d beyond %d", dev, kMaxDevices);
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_splitk_scratch);
        if (e != cudaSuccess || !ptr)
            return set_error(SKG_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
    return SKG_OK;
}

} // namespace

skg_status noalloc_error_word(unsigned int **out)
{
    void *scratch = nullptr;
    const skg_status st = scratch_address(&scratch);
    if (st == SKG_OK)
        *out = static_cast<unsigned int *>(scratch);
    return st;
}

} // namespace skg

extern "C" skg_status skg_run_noalloc(int M, int N, int K, int epilogue, const void *x, const void *W,
                                      const void *residual, void *y, void *stream)
{
    using namespace skg;
    void *scratch = nullptr;
    skg_status st = scratch_address(&scratch);
    if (st != SKG_OK)
        return st;
    CUtensorMap tmW, tmX;
    TcParams t;
    int m_pad = 0, grid = 0;
    st = prepare_splitk_launch(M, N, K, epilogue, x, W, residual, y, kScratchPartialBytes, kScratchTiles, &tmW,
                               &tmX, &t, &m_pad, &grid);
    if (st != SKG_OK)
        return st;
    unsigned char *base = static_cast<unsigned char *>(scratch);
    t.err = reinterpret_cast<unsigned int *>(base);
    t.counters = reinterpret_cast<unsigned int *>(base + kScratchErrBytes);
    t.ws = reinterpret_cast<float *>(base + kScratchErrBytes + kScratchCounterBytes);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // The array keeps the previous call's contents: the counters must start at
    // zero (the timeout word is left for skg_noalloc_check).
    cudaError_t e = cudaMemsetAsync(t.counters, 0, static_cast<size_t>(t.n_tiles) * sizeof(unsigned int), s);
    if (e == cudaSuccess)
        e = launch_splitk_tc(tmW, tmX, t, m_pad, grid, false, s);
    if (e != cudaSuccess)
        return set_error(SKG_ERR_CUDA, "skg_run_noalloc launch: %s", cudaGetErrorString(e));
    return SKG_OK;
}

extern "C" skg_status skg_noalloc_check(void *stream)
{
    using namespace skg;
    void *scratch = nullptr;
    skg_status st = scratch_address(&scratch);
    if (st != SKG_OK)
        return st;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return set_error(SKG_ERR_CUDA, "skg_noalloc_check synchronize: %s", cudaGetErrorString(e));
    unsigned int w = 0;
    e = cudaMemcpy(&w, scratch, sizeof w, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && w != 0)
        e = cudaMemset(scratch, 0, sizeof w);
    if (e != cudaSuccess)
        return set_error(SKG_ERR_CUDA, "skg_noalloc_check: %s", cudaGetErrorString(e));
    if (w != 0)
        return set_error(SKG_ERR_DEVICE_TIMEOUT,
                         "a kernel of skg_run_noalloc ran out of a bounded wait (bits 0x%x); its output is incomplete",
                         w);
    return SKG_OK;
}
