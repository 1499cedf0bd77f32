// skg_group_tc.cu -- several projections of the same M in one persistent
// split-K launch.
//
// The split-K kernel (skg_splitk_tc.cu) pays, per launch, the latency of its
// first weight bytes and the tail of its last reductions; programmatic
// dependent launch hides part of that between launches.  Here one launch
// runs a list of projections.  The work units (projection, 128-row tile,
// split) are numbered projection by projection, and a CTA takes the next
// unit from a global counter whenever its producer is ready for one.  The
// TMA ring, the two TMEM accumulators and every barrier carry on from one
// unit to the next, so the producer streams the next unit's weights while
// the epilogue still reduces the previous one.  (The single-GPU analogue of
// fusing producer and consumer in one kernel: "Hyper Optimizing Kimi K3 in
// vLLM: Moving Fast and Responsibly", method details 2.)
//
// Dependencies: projection j with dep set reads its x (and residual) only
// after every tile of projection j - 1 has been written.  The last CTA of a
// tile adds one to done[j] (release) after its y stores; a producer holding
// a unit of projection j requests its first weight tiles, then waits
// (bounded) until done[j - 1] covers all of its tiles (acquire), then loads
// x.  Units are handed out in projection order, so every unit of projection
// j - 1 already belongs to a running CTA, and that CTA waits on nothing
// later: the launch completes whatever part of the grid is resident.  (A
// fixed assignment of units to CTAs would need the whole grid resident at
// once, which kernels still running on the SMs can prevent.)  The last CTA
// to finish returns done[] and the unit counter to zero.
//
// Arithmetic: per unit exactly that of the one-projection kernel (canonical
// chunks, the same tree, the same last-CTA reduction), so every projection's
// output has the bits of skg_run at the same split, whichever CTA ran which
// unit.
//
// Ordering rule of the pages (background 2): weights may be requested before
// griddepcontrol.wait or a dependency wait; the unit counter, x, residual,
// workspace, counters and y only after.  Every wait is bounded; a timeout
// records an error bit, raises the CTA's abort flag, drains the CTA's own
// copies and MMAs, and the CTA frees its TMEM and returns (the group then
// reports the error and must be destroyed: its counters are no longer
// consistent).
#include <cuda_bf16.h>

#include <algorithm>

#include "skg_internal.h"
#include "skg_ptx.cuh"

namespace skg {
namespace {

#include "skg_tc_common.cuh"

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned *ptr)
{
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
    return v;
}

__device__ __forceinline__ void red_release_gpu_add(unsigned *ptr, unsigned v)
{
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" :: "l"(ptr), "r"(v) : "memory");
}

// Wait until *ctr >= target; false on timeout or when another role aborted.
__device__ bool wait_counter(const unsigned *ctr, unsigned target, unsigned long long timeout_ns,
                             volatile int *abort)
{
    if (ld_acquire_gpu(ctr) >= target)
        return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        __nanosleep(128);
        if (ld_acquire_gpu(ctr) >= target)
            return true;
        if (*abort)
            return false;
        if (globaltimer_ns() - t0 > timeout_ns)
            return false;
    }
}

__device__ __forceinline__ void group_failure(const GroupParams &g, volatile int *abort, unsigned bit)
{
    *abort = 1;
    if (g.err)
        atomicOr(g.err, bit);
}

// Work unit k of projection j: its tile and split, and the split's k-blocks.
struct Unit {
    int j, tile, split, leaf0, present, kb_begin, nk;
};

__device__ __forceinline__ Unit unit_at(const GroupParams &g, int j, int k)
{
    Unit r;
    const GroupProj &P = g.proj[j];
    r.j = j;
    r.tile = k % P.n_tiles;
    r.split = k / P.n_tiles;
    const int L = kChunks / P.split;
    r.leaf0 = r.split * L;
    r.present = max(0, min(L, chunks_present(P.nkb) - r.leaf0));
    r.kb_begin = chunk_begin(r.leaf0, P.nkb);
    r.nk = chunk_begin(r.leaf0 + r.present, P.nkb) - r.kb_begin;
    return r;
}

// Unit u of the launch (projection by projection).
__device__ __forceinline__ Unit unit_of(const GroupParams &g, int u)
{
    int j = 0;
    while (j + 1 < g.n && u >= g.proj[j + 1].unit_begin)
        ++j;
    return unit_at(g, j, u - g.proj[j].unit_begin);
}

// The last CTA's reduction of a tile, as in the one-projection kernel, with
// 4 loads in flight per thread (the unit loop keeps more registers live;
// 8 or 16, as there, measured slower here).
template <int MPAD>
__device__ __forceinline__ void group_reduce(const GroupProj *P, int tile, int sp, int et, int i0, int i1)
{
    switch (P->split) {
    case 2: reduce_tile_v4<2, 4>(*P, tile, sp, et, i0, i1); break;
    case 4: reduce_tile_v4<4, 4>(*P, tile, sp, et, i0, i1); break;
    default: reduce_tile_v4<8, 4>(*P, tile, sp, et, i0, i1); break;
    }
}

template <int MPAD>
__global__ void __launch_bounds__(kTcThreads, (MPAD <= 32) ? 3 : 2) splitk_group_kernel(const __grid_constant__ GroupParams g)
{
    using Sh = TcShape<MPAD>;
    constexpr int NC = Sh::kNC;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);

    const int S = g.stages;
    uint8_t *sW = smem;
    uint8_t *sX = smem + S * kWBytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(sX + S * Sh::kXBytes);
    uint64_t *empty = full + S;
    uint64_t *tfull = empty + S;      // [2]
    uint64_t *tempty = tfull + 2;     // [2]
    uint64_t *drain = tempty + 2;     // [1]
    constexpr int Q = kGroupUnitQueue;
    uint64_t *uq_full = drain + 1;    // [Q] unit id written (producer)
    uint64_t *uq_empty = uq_full + Q; // [Q] unit id read (MMA and epilogue)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(uq_empty + Q);
    volatile int *flags = reinterpret_cast<volatile int *>(tmem_slot + 1);  // [0] abort, [1] last
    volatile int *uq = flags + 2;     // [Q] unit ids, -1 = no more units

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int j = 0; j < g.n; ++j) {
            tma_prefetch_desc(&g.proj[j].tmW);
            tma_prefetch_desc(&g.proj[j].tmX);
        }
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], kEpiThreads / 32);
        }
        mbar_init(drain, 1);
        for (int i = 0; i < Q; ++i) {
            mbar_init(&uq_full[i], 1);
            mbar_init(&uq_empty[i], 2);
        }
        flags[0] = 0;
        flags[1] = 0;
        fence_mbar_init();
    }
    // As in the one-projection kernel: the producer starts once the
    // barriers exist, the MMA and epilogue warps once TMEM is allocated.
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
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_x = policy_evict_last();
            int it = 0;                   // ring stages issued so far (all units)
            bool ok = true;
            int x_ready = 0;              // projections < x_ready may have x read
            auto slot_free = [&](int k) {
                return k < S || mbar_wait(&empty[k % S], ((k / S) & 1) ^ 1, g.timeout_ns, &flags[0]);
            };
            // Until the previous grid completes: with no dependencies in the
            // group nothing ever waits for another CTA's unit, so CTA c owns
            // unit c outright and fills its ring with that unit's weights (as
            // the one-projection kernel does); otherwise every unit comes from
            // the counter, and the CTA only warms L2 with the first tiles of
            // unit c (units 0 .. grid - 1 go out first, in whatever order the
            // CTAs arrive).
            const bool own_first = g.static_first != 0;
            int armed0 = 0;
            if (static_cast<int>(blockIdx.x) < g.units) {
                const Unit U0 = unit_of(g, blockIdx.x);
                const GroupProj &P0 = g.proj[U0.j];
                const int pre0 = own_first ? (U0.nk < S ? U0.nk : S) : 0;
                for (; armed0 < pre0; ++armed0) {       // every slot is free at the start
                    mbar_arrive_expect_tx(&full[armed0], kWBytes + Sh::kXBytes);
                    tma_load_2d(sW + armed0 * kWBytes, &P0.tmW, &full[armed0], (U0.kb_begin + armed0) * kBlockK,
                                U0.tile * kTileN, pol_w);
                }
                for (int i = pre0; i < U0.nk && i < pre0 + (own_first ? P0.ahead : S + P0.ahead); ++i)
                    tma_prefetch_l2_2d(&P0.tmW, (U0.kb_begin + i) * kBlockK, U0.tile * kTileN);
            }
            pdl_wait();   // the unit counter and x only from here on
            for (int q = 0; ok; ++q) {
                if (q >= Q && !mbar_wait(&uq_empty[q % Q], ((q / Q) & 1) ^ 1, g.timeout_ns, &flags[0])) {
                    group_failure(g, &flags[0], kErrTimeoutProducer);
                    ok = false;
                    break;
                }
                const unsigned u = (own_first && q == 0)
                                       ? blockIdx.x
                                       : (own_first ? gridDim.x : 0u) + atomicAdd(&g.done[kGroupDoneNext], 1u);
                const bool last = u >= static_cast<unsigned>(g.units);
                uq[q % Q] = last ? -1 : static_cast<int>(u);
                mbar_arrive(&uq_full[q % Q]);
                if (last)
                    break;
                const Unit U = unit_of(g, static_cast<int>(u));
                if (U.nk == 0)
                    continue;
                const GroupProj &P = g.proj[U.j];
                const int tile_row = U.tile * kTileN;
                const int pre = U.nk < S ? U.nk : S;
                // the first weight tiles need no wait (weights are static)
                int armed = (own_first && q == 0) ? armed0 : 0;
                for (; armed < pre; ++armed) {
                    if (!slot_free(it + armed))
                        break;
                    const int s = (it + armed) % S;
                    mbar_arrive_expect_tx(&full[s], kWBytes + Sh::kXBytes);
                    tma_load_2d(sW + s * kWBytes, &P.tmW, &full[s], (U.kb_begin + armed) * kBlockK, tile_row,
                                pol_w);
                }
                if (armed < pre) {
                    group_failure(g, &flags[0], kErrTimeoutProducer);
                    it += armed;      // the drain below waits for these copies
                    ok = false;
                    break;
                }
                if (U.j >= x_ready) {
                    // x of this projection: after the previous projection
                    // when the group says so.  Until then the W tiles past
                    // the ring stream into L2.
                    if (P.dep && U.j > 0) {
                        for (int i = pre; i < U.nk && i < pre + P.ahead; ++i)
                            tma_prefetch_l2_2d(&P.tmW, (U.kb_begin + i) * kBlockK, tile_row);
                        if (!wait_counter(&g.done[U.j - 1], static_cast<unsigned>(g.proj[U.j - 1].n_tiles),
                                          g.timeout_ns, &flags[0])) {
                            group_failure(g, &flags[0], kErrTimeoutProducer);
                            // the W copies above were issued: wait for them below
                            it += pre;
                            ok = false;
                            break;
                        }
                    }
                    // the dependency's y stores are seen before these async-proxy reads
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                    x_ready = U.j + 1;
                }
                for (int i = 0; i < pre; ++i) {
                    const int s = (it + i) % S;
                    tma_load_2d(sX + s * Sh::kXBytes, &P.tmX, &full[s], (U.kb_begin + i) * kBlockK, 0, pol_x);
                }
                it += pre;
                for (int i = pre; i < U.nk; ++i, ++it) {
                    if (!slot_free(it)) {
                        group_failure(g, &flags[0], kErrTimeoutProducer);
                        ok = false;
                        break;
                    }
                    const int s = it % S;
                    mbar_arrive_expect_tx(&full[s], kWBytes + Sh::kXBytes);
                    tma_load_2d(sW + s * kWBytes, &P.tmW, &full[s], (U.kb_begin + i) * kBlockK, tile_row, pol_w);
                    tma_load_2d(sX + s * Sh::kXBytes, &P.tmX, &full[s], (U.kb_begin + i) * kBlockK, 0, pol_x);
                }
            }
            if (flags[0]) {
                // Abort: copies this thread issued land before the CTA exits.
                // (A stage armed for W and x whose x never came cannot
                // complete; its W bytes have landed once the wait times out.)
                for (int s = 0; s < S && s < it; ++s) {
                    const int last = s + S * ((it - 1 - s) / S);
                    volatile int never = 0;
                    mbar_wait(&full[s], (last / S) & 1, g.timeout_ns, &never);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            bool ok = true;
            int it = 0;                   // ring stages consumed (all units)
            int pc = 0;                   // chunks issued (all units): accumulator pc & 1
            for (int qi = 0; ok; ++qi) {
                if (!mbar_wait(&uq_full[qi % Q], (qi / Q) & 1, g.timeout_ns, &flags[0])) {
                    group_failure(g, &flags[0], kErrTimeoutMma);
                    ok = false;
                    break;
                }
                const int u = uq[qi % Q];
                mbar_arrive(&uq_empty[qi % Q]);
                if (u < 0)
                    break;
                const Unit U = unit_of(g, u);
                const int nkb = g.proj[U.j].nkb;
                for (int pl = 0; pl < U.present && ok; ++pl, ++pc) {
                    const int b = pc & 1;
                    const uint32_t q = static_cast<uint32_t>(pc >> 1);
                    if (!mbar_wait(&tempty[b], (q & 1) ^ 1, g.timeout_ns, &flags[0])) {
                        group_failure(g, &flags[0], kErrTimeoutMma);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem_base + static_cast<uint32_t>(b * MPAD);
                    const int kb0 = chunk_begin(U.leaf0 + pl, nkb);
                    const int kb1 = chunk_begin(U.leaf0 + pl + 1, nkb);
                    for (int kb = kb0; kb < kb1; ++kb, ++it) {
                        const int s = it % S;
                        const uint32_t ph = (it / S) & 1;
                        if (!mbar_wait(&full[s], ph, g.timeout_ns, &flags[0])) {
                            group_failure(g, &flags[0], kErrTimeoutMma);
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t ad = smem_desc_kmajor_sw128(smem_u32(sW + s * kWBytes));
                        const uint64_t bd = smem_desc_kmajor_sw128(smem_u32(sX + s * Sh::kXBytes));
#pragma unroll
                        for (int kk = 0; kk < kBlockK / 16; ++kk)
                            tc_mma_bf16(d, ad + 2 * kk, bd + 2 * kk, Sh::kIdesc, (kb > kb0 || kk > 0) ? 1u : 0u);
                        tc_commit(&empty[s]);
                    }
                    if (ok)
                        tc_commit(&tfull[b]);
                }
            }
            if (!ok) {
                // Abort: wait for the MMAs already issued before TMEM is freed.
                tc_commit(drain);
                volatile int never = 0;
                mbar_wait(drain, 0, g.timeout_ns, &never);
            }
        }
    } else {
        // ------------------------------------------------ epilogue
        pdl_wait();  // residual, workspace, counters and y only from here on
        const int ew = warp - 2;
        const int quarter = warp & 3;   // TMEM lanes this warp may access
        const int half = ew >> 2;       // which half of the m_pad columns
        const int row = quarter * 32 + lane;
        const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                   static_cast<uint32_t>(half * NC);
        const uint32_t lvl1 = lane_base + 2 * MPAD;
        const uint32_t lvl2 = lane_base + 3 * MPAD;
        int pc = 0;                     // chunks received (all units)
        for (int qi = 0;; ++qi) {
            const bool got = mbar_wait(&uq_full[qi % Q], (qi / Q) & 1, g.timeout_ns, &flags[0]);
            if (!got)
                group_failure(g, &flags[0], kErrTimeoutEpilogue);
            const int u = got ? uq[qi % Q] : -1;
            // every epilogue thread holds the unit id before the slot is released
            if (!epi_bar_and(got))
                break;
            if (ew == 0 && lane == 0)
                mbar_arrive(&uq_empty[qi % Q]);
            if (u < 0)
                break;
            const Unit U = unit_of(g, u);
            const GroupProj &P = g.proj[U.j];
            float st0[NC], cur[NC];     // per unit: nothing lives across units
            bool ok = true;
            for (int pl = 0; pl < U.present; ++pl, ++pc) {
                const int b = pc & 1;
                const uint32_t q = static_cast<uint32_t>(pc >> 1);
                if (!mbar_wait(&tfull[b], q & 1, g.timeout_ns, &flags[0])) {
                    group_failure(g, &flags[0], kErrTimeoutEpilogue);
                    ok = false;
                    break;
                }
                tc_fence_after();
                tmem_load_cols<NC>(lane_base + static_cast<uint32_t>(b * MPAD), cur);
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&tempty[b]);
                // canonical tree over this unit's chunks (as in the one-projection kernel)
                if (pl & 1) {
#pragma unroll
                    for (int c = 0; c < NC; ++c) cur[c] = st0[c] + cur[c];
                    if (pl & 2) {
                        tmem_add_cols<NC>(lvl1, cur);
                        if (pl & 4) {
                            tmem_add_cols<NC>(lvl2, cur);
                        } else {
                            tmem_store_cols<NC>(lvl2, cur);
                        }
                    } else {
                        tmem_store_cols<NC>(lvl1, cur);
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < NC; ++c) st0[c] = cur[c];
                }
            }
            ok = epi_bar_and(ok && !flags[0]);
            if (!ok)
                break;
            const int present = U.present;
            if (present != 8 && present > 0) {
                bool have = false;
                if (present & 1) {
#pragma unroll
                    for (int c = 0; c < NC; ++c) cur[c] = st0[c];
                    have = true;
                }
                if (present & 2) {
                    if (have) {
                        tmem_add_cols<NC>(lvl1, cur);
                    } else {
                        tmem_load_cols<NC>(lvl1, cur);
                    }
                    have = true;
                }
                if (present & 4) {
                    if (have) {
                        tmem_add_cols<NC>(lvl2, cur);
                    } else {
                        tmem_load_cols<NC>(lvl2, cur);
                    }
                }
            }
            const int n = U.tile * kTileN + row;
            if (present > 0 && n < P.N) {
#pragma unroll
                for (int c = 0; c < NC; ++c) {
                    const int m = half * NC + c;
                    if (m < g.M)
                        P.ws[((static_cast<size_t>(U.split) * P.n_tiles + U.tile) * P.M + m) * kTileN + row] = cur[c];
                }
            }
            // Arrive on the tile's counter (see the one-projection kernel):
            // the last R arrivals share the tile's reduction.  R > 1 only
            // when every CTA owns one unit and nothing depends on anything,
            // so a waiter waits only for CTAs that run their one unit to its
            // arrival without waiting.
            epi_bar_sync();
            const int R = P.reducers;
            if (ew == 0 && lane == 0) {
                const int old = static_cast<int>(atom_add_acq_rel_gpu(&P.counters[U.tile], 1u) & 0xFFFFu);
                const int first = P.split - R;
                int role = 0;
                if (old >= first) {
                    if (old == P.split - 1 ||
                        wait_counter(&P.counters[U.tile], static_cast<unsigned>(P.split), g.timeout_ns, &flags[0]))
                        role = old - first + 1;
                    else
                        group_failure(g, &flags[0], kErrTimeoutEpilogue);
                }
                // the last reducer to see every arrival returns the counter to zero
                if (role && R > 1 &&
                    (atom_add_acq_rel_gpu(&P.counters[U.tile], 1u << 16) >> 16) == static_cast<unsigned>(R - 1))
                    P.counters[U.tile] = 0;
                flags[1] = role;
            }
            epi_bar_sync();
            if (flags[1]) {
                const int role = flags[1];
                const int L = kChunks / P.split;
                const int sp = (chunks_present(P.nkb) + L - 1) / L;  // splits holding a value
                if (P.dep && U.j > 0 && P.res) {
                    // the residual may be the previous projection's output
                    if (ew == 0 && lane == 0 &&
                        !wait_counter(&g.done[U.j - 1], static_cast<unsigned>(g.proj[U.j - 1].n_tiles), g.timeout_ns,
                                      &flags[0]))
                        group_failure(g, &flags[0], kErrTimeoutEpilogue);
                    if (!epi_bar_and(!flags[0]))
                        break;
                }
                // splits are 2, 4 or 8 here (the group caps them; any split
                // gives the same bits); share r of R: whole columns
                // [r * ceil(M / R), (r + 1) * ceil(M / R))
                const int items = P.M * (kTileN / 4);
                const int share = (P.M + R - 1) / R * (kTileN / 4);
                group_reduce<MPAD>(&P, U.tile, sp, threadIdx.x - 64, min(items, (role - 1) * share),
                                   min(items, role * share));
                // every y store of the tile comes before the release of
                // done[j] (with one reducer; R > 1 only without dependencies,
                // where nothing reads done[j])
                epi_bar_sync();
                if (ew == 0 && lane == 0 && R == 1) {
                    P.counters[U.tile] = 0;
                    red_release_gpu_add(&g.done[U.j], 1u);
                }
            }
        }
    }

    // Lanes that ran a role alone reconverge; then the last CTA of the grid
    // returns the per-launch counters to zero (every CTA is past its waits).
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned old = atom_add_acq_rel_gpu(&g.done[kGroupDoneExit], 1u);
        if (old == gridDim.x - 1) {
            for (int j = 0; j < g.n; ++j)
                g.done[j] = 0;
            g.done[kGroupDoneNext] = 0;
            g.done[kGroupDoneExit] = 0;
        }
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, Sh::kTmemCols);
    }
}

template <int MPAD>
cudaError_t launch_group_t(const GroupParams &g, int grid, bool pdl, cudaStream_t s)
{
    const int smem = group_smem_bytes(MPAD, g.stages);
    static int attr_set[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    if (!__atomic_load_n(&attr_set[dev], __ATOMIC_ACQUIRE)) {
        e = cudaFuncSetAttribute(splitk_group_kernel<MPAD>, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(splitk_group_kernel<MPAD>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess)
            return e;
        __atomic_store_n(&attr_set[dev], 1, __ATOMIC_RELEASE);
    }
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
    return cudaLaunchKernelEx(&cfg, splitk_group_kernel<MPAD>, g);
}

// CTAs of the group kernel resident on one SM at once.  The runtime's
// occupancy query answers 1 for every kernel that allocates tensor memory,
// whatever its footprint, while such CTAs do share an SM (a kernel with 32
// TMEM columns ran four CTAs per SM side by side); so the count is taken
// from the kernel's own resources: registers (each of the four SM
// sub-partitions holds 16K, whole warps each), shared memory with the 1 KB
// the SM keeps per CTA, TMEM columns and threads.
template <int MPAD>
int ctas_per_sm_t(int stages)
{
    cudaFuncAttributes a;
    if (cudaFuncGetAttributes(&a, splitk_group_kernel<MPAD>) != cudaSuccess || a.numRegs <= 0)
        return 0;
    const int smem = group_smem_bytes(MPAD, stages);
    if (smem > 232448)
        return 0;
    const int regs_per_warp = (a.numRegs * 32 + 255) / 256 * 256;
    const int by_regs = 4 * (16384 / regs_per_warp) / (kTcThreads / 32);
    const int by_smem = 233472 / (smem + 1024);
    const int by_tmem = 512 / static_cast<int>(TcShape<MPAD>::kTmemCols);
    const int by_threads = 2048 / kTcThreads;
    return std::min(std::min(by_regs, by_smem), std::min(by_tmem, by_threads));
}

} // namespace

int group_smem_bytes(int m_pad, int stages)
{
    // the one-projection kernel's layout, then the unit queue: Q x (two
    // barriers + one id)
    return tc_smem_bytes(m_pad, stages) + kGroupUnitQueue * (2 * 8 + 4);
}

cudaError_t launch_group_tc(const GroupParams &g, int m_pad, int grid, bool pdl, cudaStream_t s)
{
    switch (m_pad) {
    case 16: return launch_group_t<16>(g, grid, pdl, s);
    case 32: return launch_group_t<32>(g, grid, pdl, s);
    case 48: return launch_group_t<48>(g, grid, pdl, s);
    case 64: return launch_group_t<64>(g, grid, pdl, s);
    default: return cudaErrorInvalidValue;
    }
}

int group_ctas_per_sm(int m_pad, int stages)
{
    switch (m_pad) {
    case 16: return ctas_per_sm_t<16>(stages);
    case 32: return ctas_per_sm_t<32>(stages);
    case 48: return ctas_per_sm_t<48>(stages);
    case 64: return ctas_per_sm_t<64>(stages);
    default: return 0;
    }
}

} // namespace skg
