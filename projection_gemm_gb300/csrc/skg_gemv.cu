// skg_gemv.cu -- the small-matrix projection kernel for M <= 2.
//
// "Hyper Optimizing Kimi K3 in vLLM: Moving Fast and Responsibly", method
// details 1 "Tune shapes for the workload": at batch 1-2 the attention input
// projections run on specialised small-matrix kernels.  At M <= 2 a
// projection is a pure weight stream (one or two FMAs per weight loaded), so
// this kernel is built for HBM bandwidth: every weight byte is read once
// (L2 evict-first), many bytes per SM are in flight before any is used, and
// accumulation is fp32 on CUDA cores -- tensor cores would idle at this
// arithmetic intensity.
//
// Forms, all with the arithmetic order below (so the same bits):
//   gemv_kernel            split 2..8: warps share a row's K range, per-lane
//                          cp.async ring, cross-warp combine (short N)
//   gemv_rows_kernel       split 1, any K: whole rows per warp, 16-byte loads
//                          into registers
//   gemv_rows_fast_kernel  the same for K % 256 == 0 (chunk width fixed)
//   gemv_rows_bulk_kernel  the same with each warp's weight batches moved by
//                          bulk copies into a shared-memory slot (default M = 2)
//   gemv_span_kernel       the bulk-copied batches in one balanced wave: CTAs
//                          own row runs, warps equal chunk runs, rows combined
//                          in shared memory (default M = 1)
//
// Reduction order (fixed, independent of the launch shape): row n is read in
// strips of 32 16-byte vectors (one coalesced 512-byte warp load; lane l
// takes vector 32 t + l of strip t).  The strips are cut into 16 canonical
// chunks of J = ceil(strips / 16) consecutive strips (the last chunks may be
// short or empty).  Inside a chunk each lane accumulates its vectors in strip
// order, each vector's 8 products in element order with fp32 FMA; the 32 lane
// sums are combined by the xor butterfly 16, 8, 4, 2, 1; the 16 chunk sums
// are combined by one balanced binary tree (empty chunks skipped).  A split of
// `split` warps per row hands each warp an aligned subtree of 16/split
// chunks, so every split gives the same bits.
#include <cuda_bf16.h>

#include <algorithm>

#include "skg_internal.h"
#include "skg_ptx.cuh"

namespace skg {
namespace {

constexpr int kWarps = kGemvThreads / 32;

template <int MM>
struct Acc {
    float v[MM];
};

// Pending left subtrees of the in-warp tree; level t holds 2^t chunk sums.
template <int MM>
struct ChunkStack {
    float lv[5][MM];

    // Chunk p (0-based within the warp's subtree) is done with sum a.
    __device__ __forceinline__ void push(int p, Acc<MM> a)
    {
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            if (p & (1 << t)) {
#pragma unroll
                for (int m = 0; m < MM; ++m)
                    a.v[m] = lv[t][m] + a.v[m];
            } else {
#pragma unroll
                for (int m = 0; m < MM; ++m)
                    lv[t][m] = a.v[m];
                return;
            }
        }
#pragma unroll
        for (int m = 0; m < MM; ++m)
            lv[4][m] = a.v[m];
    }

    // Value of the subtree after `count` chunks (any chunks after them are
    // empty): fold the complete blocks from the smallest upwards.
    __device__ __forceinline__ Acc<MM> flush(int count) const
    {
        Acc<MM> r;
        bool have = false;
#pragma unroll
        for (int t = 0; t < 5; ++t) {
            if (count & (1 << t)) {
#pragma unroll
                for (int m = 0; m < MM; ++m)
                    r.v[m] = have ? lv[t][m] + r.v[m] : lv[t][m];
                have = true;
            }
        }
        return r;
    }
};

__device__ __forceinline__ void fma8(float &acc, uint4 xv, uint4 wv)
{
    acc = fmaf(bf16lo(xv.x), bf16lo(wv.x), acc);
    acc = fmaf(bf16hi(xv.x), bf16hi(wv.x), acc);
    acc = fmaf(bf16lo(xv.y), bf16lo(wv.y), acc);
    acc = fmaf(bf16hi(xv.y), bf16hi(wv.y), acc);
    acc = fmaf(bf16lo(xv.z), bf16lo(wv.z), acc);
    acc = fmaf(bf16hi(xv.z), bf16hi(wv.z), acc);
    acc = fmaf(bf16lo(xv.w), bf16lo(wv.w), acc);
    acc = fmaf(bf16hi(xv.w), bf16hi(wv.w), acc);
}

// 16-byte shared-memory load of an x vector; volatile so the compiler does
// not hoist the (loop-invariant) x slice into registers for the whole kernel.
__device__ __forceinline__ uint4 lds_v4(const uint4 *p)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))));
    return v;
}

__device__ __forceinline__ void store_out(const GemvParams &p, int m, int n, float v)
{
    const size_t idx = static_cast<size_t>(m) * p.N + n;
    if (p.epilogue == SKG_EPI_FP32) {
        static_cast<float *>(p.y)[idx] = v;
        return;
    }
    if (p.epilogue == SKG_EPI_BF16_RESIDUAL)
        v += __uint_as_float(static_cast<uint32_t>(p.res[idx]) << 16);
    static_cast<__nv_bfloat16 *>(p.y)[idx] = __float2bfloat16_rn(v);
}

// T = the most strips one warp reads per row.  Weights land in shared
// memory: every warp owns a ring of p.ring slots of T strips (T * 512 bytes)
// and keeps p.ring - 1 rows of its K slice in flight with per-lane 16-byte
// cp.async copies (L2 evict-first).  Each lane later reads back exactly the
// vectors it copied itself, so per-thread wait_group is the only
// synchronisation the ring needs.  x is staged once per CTA in shared memory;
// the grid is persistent.
template <int MM, int T>
__global__ void __launch_bounds__(kGemvThreads) gemv_kernel(const GemvParams p)
{
    extern __shared__ uint4 dsm[];
    uint4 *xs = dsm;                              // [MM][nv]
    __shared__ float part[2][kWarps][MM];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = p.split;
    const int row_in_group = warp / split;
    const int sub = warp % split;
    const int leaves = kChunks / split;           // chunks owned by this warp
    const int ns = (p.nv + 31) >> 5;              // strips per row
    const int jc = (ns + kChunks - 1) / kChunks;  // strips per canonical chunk
    const int t0 = sub * leaves * jc;             // first strip of this warp
    const int nt = max(0, min(leaves * jc, ns - t0));
    const int my_present = (nt + jc - 1) / jc;
    const int total_present = (ns + jc - 1) / jc;
    const int split_present = (total_present + leaves - 1) / leaves;
    const int vbase = t0 * 32 + lane;
    const int R = p.ring;
    uint4 *my_ring = dsm + static_cast<size_t>(MM) * p.nv + static_cast<size_t>(warp) * R * T * 32 + lane;
    const uint64_t pol = policy_evict_first();

    auto has_row = [&](int g_) {
        return g_ < p.groups && g_ * p.rows_per_group + row_in_group < p.N && nt > 0;
    };
    // Request the K slice of group g_'s row into ring slot `slot`; always
    // commits a group so the per-thread group count stays uniform.
    auto issue = [&](int g_, int slot) {
        if (has_row(g_)) {
            const uint4 *src = p.W + static_cast<size_t>(g_ * p.rows_per_group + row_in_group) * p.nv + vbase;
            uint4 *dst = my_ring + static_cast<size_t>(slot) * T * 32;
#pragma unroll
            for (int t = 0; t < T; ++t) {
                if (t < nt && vbase + 32 * t < p.nv)
                    cp_async_16(dst + 32 * t, src + 32 * t, pol);
            }
        }
        cp_async_commit();
    };
    auto compute = [&](int slot) {
        const uint4 *w = my_ring + static_cast<size_t>(slot) * T * 32;
        ChunkStack<MM> stk;
        Acc<MM> a;
#pragma unroll
        for (int m = 0; m < MM; ++m)
            a.v[m] = 0.f;
        int cj = 0, leaf = 0;
#pragma unroll
        for (int t = 0; t < T; ++t) {
            if (t < nt) {
                const int v = vbase + 32 * t;
                if (v < p.nv) {
                    const uint4 wv = lds_v4(w + 32 * t);
#pragma unroll
                    for (int m = 0; m < MM; ++m)
                        fma8(a.v[m], lds_v4(xs + m * p.nv + v), wv);
                }
                if (++cj == jc || t + 1 == nt) {
                    // chunk complete: combine the lanes, then the tree
#pragma unroll
                    for (int m = 0; m < MM; ++m) {
#pragma unroll
                        for (int o = 16; o >= 1; o >>= 1)
                            a.v[m] += __shfl_xor_sync(0xffffffffu, a.v[m], o);
                    }
                    stk.push(leaf++, a);
#pragma unroll
                    for (int m = 0; m < MM; ++m)
                        a.v[m] = 0.f;
                    cj = 0;
                }
            }
        }
        return stk.flush(my_present);
    };
    // Publish this warp's subtree, then combine the `split` subtrees of each
    // row of group g_ (balanced tree) and write the outputs.
    auto finish = [&](int it, int g_, bool mine_valid, const Acc<MM> &mine) {
        if (lane == 0) {
#pragma unroll
            for (int m = 0; m < MM; ++m)
                part[it & 1][warp][m] = mine_valid ? mine.v[m] : 0.f;
        }
        __syncthreads();
        const int t = threadIdx.x;
        if (t < p.rows_per_group * MM) {
            const int rr = t / MM, m = t % MM;
            const int orow = g_ * p.rows_per_group + rr;
            if (orow < p.N) {
                float v[8];
#pragma unroll
                for (int s = 0; s < 8; ++s)
                    v[s] = (s < split) ? part[it & 1][rr * split + s][m] : 0.f;
#pragma unroll
                for (int stride = 1; stride < 8; stride <<= 1) {
#pragma unroll
                    for (int i = 0; i + stride < 8; i += 2 * stride) {
                        if (i + stride < split_present)
                            v[i] = v[i] + v[i + stride];
                    }
                }
                store_out(p, m, orow, v[0]);
            }
        }
    };

    // Weights are static: the first R - 1 rows are requested before the wait
    // for the previous kernel; activations are read only after it.
    int g = blockIdx.x;
    for (int i = 0; i < R - 1; ++i)
        issue(g + i * static_cast<int>(gridDim.x), i);
    pdl_wait();
    pdl_launch_dependents();
    for (int i = threadIdx.x; i < MM * p.nv; i += kGemvThreads)
        xs[i] = ld_act_v4(p.x + i);
    __syncthreads();

    const Acc<MM> zero = {};
    for (int it = 0; g < p.groups; g += gridDim.x, ++it) {
        cp_async_wait_dyn(R - 2);                 // this row's copies have landed
        const bool v0 = has_row(g);
        const Acc<MM> mine = v0 ? compute(it % R) : zero;
        issue(g + (R - 1) * static_cast<int>(gridDim.x), (it + R - 1) % R);  // slot read last iteration
        finish(it, g, v0, mine);
    }
    cp_async_wait<0>();                           // no copy in flight at exit
    if (threadIdx.x == 0)
        prefetch_next_slice(p.next_w, p.next_bytes, blockIdx.x, gridDim.x, policy_evict_last());
}

// Split 1: every warp owns whole rows and runs the complete canonical tree
// itself, so the main loop has no CTA-wide barrier.  Weights are read
// straight into registers in batches of U strips (U * 512 bytes per warp);
// x is staged once per CTA in shared memory; the grid covers all rows
// (rows_per_warp each) and the hardware scheduler keeps the SMs full.
template <int MM, int U>
__global__ void __launch_bounds__(kGemvThreads, 4) gemv_rows_kernel(const GemvParams p)
{
    extern __shared__ uint4 dsm[];
    uint4 *xs = dsm;                              // [MM][nv]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ns = (p.nv + 31) >> 5;              // strips per row
    const int jc = (ns + kChunks - 1) / kChunks;  // strips per canonical chunk
    const int present = (ns + jc - 1) / jc;
    const int row0 = (blockIdx.x * kWarps + warp) * p.rows_per_warp;
    const uint64_t pol = policy_evict_first();

    uint4 w[U];
    auto load_batch = [&](const uint4 *wrow, int s0) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int v = (s0 + u) * 32 + lane;
            if (s0 + u < ns && v < p.nv)
                w[u] = ld_weight_v4(wrow + v, pol);
        }
    };

    // Weights are static: the first batch is requested before the wait for
    // the previous kernel; activations are read only after it.
    bool preloaded = false;
    if (row0 < p.N) {
        load_batch(p.W + static_cast<size_t>(row0) * p.nv, 0);
        preloaded = true;
    }
    pdl_wait();
    pdl_launch_dependents();
    for (int i = threadIdx.x; i < MM * p.nv; i += kGemvThreads)
        xs[i] = ld_act_v4(p.x + i);
    __syncthreads();

    for (int r = 0; r < p.rows_per_warp; ++r) {
        const int row = row0 + r;
        if (row >= p.N)
            break;
        const uint4 *wrow = p.W + static_cast<size_t>(row) * p.nv;
        ChunkStack<MM> stk;
        Acc<MM> a;
#pragma unroll
        for (int m = 0; m < MM; ++m)
            a.v[m] = 0.f;
        int cj = 0, leaf = 0;
        for (int s0 = 0; s0 < ns; s0 += U) {
            if (p.ahead > 0 && lane == 0) {
                // the row is contiguous: ask the L2 for the batches that
                // follow while this one is loaded into registers
                const int a0 = s0 == 0 ? U : s0 + p.ahead * U;
                const int a1 = min(ns, s0 + (p.ahead + 1) * U);
                if (a0 < a1) {
                    const int v0 = a0 * 32, v1 = min(a1 * 32, p.nv);
                    prefetch_l2_bulk(wrow + v0, static_cast<uint32_t>((v1 - v0) * 16), pol);
                }
            }
            if (!preloaded)
                load_batch(wrow, s0);
            preloaded = false;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int t = s0 + u;
                if (t < ns) {
                    const int v = t * 32 + lane;
                    if (v < p.nv) {
#pragma unroll
                        for (int m = 0; m < MM; ++m)
                            fma8(a.v[m], lds_v4(xs + m * p.nv + v), w[u]);
                    }
                    if (++cj == jc || t + 1 == ns) {
#pragma unroll
                        for (int m = 0; m < MM; ++m) {
#pragma unroll
                            for (int o = 16; o >= 1; o >>= 1)
                                a.v[m] += __shfl_xor_sync(0xffffffffu, a.v[m], o);
                        }
                        stk.push(leaf++, a);
#pragma unroll
                        for (int m = 0; m < MM; ++m)
                            a.v[m] = 0.f;
                        cj = 0;
                    }
                }
            }
        }
        const Acc<MM> y = stk.flush(present);
        if (lane < MM)
            store_out(p, lane, row, lane == 0 ? y.v[0] : y.v[MM - 1]);
    }
    if (threadIdx.x == 0)
        prefetch_next_slice(p.next_w, p.next_bytes, blockIdx.x, gridDim.x, policy_evict_last());
}

// Whole rows per warp, specialised for K % 256 == 0 (every strip full):
// JC strips per canonical chunk is a compile-time constant, a batch is
// 8 strips = 8/JC whole chunks, and bounds are checked per chunk only.  Same
// arithmetic, same order as gemv_rows_kernel.  (Staging x as fp32 instead of
// bf16 measured slower: it doubles the shared-memory bytes read per weight.)
template <int MM, int JC>
__global__ void __launch_bounds__(kGemvThreads, 4) gemv_rows_fast_kernel(const GemvParams p)
{
    constexpr int U = 8;                          // strips per batch
    constexpr int B = U / JC;                     // chunks per batch
    extern __shared__ uint4 dsm[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nch = (p.nv >> 5) / JC;             // present chunks (<= 16)
    const int row0 = (blockIdx.x * kWarps + warp) * p.rows_per_warp;
    const uint64_t pol = policy_evict_first();

    uint4 w[U];
    auto load_batch = [&](const uint4 *wrow, int c0) {
#pragma unroll
        for (int b = 0; b < B; ++b) {
            if (c0 + b < nch) {
#pragma unroll
                for (int j = 0; j < JC; ++j)
                    w[b * JC + j] = ld_weight_v4(wrow + ((c0 + b) * JC + j) * 32 + lane, pol);
            }
        }
    };

    bool preloaded = false;
    if (row0 < p.N) {
        load_batch(p.W + static_cast<size_t>(row0) * p.nv, 0);
        preloaded = true;
    }
    pdl_wait();
    pdl_launch_dependents();
    for (int i = threadIdx.x; i < MM * p.nv; i += kGemvThreads)
        dsm[i] = ld_act_v4(p.x + i);
    __syncthreads();

    for (int r = 0; r < p.rows_per_warp; ++r) {
        const int row = row0 + r;
        if (row >= p.N)
            break;
        const uint4 *wrow = p.W + static_cast<size_t>(row) * p.nv;
        ChunkStack<MM> stk;
        for (int c0 = 0; c0 < nch; c0 += B) {
            if (p.ahead > 0 && lane == 0) {
                const int a0 = (c0 == 0 ? B : c0 + p.ahead * B) * JC * 32;
                const int a1 = min(nch, c0 + (p.ahead + 1) * B) * JC * 32;
                if (a0 < a1)
                    prefetch_l2_bulk(wrow + a0, static_cast<uint32_t>((a1 - a0) * 16), pol);
            }
            if (!preloaded)
                load_batch(wrow, c0);
            preloaded = false;
#pragma unroll
            for (int b = 0; b < B; ++b) {
                if (c0 + b < nch) {
                    Acc<MM> a;
#pragma unroll
                    for (int m = 0; m < MM; ++m)
                        a.v[m] = 0.f;
#pragma unroll
                    for (int j = 0; j < JC; ++j) {
                        const int v = ((c0 + b) * JC + j) * 32 + lane;
                        const uint4 wv = w[b * JC + j];
#pragma unroll
                        for (int m = 0; m < MM; ++m)
                            fma8(a.v[m], lds_v4(dsm + m * p.nv + v), wv);
                    }
#pragma unroll
                    for (int m = 0; m < MM; ++m) {
#pragma unroll
                        for (int o = 16; o >= 1; o >>= 1)
                            a.v[m] += __shfl_xor_sync(0xffffffffu, a.v[m], o);
                    }
                    stk.push(c0 + b, a);
                }
            }
        }
        const Acc<MM> y = stk.flush(nch);
        if (lane < MM)
            store_out(p, lane, row, lane == 0 ? y.v[0] : y.v[MM - 1]);
    }
    if (threadIdx.x == 0)
        prefetch_next_slice(p.next_w, p.next_bytes, blockIdx.x, gridDim.x, policy_evict_last());
}

// Lane reduction of a whole row at once.  Each lane holds V = 16 * MM
// partial sums (index m * 16 + c: chunk c, batch row m).  At each xor step
// 16, 8, 4, 2, 1 a lane keeps one half of its values and adds its partner's
// copy of that half, so every value is summed over the same lane pairs, in
// the same order, as by an xor butterfly of its own: the bits equal 16 * MM
// separate butterflies at a tenth of the shuffles.  Afterwards lane l holds
// value l >> (5 - log2 V); then the chunk sums of each m are combined across
// lanes by the balanced tree over 16 leaves (absent chunks skipped).  Returns
// the row sum for m = lane >> 4 (MM = 2, lanes 0 and 16) or m = 0 (MM = 1,
// lane 0).
template <int MM>
__device__ __forceinline__ float reduce_row(float (&v)[kChunks * MM], int lane, int nch)
{
    constexpr int V = kChunks * MM;
    constexpr int LS = 32 / V;                    // lanes per value at the end (1 or 2)
#pragma unroll
    for (int n = V, o = 16; n > 1; n >>= 1, o >>= 1) {
        const bool hi = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float keep = hi ? v[i + n / 2] : v[i];
            const float send = hi ? v[i] : v[i + n / 2];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    float r = v[0];
    if (LS == 2)
        r += __shfl_xor_sync(0xffffffffu, r, 1);  // the last butterfly step, both lanes of a value
    const int c = (lane / LS) & (kChunks - 1);
#pragma unroll
    for (int st = 1; st < kChunks; st <<= 1) {
        const float partner = __shfl_xor_sync(0xffffffffu, r, st * LS);
        if ((c & (2 * st - 1)) == 0 && c + st < nch)
            r = r + partner;
    }
    return r;
}

// Whole rows per warp with the copy engine on the load path: each warp keeps
// one shared-memory slot of a batch (U strips of 512 bytes, contiguous in the
// row) and lane 0 requests the next batch with one bulk copy as soon as the
// current batch has moved from the slot into registers, so the copy overlaps
// the FMAs.  The row's 16 x MM chunk sums stay per lane (fresh fp32
// accumulators, vectors in strip order as in the other forms) and are reduced
// once per row by reduce_row rather than one butterfly and tree step per
// chunk: the same bits, about a tenth of the shuffles.  Waits are bounded; a
// timeout sets an error bit and the warp stops after its copy has landed.
template <int MM, int JC, int U>
__global__ void __launch_bounds__(kGemvThreads, 4) gemv_rows_bulk_kernel(const GemvParams p)
{
    constexpr int B = U / JC;                     // chunks per batch
    extern __shared__ uint4 dsm[];
    __shared__ uint64_t wbar[kWarps];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nch = (p.nv >> 5) / JC;             // present chunks (<= 16)
    const int row0 = (blockIdx.x * kWarps + warp) * p.rows_per_warp;
    const int row_end = min(p.N, row0 + p.rows_per_warp);
    const uint64_t pol = policy_evict_first();
    uint4 *xs = dsm;                              // [MM][nv]
    uint4 *slot = dsm + static_cast<size_t>(MM) * p.nv + warp * U * 32;
    uint64_t *bar = &wbar[warp];
    uint32_t phase = 0;
    volatile int never = 0;

    auto issue = [&](int row, int c0) {
        if (lane == 0) {
            const uint32_t bytes = static_cast<uint32_t>(min(B, nch - c0) * JC) * 512u;
            mbar_arrive_expect_tx(bar, bytes);
            bulk_load(slot, p.W + static_cast<size_t>(row) * p.nv + c0 * JC * 32, bytes, bar, pol);
        }
    };
    if (lane == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    __syncwarp();
    if (row0 < row_end)
        issue(row0, 0);                           // weights are static: before the wait
    __syncwarp();
    pdl_wait();
    pdl_launch_dependents();
    for (int i = threadIdx.x; i < MM * p.nv; i += kGemvThreads)
        xs[i] = ld_act_v4(p.x + i);
    __syncthreads();

    for (int row = row0; row < row_end; ++row) {
        float acc[kChunks * MM];
#pragma unroll
        for (int i = 0; i < kChunks * MM; ++i)
            acc[i] = 0.f;
        uint4 w[U];
#pragma unroll
        for (int c = 0; c < kChunks; ++c) {
            if (c < nch) {
                if (c % B == 0) {
                    const bool got = mbar_wait(bar, phase, p.timeout_ns, &never);
                    phase ^= 1;
                    if (!__all_sync(0xffffffffu, got)) {
                        if (lane == 0 && p.err)
                            atomicOr(p.err, kErrTimeoutEpilogue);
                        mbar_wait(bar, phase ^ 1, p.timeout_ns, &never);   // let the copy land
                        return;
                    }
#pragma unroll
                    for (int b = 0; b < B; ++b) {
                        if (c + b < nch) {
#pragma unroll
                            for (int j = 0; j < JC; ++j)
                                w[b * JC + j] = lds_v4(slot + (b * JC + j) * 32 + lane);
                        }
                    }
                    // every lane's reads of the slot come before the next copy into it
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                    if (c + B < nch)
                        issue(row, c + B);
                    else if (row + 1 < row_end)
                        issue(row + 1, 0);
                }
#pragma unroll
                for (int j = 0; j < JC; ++j) {
                    const int v = (c * JC + j) * 32 + lane;
#pragma unroll
                    for (int m = 0; m < MM; ++m)
                        fma8(acc[m * kChunks + c], lds_v4(xs + m * p.nv + v), w[(c % B) * JC + j]);
                }
            }
        }
        const float r = reduce_row<MM>(acc, lane, nch);
        if ((lane & 15) == 0 && (lane >> 4) < MM)
            store_out(p, lane >> 4, row, r);
    }
    if (threadIdx.x == 0)
        prefetch_next_slice(p.next_w, p.next_bytes, blockIdx.x, gridDim.x, policy_evict_last());
}

template <int MM, int JC, int U>
cudaError_t launch_bulk_t(const GemvParams &p, const cudaLaunchConfig_t &cfg)
{
    static int done[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    if (!__atomic_load_n(&done[dev], __ATOMIC_ACQUIRE)) {
        e = cudaFuncSetAttribute(gemv_rows_bulk_kernel<MM, JC, U>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kGemvMaxSmem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(gemv_rows_bulk_kernel<MM, JC, U>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess)
            return e;
        __atomic_store_n(&done[dev], 1, __ATOMIC_RELEASE);
    }
    return cudaLaunchKernelEx(&cfg, gemv_rows_bulk_kernel<MM, JC, U>, p);
}

template <int MM>
cudaError_t launch_bulk_jc(const GemvParams &p, const cudaLaunchConfig_t &cfg, int jc)
{
    if (p.batch_strips == 4) {
        switch (jc) {
        case 1: return launch_bulk_t<MM, 1, 4>(p, cfg);
        case 2: return launch_bulk_t<MM, 2, 4>(p, cfg);
        case 4: return launch_bulk_t<MM, 4, 4>(p, cfg);
        default: return cudaErrorInvalidValue;
        }
    }
    switch (jc) {
    case 1: return launch_bulk_t<MM, 1, 8>(p, cfg);
    case 2: return launch_bulk_t<MM, 2, 8>(p, cfg);
    case 4: return launch_bulk_t<MM, 4, 8>(p, cfg);
    default: return launch_bulk_t<MM, 8, 8>(p, cfg);
    }
}

// Split 1 in one balanced wave: the grid is as many CTAs as the SMs hold,
// CTA b owns rows [b N / grid, (b+1) N / grid) and each of its warps an
// equal contiguous run of the CTA's canonical chunks -- rows are adjacent in
// memory, so a run crosses row boundaries freely and is still streamed in
// bulk-copied batches of U strips (as in the kernel above).  Every chunk sum
// is computed exactly as in the other forms and stored in shared memory;
// after one CTA barrier each row's sums are combined by the same balanced
// tree (absent chunks skipped), so the bits are the same.  No row is split
// across CTAs, so there is no cross-CTA step.
template <int MM, int JC, int U>
__global__ void __launch_bounds__(kGemvThreads, 4) gemv_span_kernel(const GemvParams p)
{
    constexpr int B = U / JC;                     // chunks per batch
    extern __shared__ uint4 dsm[];
    __shared__ uint64_t wbar[kWarps];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nch = (p.nv >> 5) / JC;             // chunks per row (<= 16)
    const int r0 = static_cast<int>(static_cast<long long>(blockIdx.x) * p.N / gridDim.x);
    const int r1 = static_cast<int>(static_cast<long long>(blockIdx.x + 1) * p.N / gridDim.x);
    const int total = (r1 - r0) * nch;
    const int g0 = static_cast<int>(static_cast<long long>(warp) * total / kWarps);
    const int g1 = static_cast<int>(static_cast<long long>(warp + 1) * total / kWarps);
    const uint64_t pol = policy_evict_first();
    uint4 *xs = dsm;                              // [MM][nv]
    uint4 *slot = dsm + static_cast<size_t>(MM) * p.nv + warp * U * 32;
    float *sums = reinterpret_cast<float *>(dsm + static_cast<size_t>(MM) * p.nv + kWarps * U * 32);  // [rows][16][MM]
    const uint4 *wbase = p.W + static_cast<size_t>(r0) * p.nv;   // chunk g starts at vector g * JC * 32
    uint64_t *bar = &wbar[warp];
    uint32_t phase = 0;
    volatile int never = 0;

    auto issue = [&](int g) {
        if (lane == 0) {
            const uint32_t bytes = static_cast<uint32_t>(min(B, g1 - g) * JC) * 512u;
            mbar_arrive_expect_tx(bar, bytes);
            bulk_load(slot, wbase + static_cast<size_t>(g) * JC * 32, bytes, bar, pol);
        }
    };
    if (lane == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    __syncwarp();
    if (g0 < g1) {
        issue(g0);                                // weights are static: before the wait
        if (p.ahead > 0 && lane == 0) {
            const int a0 = g0 + B, a1 = min(g1, g0 + (p.ahead + 1) * B);
            if (a0 < a1)
                prefetch_l2_bulk(wbase + static_cast<size_t>(a0) * JC * 32, static_cast<uint32_t>((a1 - a0) * JC) * 512u,
                                 pol);
        }
    }
    __syncwarp();
    pdl_wait();
    pdl_launch_dependents();
    for (int i = threadIdx.x; i < MM * p.nv; i += kGemvThreads)
        xs[i] = ld_act_v4(p.x + i);
    __syncthreads();

    uint4 w[U];
    bool ok = true;
    for (int gb = g0; gb < g1; gb += B) {
        if (p.ahead > 0 && lane == 0 && gb > g0) {
            const int a0 = gb + p.ahead * B, a1 = min(g1, gb + (p.ahead + 1) * B);
            if (a0 < a1)
                prefetch_l2_bulk(wbase + static_cast<size_t>(a0) * JC * 32, static_cast<uint32_t>((a1 - a0) * JC) * 512u,
                                 pol);
        }
        const bool got = mbar_wait(bar, phase, p.timeout_ns, &never);
        phase ^= 1;
        if (!__all_sync(0xffffffffu, got)) {
            if (lane == 0 && p.err)
                atomicOr(p.err, kErrTimeoutEpilogue);
            mbar_wait(bar, phase ^ 1, p.timeout_ns, &never);   // let the copy land
            ok = false;
            break;
        }
#pragma unroll
        for (int b = 0; b < B; ++b) {
            if (gb + b < g1) {
#pragma unroll
                for (int j = 0; j < JC; ++j)
                    w[b * JC + j] = lds_v4(slot + (b * JC + j) * 32 + lane);
            }
        }
        // every lane's reads of the slot come before the next copy into it
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (gb + B < g1)
            issue(gb + B);
#pragma unroll
        for (int b = 0; b < B; ++b) {
            const int g = gb + b;
            if (g < g1) {
                const int row = g / nch, c = g - row * nch;
                Acc<MM> a;
#pragma unroll
                for (int m = 0; m < MM; ++m)
                    a.v[m] = 0.f;
#pragma unroll
                for (int j = 0; j < JC; ++j) {
                    const int v = (c * JC + j) * 32 + lane;
#pragma unroll
                    for (int m = 0; m < MM; ++m)
                        fma8(a.v[m], lds_v4(xs + m * p.nv + v), w[b * JC + j]);
                }
#pragma unroll
                for (int m = 0; m < MM; ++m) {
#pragma unroll
                    for (int o = 16; o >= 1; o >>= 1)
                        a.v[m] += __shfl_xor_sync(0xffffffffu, a.v[m], o);
                }
                if (lane < MM)
                    sums[(row * kChunks + c) * MM + lane] = lane == 0 ? a.v[0] : a.v[MM - 1];
            }
        }
    }
    __syncwarp();
    ok = __syncthreads_and(ok);
    if (ok) {
        // each row's chunk sums by the balanced tree over 16 leaves, absent ones skipped
        for (int t = threadIdx.x; t < (r1 - r0) * MM; t += kGemvThreads) {
            const int row = t / MM, m = t - row * MM;
            float v[kChunks];
#pragma unroll
            for (int c = 0; c < kChunks; ++c)
                v[c] = c < nch ? sums[(row * kChunks + c) * MM + m] : 0.f;
#pragma unroll
            for (int stride = 1; stride < kChunks; stride <<= 1) {
#pragma unroll
                for (int i = 0; i + stride < kChunks; i += 2 * stride) {
                    if (i + stride < nch)
                        v[i] = v[i] + v[i + stride];
                }
            }
            store_out(p, m, r0 + row, v[0]);
        }
    }
    if (threadIdx.x == 0)
        prefetch_next_slice(p.next_w, p.next_bytes, blockIdx.x, gridDim.x, policy_evict_last());
}

template <int MM, int JC, int U>
cudaError_t launch_span_t(const GemvParams &p, const cudaLaunchConfig_t &cfg)
{
    static int done[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    if (!__atomic_load_n(&done[dev], __ATOMIC_ACQUIRE)) {
        e = cudaFuncSetAttribute(gemv_span_kernel<MM, JC, U>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kGemvMaxSmem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(gemv_span_kernel<MM, JC, U>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess)
            return e;
        __atomic_store_n(&done[dev], 1, __ATOMIC_RELEASE);
    }
    return cudaLaunchKernelEx(&cfg, gemv_span_kernel<MM, JC, U>, p);
}

template <int MM>
cudaError_t launch_span_jc(const GemvParams &p, const cudaLaunchConfig_t &cfg, int jc)
{
    if (p.batch_strips == 4) {
        switch (jc) {
        case 1: return launch_span_t<MM, 1, 4>(p, cfg);
        case 2: return launch_span_t<MM, 2, 4>(p, cfg);
        case 4: return launch_span_t<MM, 4, 4>(p, cfg);
        default: return cudaErrorInvalidValue;
        }
    }
    switch (jc) {
    case 1: return launch_span_t<MM, 1, 8>(p, cfg);
    case 2: return launch_span_t<MM, 2, 8>(p, cfg);
    case 4: return launch_span_t<MM, 4, 8>(p, cfg);
    default: return launch_span_t<MM, 8, 8>(p, cfg);
    }
}


template <int MM, int T>
cudaError_t set_gemv_attr()
{
    static int done[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    if (__atomic_load_n(&done[dev], __ATOMIC_ACQUIRE))
        return cudaSuccess;
    e = cudaFuncSetAttribute(gemv_kernel<MM, T>, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemvMaxSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemv_kernel<MM, T>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess)
        __atomic_store_n(&done[dev], 1, __ATOMIC_RELEASE);
    return e;
}

template <int MM, int T>
cudaError_t launch_t(const GemvParams &p, const cudaLaunchConfig_t &cfg)
{
    cudaError_t e = set_gemv_attr<MM, T>();
    return e != cudaSuccess ? e : cudaLaunchKernelEx(&cfg, gemv_kernel<MM, T>, p);
}

template <int MM>
cudaError_t set_rows_attr()
{
    static int done[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    if (__atomic_load_n(&done[dev], __ATOMIC_ACQUIRE))
        return cudaSuccess;
    e = cudaFuncSetAttribute(gemv_rows_kernel<MM, 8>, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemvMaxSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemv_rows_kernel<MM, 8>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess)
        __atomic_store_n(&done[dev], 1, __ATOMIC_RELEASE);
    return e;
}

template <int MM, int JC>
cudaError_t set_fast_attr()
{
    static int done[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    if (__atomic_load_n(&done[dev], __ATOMIC_ACQUIRE))
        return cudaSuccess;
    e = cudaFuncSetAttribute(gemv_rows_fast_kernel<MM, JC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kGemvMaxSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemv_rows_fast_kernel<MM, JC>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess)
        __atomic_store_n(&done[dev], 1, __ATOMIC_RELEASE);
    return e;
}

template <int MM, int JC>
cudaError_t launch_fast_t(const GemvParams &p, const cudaLaunchConfig_t &cfg)
{
    cudaError_t e = set_fast_attr<MM, JC>();
    return e != cudaSuccess ? e : cudaLaunchKernelEx(&cfg, gemv_rows_fast_kernel<MM, JC>, p);
}

template <int MM>
cudaError_t launch_fast_jc(const GemvParams &p, const cudaLaunchConfig_t &cfg, int jc)
{
    switch (jc) {
    case 1: return launch_fast_t<MM, 1>(p, cfg);
    case 2: return launch_fast_t<MM, 2>(p, cfg);
    case 4: return launch_fast_t<MM, 4>(p, cfg);
    default: return launch_fast_t<MM, 8>(p, cfg);
    }
}

template <int MM, int T>
cudaError_t occupancy_t(int smem, int *ctas)
{
    cudaError_t e = set_gemv_attr<MM, T>();
    return e != cudaSuccess ? e
                            : cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, gemv_kernel<MM, T>, kGemvThreads, smem);
}

} // namespace

// Strips per canonical chunk when every strip is full (K % 256 == 0) and the
// whole-row kernel can take it at compile time; 0 otherwise.
int gemv_fast_jc(int K)
{
    if (K % 256 != 0)
        return 0;
    const int ns = K / 256;
    const int jc = (ns + kChunks - 1) / kChunks;
    if (ns % jc != 0)
        return 0;
    return (jc == 1 || jc == 2 || jc == 4 || jc == 8) ? jc : 0;
}

bool gemv_bulk_ok(int M, int K, int batch_strips)
{
    const int jc = gemv_fast_jc(K);
    return jc > 0 && (batch_strips == 8 || (batch_strips == 4 && jc <= 4)) &&
           gemv_bulk_smem_bytes(M, K, batch_strips) <= kGemvMaxSmem;
}

int gemv_bulk_smem_bytes(int M, int K, int batch_strips)
{
    return M * K * 2 + (kGemvThreads / 32) * batch_strips * 512;   // x + one batch slot per warp
}

int gemv_span_smem_bytes(int M, int K, int batch_strips, int rows_per_cta)
{
    // x + one batch slot per warp + the chunk sums of the CTA's rows
    return gemv_bulk_smem_bytes(M, K, batch_strips) + rows_per_cta * kChunks * M * 4;
}

int gemv_span_grid(int M, int N, int K, int batch_strips, int num_sms)
{
    // one wave: as many CTAs as the SMs hold (228 KB, 1 KB reserved per CTA,
    // at most 4 by the launch bounds), never fewer than N / kGemvSpanMaxRows
    int grid = 0;
    for (int ctas = 4; ctas >= 1 && grid == 0; --ctas) {
        const int g = std::min(N, ctas * num_sms);
        const int rows = (N + g - 1) / g;
        if (rows <= kGemvSpanMaxRows && ctas * (gemv_span_smem_bytes(M, K, batch_strips, rows) + 1024 + 64) <= 233472)
            grid = g;
    }
    if (grid == 0)
        grid = std::min(N, std::max(num_sms, (N + kGemvSpanMaxRows - 1) / kGemvSpanMaxRows));
    return grid;
}

int gemv_bulk_default_batch(int M, int K)
{
    // 8-strip batches unless they cost the fourth CTA of an SM (228 KB, 1 KB
    // reserved per CTA) and 4-strip batches would keep it
    const int full = 4 * (gemv_bulk_smem_bytes(M, K, 8) + 1024 + 64);
    if (full <= 233472 || !gemv_bulk_ok(M, K, 4))
        return 8;
    return 4;
}

int gemv_smem_bytes(int M, int K, int split, int ring)
{
    if (split == 1 && ring >= 2)   // copy-engine forms at the default batch (span: one row per CTA)
        return gemv_bulk_smem_bytes(M, K, gemv_bulk_default_batch(M, K)) + (ring == 3 ? kChunks * M * 4 : 0);
    if (split == 1)   // the whole-row kernels keep weights in registers; x in shared memory
        return M * K * 2;
    return M * K * 2 + (kGemvThreads / 32) * ring * gemv_tile_strips(K, split) * 512;
}

int gemv_tile_strips(int K, int split)
{
    const int n = gemv_strips_per_warp(K, split);
    return n <= 4 ? 4 : (n <= 8 ? 8 : 16);
}

int gemv_strips_per_warp(int K, int split)
{
    const int ns = (K / 8 + 31) / 32;
    const int jc = (ns + kChunks - 1) / kChunks;
    return (kChunks / split) * jc;
}

cudaError_t gemv_occupancy(int M, int K, int split, int ring, int *ctas_per_sm)
{
    const int smem = gemv_smem_bytes(M, K, split, ring);
    if (split == 1) {
        cudaError_t e = M == 1 ? set_rows_attr<1>() : set_rows_attr<2>();
        if (e != cudaSuccess)
            return e;
        return M == 1 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, gemv_rows_kernel<1, 8>, kGemvThreads, smem)
                      : cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, gemv_rows_kernel<2, 8>, kGemvThreads, smem);
    }
    const int T = gemv_strips_per_warp(K, split);
    if (M == 1)
        return T > 8 ? occupancy_t<1, 16>(smem, ctas_per_sm)
                     : (T > 4 ? occupancy_t<1, 8>(smem, ctas_per_sm) : occupancy_t<1, 4>(smem, ctas_per_sm));
    return T > 8 ? occupancy_t<2, 16>(smem, ctas_per_sm)
                 : (T > 4 ? occupancy_t<2, 8>(smem, ctas_per_sm) : occupancy_t<2, 4>(smem, ctas_per_sm));
}

cudaError_t launch_gemv(const GemvParams &p, int grid, bool pdl, cudaStream_t s)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kGemvThreads);
    cfg.dynamicSmemBytes = gemv_smem_bytes(p.M, p.K, p.split, p.ring);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    if (p.split == 1 && p.ring == 3) {
        const int jc = gemv_fast_jc(p.K);
        const int rows = (p.N + grid - 1) / grid;
        if (!gemv_bulk_ok(p.M, p.K, p.batch_strips) || grid > p.N || rows > kGemvSpanMaxRows)
            return cudaErrorInvalidValue;
        cfg.dynamicSmemBytes = gemv_span_smem_bytes(p.M, p.K, p.batch_strips, rows);
        if (cfg.dynamicSmemBytes > static_cast<size_t>(kGemvMaxSmem))
            return cudaErrorInvalidValue;
        return p.M == 1 ? launch_span_jc<1>(p, cfg, jc) : launch_span_jc<2>(p, cfg, jc);
    }
    if (p.split == 1 && p.ring == 2) {
        const int jc = gemv_fast_jc(p.K);
        if (!gemv_bulk_ok(p.M, p.K, p.batch_strips))
            return cudaErrorInvalidValue;
        cfg.dynamicSmemBytes = gemv_bulk_smem_bytes(p.M, p.K, p.batch_strips);
        return p.M == 1 ? launch_bulk_jc<1>(p, cfg, jc) : launch_bulk_jc<2>(p, cfg, jc);
    }
    const int jc = gemv_fast_jc(p.K);
    if (p.split == 1 && jc > 0)
        return p.M == 1 ? launch_fast_jc<1>(p, cfg, jc) : launch_fast_jc<2>(p, cfg, jc);
    if (p.split == 1) {
        cudaError_t e = p.M == 1 ? set_rows_attr<1>() : set_rows_attr<2>();
        if (e != cudaSuccess)
            return e;
        return p.M == 1 ? cudaLaunchKernelEx(&cfg, gemv_rows_kernel<1, 8>, p)
                        : cudaLaunchKernelEx(&cfg, gemv_rows_kernel<2, 8>, p);
    }
    const int T = gemv_strips_per_warp(p.K, p.split);
    if (T > 16 || p.ring < 2 || p.ring > 9)
        return cudaErrorInvalidValue;
    if (p.M == 1)
        return T > 8 ? launch_t<1, 16>(p, cfg) : (T > 4 ? launch_t<1, 8>(p, cfg) : launch_t<1, 4>(p, cfg));
    return T > 8 ? launch_t<2, 16>(p, cfg) : (T > 4 ? launch_t<2, 8>(p, cfg) : launch_t<2, 4>(p, cfg));
}

} // namespace skg
