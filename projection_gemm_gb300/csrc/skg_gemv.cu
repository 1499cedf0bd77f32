// skg_gemv.cu -- the small-matrix projection kernel for M <= 2.
//
// "Hyper Optimizing Kimi K3 in vLLM: Moving Fast and Responsibly", method
// details 1 "Tune shapes for the workload": at batch 1-2 the attention input
// projections run on specialised small-matrix kernels.  At M <= 2 a
// projection is a pure weight stream (one or two FMAs per weight loaded), so
// this kernel is built for HBM bandwidth: every weight byte is read once with
// 16-byte coalesced loads (L1 no-allocate, L2 evict-first), several loads per
// lane are in flight before any is used, and accumulation is fp32 on CUDA
// cores -- tensor cores would idle at this arithmetic intensity.
//
// Reduction order (fixed, independent of the launch shape): row n's K range
// is cut into 16 canonical chunks of 16-byte vectors; inside chunk c, lane l
// accumulates vectors begin(c) + l + 32 j for j = 0, 1, ... in order, each
// vector's 8 products in element order with fp32 FMA; the 32 lane sums are
// combined by the xor butterfly 16, 8, 4, 2, 1; the 16 chunk sums are
// combined by one balanced binary tree (empty chunks skipped).  A split of
// `split` warps per row hands each warp an aligned subtree of 16/split
// chunks, so every split gives the same bits.
#include <cuda_bf16.h>

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

// U = 16-byte weight vectors each lane keeps in flight per batch.  x is
// staged once per CTA in shared memory (dynamic, M * K * 2 bytes).
template <int MM, int U>
__global__ void __launch_bounds__(kGemvThreads) gemv_kernel(const GemvParams p)
{
    extern __shared__ uint4 xs[];                 // [MM][nv]
    __shared__ float part[2][kWarps][MM];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = p.split;
    const int row_in_group = warp / split;
    const int sub = warp % split;
    const int leaves = kChunks / split;           // chunks owned by this warp
    const int c0 = sub * leaves;
    const int total_present = chunks_present(p.nv);
    const int my_present = max(0, min(leaves, total_present - c0));
    const int split_present = (total_present + leaves - 1) / leaves;
    // vectors per lane per chunk, uniform over chunks (the largest chunk)
    const int q = p.nv / kChunks, r = p.nv % kChunks;
    const int J = (q + (r ? 1 : 0) + 31) >> 5;
    const int nslots = my_present * J;
    const uint64_t pol = policy_evict_first();

    uint4 wv[U];
    bool ok[U];
    // Issue the weight loads of slots [s0, s0 + U) of row `row`.
    auto load_batch = [&](const uint4 *wrow, int s0) {
        int lc = s0 / J, lj = s0 - (s0 / J) * J;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = c0 + lc;
            const int v = chunk_begin(c, p.nv) + lane + 32 * lj;
            ok[u] = (s0 + u < nslots) && (v < chunk_begin(c + 1, p.nv));
            if (ok[u])
                wv[u] = ld_weight_v4(wrow + v, pol);
            if (++lj == J) { lj = 0; ++lc; }
        }
    };

    // Weights are static: the first batch is requested before the wait for
    // the previous kernel; activations are read only after it.
    int g = blockIdx.x;
    bool preloaded = false;
    {
        const int row = g * p.rows_per_group + row_in_group;
        if (g < p.groups && row < p.N && nslots > 0) {
            load_batch(p.W + static_cast<size_t>(row) * p.nv, 0);
            preloaded = true;
        }
    }
    pdl_wait();
    pdl_launch_dependents();
    for (int i = threadIdx.x; i < MM * p.nv; i += kGemvThreads)
        xs[i] = ld_act_v4(p.x + i);
    __syncthreads();

    for (int it = 0; g < p.groups; g += gridDim.x, ++it) {
        const int row = g * p.rows_per_group + row_in_group;
        Acc<MM> mine;
#pragma unroll
        for (int m = 0; m < MM; ++m)
            mine.v[m] = 0.f;
        if (row < p.N && nslots > 0) {
            const uint4 *wrow = p.W + static_cast<size_t>(row) * p.nv;
            ChunkStack<MM> stk;
            Acc<MM> a;
#pragma unroll
            for (int m = 0; m < MM; ++m)
                a.v[m] = 0.f;
            int cc = 0, cj = 0;      // compute cursor: chunk (relative), j
            for (int s0 = 0; s0 < nslots; s0 += U) {
                if (!preloaded)
                    load_batch(wrow, s0);
                preloaded = false;
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    if (s0 + u < nslots) {
                        if (ok[u]) {
                            const int v = chunk_begin(c0 + cc, p.nv) + lane + 32 * cj;
#pragma unroll
                            for (int m = 0; m < MM; ++m)
                                fma8(a.v[m], xs[m * p.nv + v], wv[u]);
                        }
                        if (++cj == J) {
                            // chunk cc complete: combine the lanes, then the tree
#pragma unroll
                            for (int m = 0; m < MM; ++m) {
#pragma unroll
                                for (int o = 16; o >= 1; o >>= 1)
                                    a.v[m] += __shfl_xor_sync(0xffffffffu, a.v[m], o);
                            }
                            stk.push(cc, a);
#pragma unroll
                            for (int m = 0; m < MM; ++m)
                                a.v[m] = 0.f;
                            cj = 0;
                            ++cc;
                        }
                    }
                }
            }
            mine = stk.flush(my_present);
        }
        if (lane == 0) {
#pragma unroll
            for (int m = 0; m < MM; ++m)
                part[it & 1][warp][m] = mine.v[m];
        }
        __syncthreads();
        // combine the `split` warp subtrees of each row: balanced tree
        const int t = threadIdx.x;
        if (t < p.rows_per_group * MM) {
            const int rr = t / MM, m = t % MM;
            const int orow = g * p.rows_per_group + rr;
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
    }
}

} // namespace

int gemv_smem_bytes(int M, int K) { return M * K * 2; }

cudaError_t launch_gemv(const GemvParams &p, int grid, bool pdl, cudaStream_t s)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kGemvThreads);
    cfg.dynamicSmemBytes = gemv_smem_bytes(p.M, p.K);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    static int attr_set[2][kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    int *flag = &attr_set[p.M == 1 ? 0 : 1][dev];
    if (__atomic_load_n(flag, __ATOMIC_ACQUIRE) == 0) {
        e = cudaFuncSetAttribute(p.M == 1 ? gemv_kernel<1, 8> : gemv_kernel<2, 8>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kGemvMaxSmem);
        if (e != cudaSuccess)
            return e;
        __atomic_store_n(flag, 1, __ATOMIC_RELEASE);
    }
    if (p.M == 1)
        return cudaLaunchKernelEx(&cfg, gemv_kernel<1, 8>, p);
    return cudaLaunchKernelEx(&cfg, gemv_kernel<2, 8>, p);
}

} // namespace skg
