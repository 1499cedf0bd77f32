// skg_rowpar.cu -- the cross-rank step of a projection whose K is sharded
// across ranks (row-parallel output projection).
//
// "Hyper Optimizing Kimi K3 in vLLM: Moving Fast and Responsibly", method
// details 2 "Overlap computation and communication": with tensor
// parallelism the output projection's reduction dimension is split across
// GPUs, every GPU holds a partial result, and the partials are summed (an
// all-reduce, one-shot at small batch and two-stage at large batch) and the
// attention residual is added in the same step.
//
// Here rank r of R owns canonical K chunks [16r/R, 16(r+1)/R) -- an aligned
// subtree of the 16-leaf canonical tree -- and skg_run of a sharded plan
// leaves that subtree's fp32 value.  This kernel combines the R values of
// every output by the tree's top levels in rank order, adds the residual in
// fp32 and rounds once: the same additions in the same order as one launch
// over the whole K, so the same bits.  Moving the partials between GPUs is
// the caller's (an all-gather of the [M, N] fp32 partials, or peer reads).
#include <cuda_bf16.h>

#include <algorithm>

#include "skg_internal.h"

namespace skg {
namespace {

struct CombineParams {
    const float *part[kMaxRanks];
    const uint16_t *res;
    void *y;
    int ranks, M, N, epilogue;
};

template <int R>
__global__ void __launch_bounds__(256) combine_kernel(const CombineParams p)
{
    const size_t total = static_cast<size_t>(p.M) * p.N;
    for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        float v[R];
#pragma unroll
        for (int r = 0; r < R; ++r)
            v[r] = __ldg(p.part[r] + i);
#pragma unroll
        for (int stride = 1; stride < R; stride <<= 1) {
#pragma unroll
            for (int j = 0; j + stride < R; j += 2 * stride)
                v[j] = v[j] + v[j + stride];
        }
        if (p.epilogue == SKG_EPI_FP32) {
            static_cast<float *>(p.y)[i] = v[0];
        } else {
            float o = v[0];
            if (p.epilogue == SKG_EPI_BF16_RESIDUAL)
                o += __uint_as_float(static_cast<uint32_t>(p.res[i]) << 16);
            static_cast<__nv_bfloat16 *>(p.y)[i] = __float2bfloat16_rn(o);
        }
    }
}

} // namespace

cudaError_t launch_combine(const float *const *partials, int ranks, const uint16_t *res, void *y, int M, int N,
                           int epilogue, cudaStream_t s)
{
    CombineParams p = {};
    for (int r = 0; r < ranks; ++r)
        p.part[r] = partials[r];
    p.res = res;
    p.y = y;
    p.ranks = ranks;
    p.M = M;
    p.N = N;
    p.epilogue = epilogue;
    const size_t total = static_cast<size_t>(M) * N;
    const unsigned grid = static_cast<unsigned>(std::min<size_t>((total + 255) / 256, 152 * 8));
    switch (ranks) {
    case 1: combine_kernel<1><<<grid, 256, 0, s>>>(p); break;
    case 2: combine_kernel<2><<<grid, 256, 0, s>>>(p); break;
    case 4: combine_kernel<4><<<grid, 256, 0, s>>>(p); break;
    case 8: combine_kernel<8><<<grid, 256, 0, s>>>(p); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

} // namespace skg
