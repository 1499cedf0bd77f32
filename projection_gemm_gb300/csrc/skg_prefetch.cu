// skg_prefetch.cu -- L2 weight prefetch and the bounded-wait self test.
//
// "Hyper Optimizing Kimi K3 in vLLM: Moving Fast and Responsibly", method
// details 4 "Prefetching upcoming weights into cache": small-batch decode is
// bound by loading weights from HBM, yet some phases leave HBM bandwidth
// unused; a dedicated kernel on a side stream loads the next operation's
// weights into cache meanwhile, so that operation starts with a much higher
// cache hit rate.  Here the kernel issues bulk L2 prefetches
// (cp.async.bulk.prefetch.L2, no data written anywhere) with an evict-last
// policy, so the projection running beside it, which streams its own weight
// with evict-first, does not push the prefetched lines out.
#include "skg_internal.h"
#include "skg_ptx.cuh"

namespace skg {
namespace {

constexpr uint32_t kPiece = 32768;   // bytes per bulk prefetch
constexpr int kPrefetchThreads = 128;

__global__ void __launch_bounds__(kPrefetchThreads)
prefetch_l2_kernel(const uint8_t *base, size_t bytes)
{
    const uint64_t pol = policy_evict_last();
    const size_t nth = static_cast<size_t>(gridDim.x) * blockDim.x;
    for (size_t off = (static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x) * kPiece;
         off < bytes; off += nth * kPiece) {
        const size_t left = bytes - off;
        const uint32_t sz = static_cast<uint32_t>(left < kPiece ? left : kPiece);
        prefetch_l2_bulk(base + off, sz, pol);
    }
}

// One thread waits, bounded by timeout_ns, on a barrier nobody arrives at,
// then records the expiry and returns: the failure-detection path without
// any fault.
__global__ void debug_wait_kernel(unsigned int *err, unsigned long long timeout_ns)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        volatile int never = 0;
        if (!mbar_wait(&bar, 0, timeout_ns, &never))
            atomicOr(err, kErrTimeoutDebug);
        mbar_inval(&bar);
    }
}

} // namespace

cudaError_t launch_prefetch_l2(const void *base, size_t bytes, cudaStream_t s)
{
    if (bytes == 0)
        return cudaSuccess;
    const size_t pieces = (bytes + kPiece - 1) / kPiece;
    size_t grid = (pieces + kPrefetchThreads - 1) / kPrefetchThreads;
    if (grid > 64)
        grid = 64;
    prefetch_l2_kernel<<<static_cast<unsigned>(grid), kPrefetchThreads, 0, s>>>(
        static_cast<const uint8_t *>(base), bytes);
    return cudaGetLastError();
}

cudaError_t launch_debug_wait(unsigned int *err, unsigned long long timeout_ns, cudaStream_t s)
{
    debug_wait_kernel<<<1, 32, 0, s>>>(err, timeout_ns);
    return cudaGetLastError();
}

} // namespace skg
