// skg_tc_common.cuh -- device code shared by the split-K tensor-core kernels
// (one projection per launch, and a group of projections in one persistent
// launch): tile shapes, TMEM column helpers, the epilogue barriers, the
// output store and the last-CTA split reduction over the tile-major fp32
// workspace.  The output and reduction helpers take any parameter type with
// the fields they read (M, N, ws, n_tiles, y, res, epilogue), so each kernel
// passes its own parameters in place.  Included inside namespace skg's
// anonymous namespace.
#pragma once

constexpr uint32_t kWBytes = kTileN * kBlockK * 2;  // 16 KB per stage
constexpr int kEpiThreads = 256;

template <int MPAD>
struct TcShape {
    static constexpr uint32_t kXBytes = MPAD * kBlockK * 2;  // multiple of 1 KB
    // two accumulators + tree levels 1 and 2, rounded up to a power of two
    static constexpr uint32_t kTmemCols = (4 * MPAD <= 32) ? 32 : (4 * MPAD <= 64 ? 64 : (4 * MPAD <= 128 ? 128 : 256));
    static constexpr int kNC = MPAD / 2;                     // columns per epilogue thread
    static constexpr uint32_t kIdesc = idesc_bf16_f32(kTileN, MPAD);
};

__device__ __forceinline__ void record_failure(const TcParams &p, volatile int *abort, unsigned bit)
{
    *abort = 1;
    if (p.err)
        atomicOr(p.err, bit);
}

__device__ __forceinline__ void epi_bar_sync()
{
    asm volatile("bar.sync 1, 256;" ::: "memory");
}

// Barrier over the 256 epilogue threads that also ANDs a predicate.
__device__ __forceinline__ bool epi_bar_and(bool v)
{
    uint32_t out;
    asm volatile("{\n\t.reg .pred pi, po;\n\t"
                 "setp.ne.u32 pi, %1, 0;\n\t"
                 "bar.red.and.pred po, 1, 256, pi;\n\t"
                 "selp.u32 %0, 1, 0, po;\n\t}"
                 : "=r"(out) : "r"(v ? 1u : 0u) : "memory");
    return out != 0;
}

__device__ __forceinline__ unsigned atom_add_acq_rel_gpu(unsigned *ptr, unsigned v)
{
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(ptr), "r"(v) : "memory");
    return old;
}

template <class PP>
__device__ __forceinline__ void store_out(const PP &p, int m, int n, float v)
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

// Read NC consecutive fp32 columns of this thread's TMEM lane into v.  The
// empty asm statements after the wait tie every use of the loaded registers
// to a point after tcgen05.wait::ld.
template <int NC>
__device__ __forceinline__ void tmem_load_cols(uint32_t taddr, float (&v)[NC])
{
    uint32_t r[NC];
#pragma unroll
    for (int j = 0; j < NC / 8; ++j)
        tmem_ld_x8(taddr + 8 * j, *reinterpret_cast<uint32_t(*)[8]>(&r[8 * j]));
    tmem_wait_ld();
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        asm volatile("" : "+r"(r[c]));
        v[c] = __uint_as_float(r[c]);
    }
}

// acc[c] = TMEM[c] + acc[c] for NC columns, 8 at a time (keeps registers low).
template <int NC>
__device__ __forceinline__ void tmem_add_cols(uint32_t taddr, float (&acc)[NC])
{
#pragma unroll
    for (int j = 0; j < NC / 8; ++j) {
        uint32_t r[8];
        tmem_ld_x8(taddr + 8 * j, r);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            asm volatile("" : "+r"(r[c]));
            acc[8 * j + c] = __uint_as_float(r[c]) + acc[8 * j + c];
        }
    }
}

template <int NC>
__device__ __forceinline__ void tmem_store_cols(uint32_t taddr, const float (&v)[NC])
{
#pragma unroll
    for (int j = 0; j < NC / 8; ++j) {
        uint32_t r[8];
#pragma unroll
        for (int c = 0; c < 8; ++c)
            r[c] = __float_as_uint(v[8 * j + c]);
        tmem_st_x8(taddr + 8 * j, r);
    }
    tmem_wait_st();
}

// The workspace holds, for every split s and tile, the tile's partial sums
// as one contiguous block [M][128] of fp32 (m-major, the tile's 128 rows
// innermost): a warp's stores and loads of one column m are coalesced, and a
// tile's S partials are S compact blocks instead of M x S row pieces spread
// N floats apart (measured: 29.3 -> 25.0 us at M = 64, K = N = 7168).
//
// The last CTA of a tile: y[m, n] for this thread's row n and columns
// [half * NC, half * NC + NC) from the S split values in the workspace,
// combined by the top levels of the canonical tree.  Loads are issued in
// batches of whole columns x all S values (24 or 48 independent loads, as
// the register budget of the CTA shape allows), so the tile costs a few L2
// round trips instead of one per column.
template <int S, int NC, class PP>
__device__ __forceinline__ void reduce_tile(const PP &p, int tile, int row, int half, int sp)
{
    const int n = tile * kTileN + row;

    constexpr int kLoads = NC >= 24 ? 48 : 24;
    constexpr int G0 = kLoads / S < 1 ? 1 : kLoads / S;
    constexpr int G = G0 < NC ? G0 : NC;                 // columns per batch
#pragma unroll 1
    for (int c0 = 0; c0 < NC; c0 += G) {
        const int mb = half * NC + c0;
        if (mb >= p.M)
            break;
        float v[G][S];
#pragma unroll
        for (int g = 0; g < G; ++g) {
#pragma unroll
            for (int s = 0; s < S; ++s) {
                const int m = mb + g;
                v[g][s] = (s < sp && m < p.M)
                              ? __ldcg(&p.ws[((static_cast<size_t>(s) * p.n_tiles + tile) * p.M + m) * kTileN + row])
                              : 0.f;
            }
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
#pragma unroll
            for (int stride = 1; stride < S; stride <<= 1) {
#pragma unroll
                for (int i = 0; i + stride < S; i += 2 * stride) {
                    if (i + stride < sp)
                        v[g][i] = v[g][i] + v[g][i + stride];
                }
            }
            if (mb + g < p.M)
                store_out(p, mb + g, n, v[g][0]);
        }
    }
}

// The last CTA of a tile, with 16-byte loads: work item (m, g) is rows
// 4g..4g+3 of column m, so the 32 lanes of a warp read 512 contiguous bytes
// of each split's block, and each output is combined exactly as in
// reduce_tile (the top levels of the canonical tree, in index order).  The
// 256 epilogue threads take items i_begin + et, + 256, ... below i_end (all
// items by default); IB = L / S items per batch keep L loads in flight (L as
// the CTA shape's register budget allows).
template <class PP>
__device__ __forceinline__ void store_out4(const PP &p, int m, int n0, int cnt, const float4 &v)
{
    const size_t idx = static_cast<size_t>(m) * p.N + n0;
    const float a[4] = {v.x, v.y, v.z, v.w};
    if (cnt == 4 && (p.N & 3) == 0) {
        if (p.epilogue == SKG_EPI_FP32) {
            *reinterpret_cast<float4 *>(static_cast<float *>(p.y) + idx) = v;
            return;
        }
        float b[4] = {a[0], a[1], a[2], a[3]};
        if (p.epilogue == SKG_EPI_BF16_RESIDUAL) {
            const uint2 r = *reinterpret_cast<const uint2 *>(p.res + idx);
            b[0] += bf16lo(r.x);
            b[1] += bf16hi(r.x);
            b[2] += bf16lo(r.y);
            b[3] += bf16hi(r.y);
        }
        uint2 o;
        o.x = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(b[0]))) |
              (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(b[1]))) << 16);
        o.y = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(b[2]))) |
              (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(b[3]))) << 16);
        *reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(p.y) + idx) = o;
        return;
    }
    for (int i = 0; i < cnt; ++i)
        store_out(p, m, n0 + i, a[i]);
}

template <int S, int L, class PP>
__device__ __forceinline__ void reduce_tile_v4(const PP &p, int tile, int sp, int et, int i_begin = 0,
                                               int i_end = -1)
{
    constexpr int IB = S >= L ? 1 : L / S;        // items per batch
    const int rows = min(kTileN, p.N - tile * kTileN);
    const int items = i_end < 0 ? p.M * (kTileN / 4) : i_end;
    const float *base = p.ws + static_cast<size_t>(tile) * p.M * kTileN;
    const size_t sstride = static_cast<size_t>(p.n_tiles) * p.M * kTileN;
#pragma unroll 1
    for (int i0 = i_begin + et; i0 < items; i0 += kEpiThreads * IB) {
        float4 v[IB][S];
#pragma unroll
        for (int b = 0; b < IB; ++b) {
            const int it = i0 + b * kEpiThreads;
            const int m = it >> 5, g = it & 31;
#pragma unroll
            for (int s = 0; s < S; ++s) {
                v[b][s] = (s < sp && it < items && 4 * g < rows)
                              ? __ldcg(reinterpret_cast<const float4 *>(base + s * sstride + m * kTileN + 4 * g))
                              : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
#pragma unroll
        for (int b = 0; b < IB; ++b) {
            const int it = i0 + b * kEpiThreads;
            const int m = it >> 5, g = it & 31;
            if (it >= items || 4 * g >= rows)
                continue;
#pragma unroll
            for (int stride = 1; stride < S; stride <<= 1) {
#pragma unroll
                for (int i = 0; i + stride < S; i += 2 * stride) {
                    if (i + stride < sp) {
                        v[b][i].x = v[b][i].x + v[b][i + stride].x;
                        v[b][i].y = v[b][i].y + v[b][i + stride].y;
                        v[b][i].z = v[b][i].z + v[b][i + stride].z;
                        v[b][i].w = v[b][i].w + v[b][i + stride].w;
                    }
                }
            }
            store_out4(p, m, tile * kTileN + 4 * g, min(4, rows - 4 * g), v[b][0]);
        }
    }
}
