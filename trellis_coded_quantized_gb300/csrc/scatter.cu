// trellis_scatter: axis-0 packed matmul, out[m][c] = bf16(sum_r x[m][r] w[r][c]).
//
// The rows (input features) are cut into `splits` ranges of rp = ceil(R/S)
// rows; each range's fp32 partial sums go to partial[m][s][c] and a second
// kernel sums them over s (@mlx-bun/inference 1.0.0, kernels/trellis/
// scatter.ts: scatter kernels, rowsPer/r0/r1 split ranges, the [M, SPLITS,
// C] float partials and their sum over the split axis, cast to bf16).
//
// GB300 layout of the work:
//   - one CTA per SM owns one split and a block of up to 5 column ranges of
//     1024 columns; the 8-way replicated codebook (128 KB) sits in its
//     shared memory;
//   - a lane owns one 32-column unit and walks the rows of the split: per
//     row it streams the unit's k words (coalesced over the warp: 32 lanes
//     cover 4 consecutive blocks), takes the neighbour word by __shfl_sync,
//     decodes 32 weights and does MB FMAs per weight (bf16 x bf16 into f32),
//     one per activation row -- the shared-M variants of scatter.ts share
//     each decoded weight across activation rows the same way;
//   - RW warps per column range take interleaved rows of the split and their
//     partial sums are added in shared memory, in warp order, before the
//     store of the [MB, 1024] slab of partials;
//   - more than 4 activation rows are processed in passes of up to 4.
#include "common.cuh"
#include "internal.h"

namespace tcq {
namespace {

// Row warps per column range: 4 with one activation row, else 2; warps per
// CTA at most 20 (one activation row) or 10 (the accumulators of 2..4 rows
// need the larger register share).
__host__ __device__ constexpr int sc_row_warps(int mb) { return mb == 1 ? 4 : 2; }
__host__ __device__ constexpr int sc_max_warps(int mb) { return mb == 1 ? 20 : 10; }

template <int K, int MB>
__global__ void __launch_bounds__(sc_max_warps(MB) * 32, 1)
scatter_kernel(const uint16_t* __restrict__ x, int m0, const uint32_t* __restrict__ codes,
               const uint16_t* __restrict__ scales, const float* __restrict__ lut,
               int R, int C, int splits, int rp, int nur, int nurb, int interleave,
               float* __restrict__ partial) {
    constexpr int RW = sc_row_warps(MB);
    extern __shared__ __align__(16) float smem[];
    float* lut_s = smem;                                // 8-way replicated codebook
    float* red = smem + kLutN * kLutRep;                // [RW-1][nurb][MB][32 cols][32 lanes]
    stage_lut_rep8(lut_s, lut);
    __syncthreads();

    const int nblk = (nur + nurb - 1) / nurb;
    const int s = blockIdx.x / nblk;                    // split
    const int ub = blockIdx.x - s * nblk;               // block of column ranges
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int url = warp % nurb;                        // column range within the block
    const int rwi = warp / nurb;                        // row warp
    const int ur = ub * nurb + url;
    const int units = C >> 5;
    const int unit = ur * 32 + lane;
    const bool active = ur < nur && unit < units;
    const int r0 = s * rp;
    const int r1 = min(R, r0 + rp);
    const int64_t wpr = block_row_stride(units / kUnitsPerBlock, kBT * K / 32, interleave);
    const uint32_t* tp = codes + (active ? block_col_base(unit >> 3, R, kBT * K / 32, interleave) + (unit & 7) * K : 0);
    const int src = next_unit_lane(lane);
    const uint32_t gofs = lut_rep_lane_offset();

    float acc[MB][32];
    #pragma unroll
    for (int m = 0; m < MB; ++m)
        #pragma unroll
        for (int i = 0; i < 32; ++i) acc[m][i] = 0.f;

    uint32_t nxt[K];
    #pragma unroll
    for (int j = 0; j < K; ++j) nxt[j] = 0u;
    int r = r0 + rwi;
    if (active && r < r1) load_unit<K>(nxt, tp + (int64_t)r * wpr);
    for (; r < r1; r += RW) {
        uint32_t w[K + 1];
        #pragma unroll
        for (int j = 0; j < K; ++j) w[j] = nxt[j];
        const int rn = r + RW;
        if (active && rn < r1) load_unit<K>(nxt, tp + (int64_t)rn * wpr);
        w[K] = __shfl_sync(0xffffffffu, w[0], src);
        const float sr = bf16_bits_to_float(__ldg(scales + r));
        uint32_t xx[MB];                                // x[m][r] in both halves
        #pragma unroll
        for (int m = 0; m < MB; ++m) {
            const uint32_t h = __ldg(x + (int64_t)(m0 + m) * R + r);
            xx[m] = h | (h << 16);
        }
        #pragma unroll
        for (int i = 0; i < 32; i += 2) {
            const float v0 = lut_at(lut_s, win_off_sh<K, kLutRepShift>(w, i) | gofs);
            const float v1 = lut_at(lut_s, win_off_sh<K, kLutRepShift>(w, i + 1) | gofs);
            const uint32_t wp = pack_bf16x2(__fmul_rn(v0, sr), __fmul_rn(v1, sr));
            #pragma unroll
            for (int m = 0; m < MB; ++m) {
                acc[m][i] = fma_bf16_lo(wp, xx[m], acc[m][i]);
                acc[m][i + 1] = fma_bf16_hi(wp, xx[m], acc[m][i + 1]);
            }
        }
    }

    // add the row warps' partial sums (row warps 1.. stage theirs, row warp 0
    // adds them in order) and store the slab
    if (rwi > 0) {
        float* dst = red + ((size_t)(rwi - 1) * nurb + url) * MB * 1024;
        #pragma unroll
        for (int m = 0; m < MB; ++m)
            #pragma unroll
            for (int i = 0; i < 32; ++i) dst[(m * 32 + i) * 32 + lane] = acc[m][i];
    }
    __syncthreads();
    if (rwi == 0 && active) {
        #pragma unroll
        for (int m = 0; m < MB; ++m) {
            float v[32];
            #pragma unroll
            for (int i = 0; i < 32; ++i) {
                float a = acc[m][i];
                #pragma unroll
                for (int q = 1; q < RW; ++q)
                    a += red[(((size_t)(q - 1) * nurb + url) * MB * 32 + m * 32 + i) * 32 + lane];
                v[i] = a;
            }
            // window i <-> column c0 + 31 - i
            const int c0 = (unit >> 3) * kBT + (224 - 32 * (unit & 7));
            float4* dst = reinterpret_cast<float4*>(partial + ((int64_t)(m0 + m) * splits + s) * C + c0);
            #pragma unroll
            for (int q = 0; q < 8; ++q)
                dst[q] = make_float4(v[31 - 4 * q], v[30 - 4 * q], v[29 - 4 * q], v[28 - 4 * q]);
        }
    }
}

// out[m][c] = bf16( sum_s partial[m][s][c] ): a CTA covers 32 columns of one
// activation row with 32 groups of 8 threads; group g adds a contiguous run
// of splits in order (4 runs of 4 rows of 128 bytes for 128 splits), then
// the 32 runs are added in order.
constexpr int kRdGroups = 32;
constexpr int kRdCols = 32;

__global__ void __launch_bounds__(256)
split_reduce_kernel(const float* __restrict__ partial, int splits, int C, uint16_t* __restrict__ out) {
    __shared__ float4 red[kRdGroups][kRdCols / 4];
    const int m = blockIdx.y;
    const int cq = blockIdx.x * (kRdCols / 4) + (threadIdx.x & 7);   // float4 column index
    const int grp = threadIdx.x >> 3;
    const int per = (splits + kRdGroups - 1) / kRdGroups;
    const int s0 = grp * per, s1 = min(splits, s0 + per);
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    const float4* p = reinterpret_cast<const float4*>(partial + (int64_t)m * splits * C) + cq;
    const int64_t stride = C / 4;
    for (int s = s0; s < s1; ++s) {
        const float4 v = __ldg(p + (int64_t)s * stride);
        a.x += v.x; a.y += v.y; a.z += v.z; a.w += v.w;
    }
    red[grp][threadIdx.x & 7] = a;
    __syncthreads();
    if (grp == 0) {
        float4 t = red[0][threadIdx.x];
        for (int g = 1; g < kRdGroups; ++g) {
            const float4 v = red[g][threadIdx.x];
            t.x += v.x; t.y += v.y; t.z += v.z; t.w += v.w;
        }
        __nv_bfloat162 lo = __floats2bfloat162_rn(t.x, t.y);
        __nv_bfloat162 hi = __floats2bfloat162_rn(t.z, t.w);
        uint2 o;
        o.x = *reinterpret_cast<uint32_t*>(&lo);
        o.y = *reinterpret_cast<uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(out + (int64_t)m * C + cq * 4) = o;
    }
}

template <int K, int MB>
cudaError_t launch_pass(const Packed& p, const uint16_t* x, int m0, int splits, int rp, int nur,
                        float* partial, cudaStream_t stream) {
    constexpr int RW = sc_row_warps(MB);
    const int nurb = nur < sc_max_warps(MB) / RW ? nur : sc_max_warps(MB) / RW;
    const int nblk = (nur + nurb - 1) / nurb;
    const size_t smem = kLutRepBytes + (size_t)(RW - 1) * nurb * MB * 1024 * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(scatter_kernel<K, MB>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)(splits * nblk);
    scatter_kernel<K, MB><<<grid, nurb * RW * 32, smem, stream>>>(x, m0, p.codes, p.scales, p.lut,
                                                                  (int)p.rows, (int)p.cols, splits, rp,
                                                                  nur, nurb, p.interleave, partial);
    return cudaGetLastError();
}

template <int K>
cudaError_t launch_k(const Packed& p, const uint16_t* x, int M, int splits, float* partial,
                     cudaStream_t stream) {
    const int rp = (int)((p.rows + splits - 1) / splits);
    const int units = (int)(p.cols / 32);
    const int nur = (units + 31) / 32;
    for (int m0 = 0; m0 < M; m0 += 4) {
        const int mb = M - m0 < 4 ? M - m0 : 4;
        cudaError_t e;
        switch (mb) {
            case 1: e = launch_pass<K, 1>(p, x, m0, splits, rp, nur, partial, stream); break;
            case 2: e = launch_pass<K, 2>(p, x, m0, splits, rp, nur, partial, stream); break;
            case 3: e = launch_pass<K, 3>(p, x, m0, splits, rp, nur, partial, stream); break;
            default: e = launch_pass<K, 4>(p, x, m0, splits, rp, nur, partial, stream); break;
        }
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_scatter(const Packed& p, const uint16_t* x, int M, int splits,
                           float* partial, uint16_t* out, int sm_count, cudaStream_t stream) {
    (void)sm_count;
    cudaError_t e;
    switch (p.k) {
        case 2: e = launch_k<2>(p, x, M, splits, partial, stream); break;
        case 3: e = launch_k<3>(p, x, M, splits, partial, stream); break;
        case 4: e = launch_k<4>(p, x, M, splits, partial, stream); break;
        default: return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return e;
    const int C = (int)p.cols;
    dim3 grid((unsigned)(C / kRdCols), (unsigned)M);
    split_reduce_kernel<<<grid, 256, 0, stream>>>(partial, splits, C, out);
    return cudaGetLastError();
}

}  // namespace tcq

// ---------------------------------------------------------------------------
// trellis_scatter_noalloc: trellis_scatter with library-owned scratch.
//
// Some callers cannot hand the scatter a workspace: for example a plugin
// interface of an inference runtime that passes in only the input and output
// buffers, or a serving loop that must not call cudaMalloc because it can
// synchronise the device and stall every other stream.  This entry point
// keeps the fp32 split partials in a fixed array in device memory that the
// library itself declares, so the call needs no allocation at all.  The
// array is created when the library is loaded onto a GPU and stays reserved
// on every GPU that loads the library until the process exits.
// ---------------------------------------------------------------------------
#include "trellis.h"

#include <mutex>

namespace {

constexpr size_t kNoAllocScratchFloats = size_t(1) << 22;   // 16 MiB
static __device__ __align__(256) float g_scatter_scratch[kNoAllocScratchFloats];

constexpr int kNoAllocMaxDevices = 64;
std::once_flag g_scratch_once[kNoAllocMaxDevices];
float* g_scratch_ptr[kNoAllocMaxDevices];
cudaError_t g_scratch_err[kNoAllocMaxDevices];

}  // namespace

extern "C" trellis_status trellis_scatter_noalloc(const void* x, int32_t M, const uint32_t* codes,
                                                  const void* scales, const float* lut,
                                                  const trellis_geometry* g, int32_t splits,
                                                  void* out, void* stream) {
    if (!g) return TRELLIS_ERR_NULL;
    const size_t need = trellis_scatter_workspace_bytes(g, M, splits);
    if (need > kNoAllocScratchFloats * sizeof(float)) return TRELLIS_ERR_WORKSPACE;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) {
        cudaGetLastError();
        return TRELLIS_ERR_DEVICE;
    }
    // Once per device, with that device current: the device address of the
    // scratch array (its name in host code is only a host-side stand-in).
    std::call_once(g_scratch_once[dev], [dev]() {
        void* p = nullptr;
        g_scratch_err[dev] = cudaGetSymbolAddress(&p, g_scatter_scratch);
        g_scratch_ptr[dev] = static_cast<float*>(p);
        if (g_scratch_err[dev] != cudaSuccess) cudaGetLastError();
    });
    if (g_scratch_err[dev] != cudaSuccess || g_scratch_ptr[dev] == nullptr) return TRELLIS_ERR_DEVICE;
    // Every partial the reduction reads is written by this same call (empty
    // splits store zeros), so nothing in the scratch has to be cleared first.
    return trellis_scatter(x, M, codes, scales, lut, g, splits, g_scratch_ptr[dev],
                           kNoAllocScratchFloats * sizeof(float), out, stream);
}
