// trellis_expand: decode a packed matrix to dense bf16 weights (and windows).
//
// Verification export only (@mlx-bun/inference 1.0.0,
// kernels/trellis/vector-expand.ts, expand kernel: the caller then owns an
// ordinary matmul).  One thread decodes one 32-column unit of one row and
// writes its 32 weights (64 bytes) and windows with 16-byte stores.
#include "common.cuh"
#include "internal.h"

namespace tcq {
namespace {

template <int K>
__global__ void __launch_bounds__(256)
expand_kernel(const uint32_t* __restrict__ codes, const uint16_t* __restrict__ scales,
              const float* __restrict__ lut, int64_t rows, int64_t units_per_row, int interleave,
              uint16_t* __restrict__ w_out, uint16_t* __restrict__ win_out) {
    __shared__ __align__(16) float lut_s[kLutN];
    stage_lut(lut_s, lut);
    __syncthreads();
    const int64_t cols = units_per_row * 32;
    constexpr int wpb = kBT * K / 32;
    const int64_t rs = block_row_stride(units_per_row / kUnitsPerBlock, wpb, interleave);
    const int64_t total = rows * units_per_row;
    for (int64_t id = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; id < total;
         id += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = id / units_per_row;
        const int64_t unit = id - r * units_per_row;
        const int u = (int)(unit & 7);
        const uint32_t* blk = codes + r * rs + block_col_base(unit >> 3, rows, wpb, interleave);
        uint32_t w[K + 1];
        #pragma unroll
        for (int j = 0; j < K; ++j) w[j] = __ldg(blk + u * K + j);
        // neighbour: first word of the next unit of the same block (unit 7 -> unit 0)
        w[K] = __ldg(blk + ((u == 7) ? 0 : (u + 1) * K));
        const float s = bf16_bits_to_float(scales[r]);
        // columns c0 .. c0+31 of this unit; window i is column c0 + 31 - i
        const int64_t c0 = (unit >> 3) * kBT + (224 - 32 * u);
        uint32_t wp[16], vp[16];  // bf16 / u16 pairs in ascending column order
        #pragma unroll
        for (int e = 0; e < 32; e += 2) {
            // columns c0+e (window 31-e) and c0+e+1 (window 30-e)
            const uint32_t o_lo = win_off<K>(w, 31 - e);
            const uint32_t o_hi = win_off<K>(w, 30 - e);
            const __nv_bfloat162 h = __floats2bfloat162_rn(__fmul_rn(lut_at(lut_s, o_lo), s),
                                                           __fmul_rn(lut_at(lut_s, o_hi), s));
            wp[e / 2] = *reinterpret_cast<const uint32_t*>(&h);
            vp[e / 2] = (o_lo >> 2) | ((o_hi >> 2) << 16);
        }
        uint4* wdst = reinterpret_cast<uint4*>(w_out + r * cols + c0);
        #pragma unroll
        for (int q = 0; q < 4; ++q)
            wdst[q] = make_uint4(wp[4 * q], wp[4 * q + 1], wp[4 * q + 2], wp[4 * q + 3]);
        if (win_out) {
            uint4* vdst = reinterpret_cast<uint4*>(win_out + r * cols + c0);
            #pragma unroll
            for (int q = 0; q < 4; ++q)
                vdst[q] = make_uint4(vp[4 * q], vp[4 * q + 1], vp[4 * q + 2], vp[4 * q + 3]);
        }
    }
}

}  // namespace

cudaError_t launch_expand(const Packed& p, uint16_t* w_out, uint16_t* win_out,
                          int sm_count, cudaStream_t stream) {
    const int64_t units = p.cols / 32;
    const int64_t total = p.rows * units;
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = (int64_t)sm_count * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    switch (p.k) {
        case 2: expand_kernel<2><<<(unsigned)blocks, 256, 0, stream>>>(p.codes, p.scales, p.lut, p.rows, units, p.interleave, w_out, win_out); break;
        case 3: expand_kernel<3><<<(unsigned)blocks, 256, 0, stream>>>(p.codes, p.scales, p.lut, p.rows, units, p.interleave, w_out, win_out); break;
        case 4: expand_kernel<4><<<(unsigned)blocks, 256, 0, stream>>>(p.codes, p.scales, p.lut, p.rows, units, p.interleave, w_out, win_out); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace tcq
