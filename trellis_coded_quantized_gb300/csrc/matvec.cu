// trellis_matvec: M = 1 axis-1 packed matvec, out[r] = bf16(sum_c x[c] w[r][c]).
//
// Arithmetic: the decoded weight is bf16(f32(lut[win] * scale[r])) and the
// dot product accumulates in fp32 (@mlx-bun/inference 1.0.0,
// kernels/trellis/tiled-prefill.ts, prefill tile kernel; the pages name the
// default M=1 matvec without showing it, and wide-prefill.ts shows the
// shuffle reduction of per-lane partial sums).
//
// GB300 layout of the work (warp FMA, no tensor cores at M = 1):
//   - one CTA per SM, up to 640 threads; the codebook sits in shared memory
//     as 8 interleaved copies (128 KB), lane group lane % 8 reading only its
//     own 4 banks, which cuts the bank conflicts of the random gathers;
//   - a "row group" of TG threads covers one whole row: thread t owns the
//     32-column unit t of every row and keeps those 32 activations in
//     registers as bf16 pairs for the whole kernel, so x is read once per CTA;
//   - per row, a thread streams its unit's k words (one 16/8-byte load, or
//     three 4-byte loads at k=3, coalesced across the warp; two rows ahead),
//     takes the neighbour word from the next lane with __shfl_sync, and does
//     32 window extractions, codebook gathers and scale multiplies, 16 paired
//     bf16 roundings and 32 bf16 x bf16 -> f32 FMAs;
//   - RB rows are accumulated side by side, then a butterfly reduce-scatter
//     over the warp (RB shuffles for RB rows) and a sum over the warps of the
//     group in shared memory produce the RB outputs.
// The unrounded contract (scatter.ts, balanced scatter kernels; the default
// matvec per tiled-prefill.ts) drops the bf16 rounding of the weight: the
// codebook values are contracted with x in f32 and the row's scale
// multiplies the row sum, one multiply per row instead of one per weight.
#include "common.cuh"
#include "internal.h"

namespace tcq {
namespace {

// Threads per CTA and rows per reduction batch (a power of two <= 32); the
// macros let a build try other shapes.
#ifndef TCQ_MV_THREADS
#define TCQ_MV_THREADS 640
#endif
#ifndef TCQ_MV_RB
#define TCQ_MV_RB 16
#endif
constexpr int kMvThreads = TCQ_MV_THREADS;
constexpr int kRB = TCQ_MV_RB;

// Butterfly reduce-scatter of a[0..RB) over the 32 lanes: afterwards a[0] of
// lane l holds the warp sum of row (l >> (5 - log2 RB)) & (RB - 1).
template <int N>
__device__ __forceinline__ void rs_stage(float* a, int lane, int off) {
    const bool upper = (lane & off) != 0;
    #pragma unroll
    for (int j = 0; j < N; ++j) {
        const float send = upper ? a[j] : a[j + N];
        const float keep = upper ? a[j + N] : a[j];
        a[j] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
}

// Reduce-scatter of RB row sums over the warp: log2(RB) halving stages, then
// plain butterfly stages; afterwards lane l holds row (l >> (5 - log2 RB)) & (RB-1).
template <int RB>
__device__ __forceinline__ float reduce_scatter(float* a, int lane) {
    static_assert(RB == 8 || RB == 16 || RB == 32, "batch of 8, 16 or 32 rows");
    if constexpr (RB == 32) rs_stage<16>(a, lane, 16);
    if constexpr (RB >= 16) rs_stage<8>(a, lane, RB == 32 ? 8 : 16);
    rs_stage<4>(a, lane, RB == 32 ? 4 : RB == 16 ? 8 : 16);
    rs_stage<2>(a, lane, RB == 32 ? 2 : RB == 16 ? 4 : 8);
    rs_stage<1>(a, lane, RB == 32 ? 1 : RB == 16 ? 2 : 4);
    #pragma unroll
    for (int off = (RB == 32 ? 0 : RB == 16 ? 1 : 2); off >= 1; off >>= 1)
        a[0] += __shfl_xor_sync(0xffffffffu, a[0], off);
    return a[0];
}
constexpr int kRowShift = kRB == 32 ? 0 : kRB == 16 ? 1 : 2;   // lane -> row of the batch

// GATEUP: the gate and up projections of a SwiGLU layer in one launch.  The
// kernel walks 2*rows "virtual" rows, 2r the gate's row r and 2r+1 the up
// projection's; a CTA owns whole pairs, and the epilogue writes
// out[r] = bf16(silu(bf16(gate_r)) * bf16(up_r)) instead of the two sums.
template <int K, bool UNR, bool GATEUP>
__global__ void __launch_bounds__(kMvThreads, 1)
matvec_kernel(const uint16_t* __restrict__ x, const uint32_t* __restrict__ codes,
              const uint16_t* __restrict__ scales, const uint32_t* __restrict__ codes_u,
              const uint16_t* __restrict__ scales_u, const float* __restrict__ lut,
              int rows, int units, int tg, int ng, int interleave, uint16_t* __restrict__ out) {
    extern __shared__ __align__(16) float smem[];
    pdl_release();
    // The codebook, codes and scales are read before griddepcontrol.wait,
    // while the previous kernel of the stream may still be finishing; only
    // the activations (and the output) wait for it.
    float* lut_s = smem;                              // 8-way replicated codebook
    const int wg = tg >> 5;                           // warps per row group
    float* red = smem + kLutN * kLutRep;              // [2][ng][wg][kRB]
    stage_lut_rep8(lut_s, lut);

    const int g = threadIdx.x / tg;
    const int t = threadIdx.x - g * tg;
    const int lane = threadIdx.x & 31;
    const int wig = t >> 5;
    const bool active = t < units;
    const int64_t wpr = block_row_stride(units / kUnitsPerBlock, kBT * K / 32, interleave);
    const uint32_t gofs = lut_rep_lane_offset();


    // this CTA's (virtual) rows [r0, r1)
    const int vm = GATEUP ? 2 : 1;
    const int r0 = vm * (int)((int64_t)rows * blockIdx.x / gridDim.x);
    const int r1 = vm * (int)((int64_t)rows * (blockIdx.x + 1) / gridDim.x);
    const int per_group = (r1 - r0 + ng - 1) / ng;
    const int src = next_unit_lane(lane);
    const int64_t tofs = active ? block_col_base(t >> 3, rows, kBT * K / 32, interleave) + (t & 7) * K : 0;
    const uint32_t* tp = codes + tofs;
    const uint32_t* tpu = GATEUP ? codes_u + tofs : tp;
    // this thread's words of virtual row v, and the scale of v
    auto row_words = [&](int v) -> const uint32_t* {
        if constexpr (GATEUP) return ((v & 1) ? tpu : tp) + (int64_t)(v >> 1) * wpr;
        else return tp + (int64_t)v * wpr;
    };
    auto row_scale = [&](int v) -> float {
        if constexpr (GATEUP) return bf16_bits_to_float(__ldg(((v & 1) ? scales_u : scales) + (v >> 1)));
        else return bf16_bits_to_float(__ldg(scales + v));
    };

    // two rows in flight ahead of the one being decoded
    uint32_t pa[K], pb[K];
    {
        const int ra = r0 + g, rb = r0 + g + ng;
        if (active && ra < r1) load_unit<K>(pa, row_words(ra));
        else {
            #pragma unroll
            for (int j = 0; j < K; ++j) pa[j] = 0u;
        }
        if (active && rb < r1) load_unit<K>(pb, row_words(rb));
        else {
            #pragma unroll
            for (int j = 0; j < K; ++j) pb[j] = 0u;
        }
    }

    pdl_wait();
    // activations of this thread's unit as bf16 pairs: xp[j] holds windows
    // 2j (high half) and 2j+1 (low half), i.e. columns c0+31-2j and c0+30-2j
    uint32_t xp[16];
    if (active) {
        const int c0 = (t >> 3) * kBT + (224 - 32 * (t & 7));
        const uint4* src = reinterpret_cast<const uint4*>(x + c0);
        #pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 v = __ldg(src + q);
            // word e of chunk q holds columns c0+8q+2e (lo) and c0+8q+2e+1 (hi)
            xp[15 - 4 * q] = v.x;
            xp[14 - 4 * q] = v.y;
            xp[13 - 4 * q] = v.z;
            xp[12 - 4 * q] = v.w;
        }
    } else {
        #pragma unroll
        for (int j = 0; j < 16; ++j) xp[j] = 0u;
    }
    __syncthreads();

    int buf = 0;
    for (int j0 = 0; j0 < per_group; j0 += kRB, buf ^= 1) {
        float acc[kRB];
        #pragma unroll
        for (int rho = 0; rho < kRB; ++rho) {
            const int row = r0 + g + ng * (j0 + rho);
            uint32_t w[K + 1];
            #pragma unroll
            for (int j = 0; j < K; ++j) { w[j] = pa[j]; pa[j] = pb[j]; }
            const int rn = row + 2 * ng;
            if (active && rn < r1) load_unit<K>(pb, row_words(rn));
            acc[rho] = 0.f;
            if (row < r1) {                              // uniform over the row group
                w[K] = __shfl_sync(0xffffffffu, w[0], src);
                float a0 = 0.f, a1 = 0.f;
                if constexpr (UNR) {
                    #pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float v0 = lut_at(lut_s, win_off_sh<K, kLutRepShift>(w, 2 * j) | gofs);
                        const float v1 = lut_at(lut_s, win_off_sh<K, kLutRepShift>(w, 2 * j + 1) | gofs);
                        a0 = fmaf(v0, __uint_as_float(xp[j] & 0xffff0000u), a0);
                        a1 = fmaf(v1, __uint_as_float(xp[j] << 16), a1);
                    }
                } else {
                    const float s = row_scale(row);
                    #pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float v0 = lut_at(lut_s, win_off_sh<K, kLutRepShift>(w, 2 * j) | gofs);
                        const float v1 = lut_at(lut_s, win_off_sh<K, kLutRepShift>(w, 2 * j + 1) | gofs);
                        // pair laid out like xp[j]: window 2j high, window 2j+1 low
                        const uint32_t wp = pack_bf16x2(__fmul_rn(v1, s), __fmul_rn(v0, s));
                        a0 = fma_bf16_hi(wp, xp[j], a0);
                        a1 = fma_bf16_lo(wp, xp[j], a1);
                    }
                }
                acc[rho] = a0 + a1;
            }
        }
        // rows of this batch: warp reduce-scatter, then sum the warps of the group
        const float v = reduce_scatter<kRB>(acc, lane);
        float* rb = red + (size_t)buf * ng * wg * kRB;
        if ((lane & ((1 << kRowShift) - 1)) == 0) rb[((size_t)g * wg + wig) * kRB + ((lane >> kRowShift) & (kRB - 1))] = v;
        __syncthreads();
        if constexpr (GATEUP) {
            // the batch is the contiguous virtual rows base .. base + ng*kRB - 1
            // (row g + ng*t of the batch sits at rb[g][.][t]); thread i takes pair i
            const int base = r0 + ng * j0;
            const int i = threadIdx.x;
            if (i < ng * kRB / 2 && base + 2 * i < r1) {
                float sum[2];
                #pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int o = 2 * i + h, og = o % ng, ot = o / ng;
                    float a = 0.f;
                    for (int w = 0; w < wg; ++w) a += rb[((size_t)og * wg + w) * kRB + ot];
                    if constexpr (UNR) a *= row_scale(base + o);
                    sum[h] = bf16_bits_to_float(__bfloat16_as_ushort(__float2bfloat16_rn(a)));
                }
                out[(base >> 1) + i] = __bfloat16_as_ushort(__float2bfloat16_rn(silu_mul_f32(sum[0], sum[1])));
            }
        } else if (t < kRB) {
            const int row = r0 + g + ng * (j0 + t);
            if (row < r1) {
                float sum = 0.f;
                for (int w = 0; w < wg; ++w) sum += rb[((size_t)g * wg + w) * kRB + t];
                if constexpr (UNR) sum *= row_scale(row);
                out[row] = __bfloat16_as_ushort(__float2bfloat16_rn(sum));
            }
        }
        // the other buffer is written next; one barrier per batch suffices
    }
}

template <int K, bool UNR, bool GATEUP>
cudaError_t launch_mv(const Packed& p, const uint32_t* codes_u, const uint16_t* scales_u, const uint16_t* x,
                      uint16_t* out, int grid, int threads, size_t smem, int units, int tg, int ng,
                      cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(matvec_kernel<K, UNR, GATEUP>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(matvec_kernel<K, UNR, GATEUP>, dim3(grid), dim3(threads), smem, stream, x, p.codes, p.scales,
                   codes_u, scales_u, p.lut, (int)p.rows, units, tg, ng, p.interleave, out);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <bool GATEUP>
cudaError_t launch_any(const Packed& p, const uint32_t* codes_u, const uint16_t* scales_u, const uint16_t* x,
                       uint16_t* out, int sm_count, cudaStream_t stream) {
    const int units = (int)(p.cols / 32);
    const int tg = ((units + 31) / 32) * 32;
    if (tg > kMvThreads) return cudaErrorInvalidValue;
    int ng = kMvThreads / tg;
    const int threads = tg * ng;
    int grid = sm_count;
    if ((int64_t)grid > p.rows) grid = (int)p.rows;
    const size_t smem = kLutRepBytes + (size_t)(2 * ng * (tg / 32) * kRB) * sizeof(float);
    switch (p.k * 2 + (p.unrounded ? 1 : 0)) {
        case 4: return launch_mv<2, false, GATEUP>(p, codes_u, scales_u, x, out, grid, threads, smem, units, tg, ng, stream);
        case 5: return launch_mv<2, true, GATEUP>(p, codes_u, scales_u, x, out, grid, threads, smem, units, tg, ng, stream);
        case 6: return launch_mv<3, false, GATEUP>(p, codes_u, scales_u, x, out, grid, threads, smem, units, tg, ng, stream);
        case 7: return launch_mv<3, true, GATEUP>(p, codes_u, scales_u, x, out, grid, threads, smem, units, tg, ng, stream);
        case 8: return launch_mv<4, false, GATEUP>(p, codes_u, scales_u, x, out, grid, threads, smem, units, tg, ng, stream);
        case 9: return launch_mv<4, true, GATEUP>(p, codes_u, scales_u, x, out, grid, threads, smem, units, tg, ng, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_matvec(const Packed& p, const uint16_t* x, uint16_t* out,
                          int sm_count, cudaStream_t stream) {
    return launch_any<false>(p, nullptr, nullptr, x, out, sm_count, stream);
}

cudaError_t launch_gate_up_matvec(const Packed& gate, const uint32_t* up_codes, const uint16_t* up_scales,
                                  const uint16_t* x, uint16_t* h, int sm_count, cudaStream_t stream) {
    return launch_any<true>(gate, up_codes, up_scales, x, h, sm_count, stream);
}

}  // namespace tcq
