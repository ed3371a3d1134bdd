// TurboQuant packed K/V decode (@mlx-bun/inference 1.0.0,
// kernels/turboquant/decode.ts, joint K/V decode kernel, and
// kernels/turboquant/inverse.ts, the decode with the inverse 256-point
// rotation of the values).
//
// Row r of the cache holds D keys at KBITS bits and D values at VBITS bits,
// code `col` at bit offset col * BITS of the row's byte string, low bits
// first.  The keys are bf16((f32(code) + f32(zero)) * f32(scale)) -- the
// zero is added before the scale, in f32 -- with an 8-bit key code read as a
// signed byte; the values are f32(centroid[code]) * f32(scale).  Scales and
// zeros hold one entry per group of KG (keys) or VG (values) columns.
//
// GB300 layout of the work: plain HBM streaming, no tensor cores.  A thread
// owns 8 consecutive columns of one row, so its key codes are KBITS whole
// bytes and its value codes VBITS whole bytes starting on a byte boundary
// (one 8/4/2-byte load when aligned, byte loads for 3 and 5); a warp reads a
// contiguous run of each row's codes.  The 8 keys leave as one 16-byte store,
// the values as one (bf16) or two (f32) 16-byte stores.  The centroid table
// (at most 256 floats) is staged in shared memory per CTA.
//
// The inverse kernel gives each row to one warp: lane l holds columns
// 8l .. 8l+7, so column bits 0..2 are the register index and bits 3..7 the
// lane.  The Walsh-Hadamard butterflies run in the page's order (bits 0, 1,
// 2, 3, then 4, 5, 6, 7; each stage a + b and a - b in f32): bits 0..2 in
// registers, bits 3..7 across lanes with __shfl_xor_sync.  Same operands in
// the same order as the page's two radix-16 passes, so the f32 results are
// the same; then x 1/16 (exact), x sign[col], bf16.
#include <cuda_fp16.h>

#include "common.cuh"
#include "internal.h"

namespace tcq {
namespace {

constexpr int kTqThreads = 256;
constexpr int kTqUnroll = 1;          // chunks per thread and iteration (joint decode)
constexpr int kTqRowUnroll = 1;       // rows per warp and iteration (inverse)

__device__ __forceinline__ float load_scalar(const void* p, int64_t i, int dtype) {
    if (dtype == kDtF32) return __ldg(static_cast<const float*>(p) + i);
    const uint16_t b = __ldg(static_cast<const uint16_t*>(p) + i);
    if (dtype == kDtF16) return __half2float(__ushort_as_half(b));
    return bf16_bits_to_float(b);
}

// NB bytes of a code run starting at byte offset `off` of `row` (NB <= 8),
// little endian: byte 0 in bits 0..7.
template <int NB>
__device__ __forceinline__ uint64_t load_run(const uint8_t* __restrict__ row, int64_t off) {
    const uint8_t* p = row + off;
    if constexpr (NB == 8) {
        return __ldg(reinterpret_cast<const unsigned long long*>(p));
    } else if constexpr (NB == 4) {
        return __ldg(reinterpret_cast<const unsigned int*>(p));
    } else if constexpr (NB == 2) {
        return __ldg(reinterpret_cast<const unsigned short*>(p));
    } else {
        uint64_t v = 0;
        #pragma unroll
        for (int i = 0; i < NB; ++i) v |= (uint64_t)__ldg(p + i) << (8 * i);
        return v;
    }
}

// The 8 keys of one thread's columns (bf16 pairs) from its code run.
template <int KB>
__device__ __forceinline__ uint4 decode_keys8(uint64_t run, float zero, float scale) {
    uint32_t w[4];
    #pragma unroll
    for (int p = 0; p < 4; ++p) {
        float k[2];
        #pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int e = 2 * p + h;
            const uint32_t u = (uint32_t)(run >> (e * KB)) & ((1u << KB) - 1u);
            const float code = KB == 8 ? (float)(int)(int8_t)(uint8_t)u : (float)u;
            k[h] = __fmul_rn(__fadd_rn(code, zero), scale);
        }
        w[p] = pack_bf16x2(k[0], k[1]);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

template <int KB, int VB>
__global__ void __launch_bounds__(kTqThreads)
kv_decode_kernel(const uint8_t* __restrict__ kp, const void* __restrict__ ks, const void* __restrict__ kz,
                 const uint8_t* __restrict__ vp, const void* __restrict__ vs, const float* __restrict__ centroids,
                 int64_t rows, int D, int kg, int vg, int ks_dt, int kz_dt, int vs_dt, int v_bf16,
                 uint16_t* __restrict__ k_out, void* __restrict__ v_out) {
    __shared__ float cent[1 << VB];
    pdl_release();
    for (int i = threadIdx.x; i < (1 << VB); i += blockDim.x) cent[i] = __ldg(centroids + i);
    // the centroid table is a constant input; the codes and scales (written
    // at run time by the cache update) and the outputs wait for the
    // previous kernel of the stream
    pdl_wait();
    __syncthreads();
    const int cpr = D >> 3;           // 8-column chunks per row: 8 .. 64, a power of two
    const int cshift = 31 - __clz(cpr);
    const int64_t total = rows * cpr;
    const int kgs = 31 - __clz(kg), vgs = 31 - __clz(vg);   // groups of 32 or 64
    const int kgr = D >> kgs, vgr = D >> vgs;
    // kTqUnroll chunks per thread and iteration, all their loads issued
    // before the first is used
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t t0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t0 < total; t0 += kTqUnroll * stride) {
        uint64_t krun[kTqUnroll], vrun[kTqUnroll];
        float kzv[kTqUnroll], ksv[kTqUnroll], vsv[kTqUnroll];
        #pragma unroll
        for (int u = 0; u < kTqUnroll; ++u) {
            const int64_t t = t0 + u * stride;
            if (t >= total) break;
            const int64_t r = t >> cshift;
            const int c = (int)t & (cpr - 1);
            const int col = c << 3;
            krun[u] = load_run<KB>(kp + r * (int64_t)(D * KB / 8), (int64_t)c * KB);
            vrun[u] = load_run<VB>(vp + r * (int64_t)(D * VB / 8), (int64_t)c * VB);
            const int64_t kgi = r * kgr + (col >> kgs);
            kzv[u] = load_scalar(kz, kgi, kz_dt);
            ksv[u] = load_scalar(ks, kgi, ks_dt);
            vsv[u] = load_scalar(vs, r * vgr + (col >> vgs), vs_dt);
        }
        #pragma unroll
        for (int u = 0; u < kTqUnroll; ++u) {
            const int64_t t = t0 + u * stride;
            if (t >= total) break;
            const int64_t r = t >> cshift;
            const int col = ((int)t & (cpr - 1)) << 3;
            *reinterpret_cast<uint4*>(k_out + r * D + col) = decode_keys8<KB>(krun[u], kzv[u], ksv[u]);
            float v[8];
            #pragma unroll
            for (int e = 0; e < 8; ++e)
                v[e] = __fmul_rn(cent[(uint32_t)(vrun[u] >> (e * VB)) & ((1u << VB) - 1u)], vsv[u]);
            if (v_bf16) {
                const uint4 o = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                                           pack_bf16x2(v[6], v[7]));
                *reinterpret_cast<uint4*>(static_cast<uint16_t*>(v_out) + r * D + col) = o;
            } else {
                float4* o = reinterpret_cast<float4*>(static_cast<float*>(v_out) + r * D + col);
                o[0] = make_float4(v[0], v[1], v[2], v[3]);
                o[1] = make_float4(v[4], v[5], v[6], v[7]);
            }
        }
    }
}

// One warp per row; D = 256, 8-bit keys, 3-bit values, groups of 32.
__global__ void __launch_bounds__(kTqThreads, 6)
kv_inverse256_kernel(const uint8_t* __restrict__ kp, const void* __restrict__ ks, const void* __restrict__ kz,
                     const uint8_t* __restrict__ vp, const void* __restrict__ vs,
                     const float* __restrict__ centroids, const float* __restrict__ signs, int64_t rows,
                     int ks_dt, int kz_dt, int vs_dt, uint16_t* __restrict__ k_out, uint16_t* __restrict__ v_out) {
    __shared__ float cent[8];
    __shared__ float sgn[256];
    pdl_release();
    const int lane = threadIdx.x & 31;
    if (threadIdx.x < 8) cent[threadIdx.x] = __ldg(centroids + threadIdx.x);
    for (int i = threadIdx.x; i < 256; i += blockDim.x) sgn[i] = __ldg(signs + i);
    pdl_wait();
    __syncthreads();
    const int col = 8 * lane;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t r0 = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r0 < rows;
         r0 += kTqRowUnroll * warps) {
        uint64_t krun[kTqRowUnroll], vrun[kTqRowUnroll];
        float kzv[kTqRowUnroll], ksv[kTqRowUnroll], vsv[kTqRowUnroll];
        #pragma unroll
        for (int u = 0; u < kTqRowUnroll; ++u) {
            const int64_t r = r0 + u * warps;
            if (r >= rows) break;
            const int64_t gi = r * 8 + (col >> 5);       // 8 groups of 32 per row
            krun[u] = load_run<8>(kp + r * 256, col);
            vrun[u] = load_run<3>(vp + r * 96, 3 * lane);
            kzv[u] = load_scalar(kz, gi, kz_dt);
            ksv[u] = load_scalar(ks, gi, ks_dt);
            vsv[u] = load_scalar(vs, gi, vs_dt);
        }
        #pragma unroll
        for (int u = 0; u < kTqRowUnroll; ++u) {
            const int64_t r = r0 + u * warps;
            if (r >= rows) break;                        // uniform over the warp
            *reinterpret_cast<uint4*>(k_out + r * 256 + col) = decode_keys8<8>(krun[u], kzv[u], ksv[u]);
            float x[8];
            #pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = __fmul_rn(cent[(uint32_t)(vrun[u] >> (3 * e)) & 7u], vsv[u]);
            // column bits 0, 1, 2: pairs of registers
            #pragma unroll
            for (int st = 0; st < 3; ++st) {
                const int h = 1 << st;
                #pragma unroll
                for (int e = 0; e < 8; ++e) {
                    if (e & h) continue;
                    const float a = x[e], b = x[e + h];
                    x[e] = __fadd_rn(a, b);
                    x[e + h] = __fsub_rn(a, b);
                }
            }
            // column bits 3..7: lane bits 0..4; the lane with the bit clear holds a
            #pragma unroll
            for (int st = 0; st < 5; ++st) {
                const int m = 1 << st;
                const bool upper = (lane & m) != 0;
                #pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float p = __shfl_xor_sync(0xffffffffu, x[e], m);
                    x[e] = upper ? __fsub_rn(p, x[e]) : __fadd_rn(x[e], p);
                }
            }
            uint32_t w[4];
            #pragma unroll
            for (int p = 0; p < 4; ++p)
                w[p] = pack_bf16x2(__fmul_rn(__fmul_rn(x[2 * p], 0.0625f), sgn[col + 2 * p]),
                                   __fmul_rn(__fmul_rn(x[2 * p + 1], 0.0625f), sgn[col + 2 * p + 1]));
            *reinterpret_cast<uint4*>(v_out + r * 256 + col) = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

// Enough CTAs for the work, at most one full wave (`per_sm` resident CTAs
// per SM); the kernels loop over the rest.
int tq_grid(int64_t work_items, int per_block, int sm_count, int per_sm) {
    int64_t g = (work_items + per_block - 1) / per_block;
    const int64_t cap = (int64_t)(sm_count > 0 ? sm_count : 152) * per_sm;
    if (g > cap) g = cap;
    return g < 1 ? 1 : (int)g;
}

template <int KB, int VB>
cudaError_t launch_kv(const KvArgs& a, int sm_count, cudaStream_t stream) {
    const int grid = tq_grid(a.rows * (a.D / 8), kTqThreads, sm_count, 8);
    const cudaError_t e = launch_pdl(kv_decode_kernel<KB, VB>, dim3(grid), dim3(kTqThreads), 0, stream, a.kp, a.ks,
                                     a.kz, a.vp, a.vs, a.centroids, a.rows, a.D, a.kg, a.vg, a.ks_dt, a.kz_dt,
                                     a.vs_dt, a.v_bf16, static_cast<uint16_t*>(a.k_out), a.v_out);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int KB>
cudaError_t launch_kv_k(const KvArgs& a, int sm_count, cudaStream_t stream) {
    switch (a.vbits) {
        case 2: return launch_kv<KB, 2>(a, sm_count, stream);
        case 3: return launch_kv<KB, 3>(a, sm_count, stream);
        case 4: return launch_kv<KB, 4>(a, sm_count, stream);
        case 5: return launch_kv<KB, 5>(a, sm_count, stream);
        case 8: return launch_kv<KB, 8>(a, sm_count, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_kv_decode(const KvArgs& a, int sm_count, cudaStream_t stream) {
    switch (a.kbits) {
        case 2: return launch_kv_k<2>(a, sm_count, stream);
        case 4: return launch_kv_k<4>(a, sm_count, stream);
        case 5: return launch_kv_k<5>(a, sm_count, stream);
        case 8: return launch_kv_k<8>(a, sm_count, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_kv_inverse256(const KvArgs& a, const float* signs, int sm_count, cudaStream_t stream) {
    const int grid = tq_grid(a.rows, kTqThreads / 32, sm_count, 6);
    const cudaError_t e = launch_pdl(kv_inverse256_kernel, dim3(grid), dim3(kTqThreads), 0, stream, a.kp, a.ks, a.kz,
                                     a.vp, a.vs, a.centroids, signs, a.rows, a.ks_dt, a.kz_dt, a.vs_dt,
                                     static_cast<uint16_t*>(a.k_out), static_cast<uint16_t*>(a.v_out));
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace tcq
