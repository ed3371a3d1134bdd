// Glue of a SwiGLU MLP layer (RMSNorm, silu * up) and the shared-memory
// gather probe.  None of this is a step of the trellis method.
#include "common.cuh"
#include "internal.h"

namespace tcq {
namespace {

// One CTA per activation row, the row held in registers: 16-byte loads of 8
// values, fp32 sum of squares, then x * rsqrt(mean + eps) and 16-byte
// stores -- one pass over memory (rows of 8 * 256 * kRmsChunks values at
// most; x and out 16-byte aligned, D a multiple of 8).
constexpr int kRmsChunks = 4;
__global__ void __launch_bounds__(256)
rmsnorm_vec_kernel(const uint16_t* __restrict__ x, int64_t D, float eps, uint16_t* __restrict__ out) {
    __shared__ float part[8];
    pdl_wait();
    pdl_release();
    const uint4* xr = reinterpret_cast<const uint4*>(x + (int64_t)blockIdx.x * D);
    uint4* orow = reinterpret_cast<uint4*>(out + (int64_t)blockIdx.x * D);
    const int nc = (int)(D >> 3);
    uint4 v[kRmsChunks];
    float ss = 0.f;
    #pragma unroll
    for (int i = 0; i < kRmsChunks; ++i) {
        const int c = threadIdx.x + 256 * i;
        v[i] = c < nc ? xr[c] : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
        #pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float lo = bf16_bits_to_float(w[q] & 0xffffu), hi = bf16_bits_to_float(w[q] >> 16);
            ss = fmaf(lo, lo, ss);
            ss = fmaf(hi, hi, ss);
        }
    }
    #pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
    #pragma unroll
    for (int w = 0; w < 8; ++w) tot += part[w];
    const float inv = 1.0f / sqrtf(tot / (float)D + eps);
    #pragma unroll
    for (int i = 0; i < kRmsChunks; ++i) {
        const int c = threadIdx.x + 256 * i;
        if (c >= nc) continue;
        const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
        uint32_t o[4];
        #pragma unroll
        for (int q = 0; q < 4; ++q)
            o[q] = pack_bf16x2(bf16_bits_to_float(w[q] & 0xffffu) * inv, bf16_bits_to_float(w[q] >> 16) * inv);
        orow[c] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// One CTA per activation row: fp32 sum of squares, then x * rsqrt(mean + eps)
// (any D and alignment; two passes over the row).
__global__ void __launch_bounds__(256)
rmsnorm_kernel(const uint16_t* __restrict__ x, int64_t D, float eps, uint16_t* __restrict__ out) {
    __shared__ float part[8];
    pdl_wait();
    pdl_release();
    const uint16_t* xr = x + (int64_t)blockIdx.x * D;
    uint16_t* orow = out + (int64_t)blockIdx.x * D;
    float ss = 0.f;
    for (int64_t d = threadIdx.x; d < D; d += blockDim.x) {
        const float v = bf16_bits_to_float(xr[d]);
        ss = fmaf(v, v, ss);
    }
    #pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
    #pragma unroll
    for (int w = 0; w < 8; ++w) tot += part[w];
    const float inv = 1.0f / sqrtf(tot / (float)D + eps);
    for (int64_t d = threadIdx.x; d < D; d += blockDim.x)
        orow[d] = __bfloat16_as_ushort(__float2bfloat16_rn(bf16_bits_to_float(xr[d]) * inv));
}

// out[i] = bf16_rn(in[i]): the output rounding of the packed matmul, for a
// sum that was finished outside the library (an all-reduce across GPUs).
__global__ void round_bf16_kernel(const float* __restrict__ in, int64_t n, uint16_t* __restrict__ out) {
    pdl_wait();
    pdl_release();
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        out[i] = __bfloat16_as_ushort(__float2bfloat16_rn(in[i]));
}

__global__ void silu_mul_kernel(const uint16_t* __restrict__ g, const uint16_t* __restrict__ u,
                                int64_t n, uint16_t* __restrict__ out) {
    pdl_wait();
    pdl_release();
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const float gv = bf16_bits_to_float(g[i]);
        const float uv = bf16_bits_to_float(u[i]);
        out[i] = __bfloat16_as_ushort(__float2bfloat16_rn(silu_mul_f32(gv, uv)));
    }
}

// Random 4-byte gathers from a 4096-entry shared-memory table: 8 independent
// xorshift streams per thread, one gather per draw.  Each draw costs a few
// integer operations, well under what the shared-memory port needs, so the
// kernel runs at the gather rate of the SM.  With REP = 8 (or 4) the table is
// replicated so that lane group g = lane % REP only reads banks congruent to
// g mod REP: entry e of copy g sits at word REP*e + g.
template <int REP>
__global__ void __launch_bounds__(1024, 1)
gather_probe_kernel(const float* __restrict__ lut, int iters, float* __restrict__ sink) {
    extern __shared__ __align__(16) float lut_s[];
    for (int i = threadIdx.x; i < kLutN * REP; i += blockDim.x) lut_s[i] = __ldg(lut + i / REP);
    __syncthreads();
    uint32_t st[8];
    const uint32_t tid = blockIdx.x * blockDim.x + threadIdx.x;
    const uint32_t gofs = (threadIdx.x % REP) * 4u;
    #pragma unroll
    for (int j = 0; j < 8; ++j) st[j] = 0x9E3779B9u * (tid * 8u + j + 1u);
    float acc = 0.f;
    for (int it = 0; it < iters; ++it) {
        #pragma unroll
        for (int j = 0; j < 8; ++j) {
            st[j] ^= st[j] << 13;
            st[j] ^= st[j] >> 17;
            st[j] ^= st[j] << 5;
            constexpr uint32_t mask = 0xFFFu * 4u * REP;
            acc += lut_at(lut_s, (st[j] & mask) | gofs);
        }
    }
    sink[tid] = acc;
}

}  // namespace

cudaError_t launch_rmsnorm(const uint16_t* x, int64_t M, int64_t D, float eps,
                           uint16_t* out, cudaStream_t stream) {
    const bool vec = D % 8 == 0 && D <= (int64_t)8 * 256 * kRmsChunks &&
                     (reinterpret_cast<uintptr_t>(x) & 15u) == 0 && (reinterpret_cast<uintptr_t>(out) & 15u) == 0;
    const cudaError_t e = vec ? launch_pdl(rmsnorm_vec_kernel, dim3((unsigned)M), dim3(256), 0, stream, x, D, eps, out)
                              : launch_pdl(rmsnorm_kernel, dim3((unsigned)M), dim3(256), 0, stream, x, D, eps, out);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_silu_mul(const uint16_t* g, const uint16_t* u, int64_t n,
                            uint16_t* out, cudaStream_t stream) {
    int64_t blocks = (n + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    if (blocks < 1) blocks = 1;
    const cudaError_t e = launch_pdl(silu_mul_kernel, dim3((unsigned)blocks), dim3(256), 0, stream, g, u, n, out);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_round_bf16(const float* in, int64_t n, uint16_t* out, cudaStream_t stream) {
    int64_t blocks = (n + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    if (blocks < 1) blocks = 1;
    const cudaError_t e = launch_pdl(round_bf16_kernel, dim3((unsigned)blocks), dim3(256), 0, stream, in, n, out);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_gather_probe(const float* lut, int blocks, int iters, int replicas, float* sink,
                                cudaStream_t stream) {
    const size_t smem = (size_t)kLutN * replicas * sizeof(float);
    cudaError_t e = cudaSuccess;
    switch (replicas) {
        case 1: gather_probe_kernel<1><<<(unsigned)blocks, 1024, smem, stream>>>(lut, iters, sink); break;
        case 4:
            e = cudaFuncSetAttribute(gather_probe_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            gather_probe_kernel<4><<<(unsigned)blocks, 1024, smem, stream>>>(lut, iters, sink); break;
        case 8:
            e = cudaFuncSetAttribute(gather_probe_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            gather_probe_kernel<8><<<(unsigned)blocks, 1024, smem, stream>>>(lut, iters, sink); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace tcq
