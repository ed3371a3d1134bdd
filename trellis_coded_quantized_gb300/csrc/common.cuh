// Device primitives shared by the libtrellis kernels (sm_103a).
//
// A "unit" is 32 consecutive symbol slots of one block, starting on a word
// boundary: unit u (0..7) of a block holds block bits [32uk, 32uk + 32k), i.e.
// words [u*k, u*k + k).  Window i (0..31) of the unit starts at unit-local bit
// k*i and belongs to block column t = 255 - 32u - i (the window of column t
// starts at block bit (BT-1-t)*k: @mlx-bun/inference 1.0.0,
// kernels/trellis/tiled-prefill.ts, prefill tile kernel).  The last window
// spills into the first word of the next unit of the same block, and unit 7
// spills into unit 0 (the tail-biting wrap to word 0 of the block).  A unit
// therefore needs its k words plus one neighbour word.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace tcq {

constexpr int kBT = 256;        // block length in columns
constexpr int kL = 12;          // window bits
constexpr int kLutN = 1 << kL;  // codebook entries
constexpr int kUnitsPerBlock = kBT / 32;

// Byte offset 4*win of window i of a unit held in w[0..K] (w[K] = neighbour).
// The shift is taken two bits early so the masked value is the table offset.
// With i a compile-time constant after unrolling, this is one funnel shift and
// one AND.
template <int K>
__device__ __forceinline__ uint32_t win_off(const uint32_t* w, int i) {
    const int b = K * i;
    const int q = b >> 5;
    const int s = b & 31;
    uint32_t f;
    if (s >= 2)
        f = __funnelshift_r(w[q], w[q + 1], s - 2);
    else if (q > 0)
        f = __funnelshift_r(w[q - 1], w[q], 30 + s);
    else
        f = w[0] << (2 - s);
    return f & 0x3FFCu;
}

// The same with the window placed at bit SH of the result: the byte offset of
// entry win in a table whose entries are 2^SH bytes apart (SH = 5 for the
// 8-way replicated codebook below, where the lane's copy is OR-ed in).
template <int K, int SH>
__device__ __forceinline__ uint32_t win_off_sh(const uint32_t* w, int i) {
    const int b = K * i;
    const int q = b >> 5;
    const int s = b & 31;
    uint32_t f;
    if (s >= SH)
        f = __funnelshift_r(w[q], w[q + 1], s - SH);
    else if (q > 0)
        f = __funnelshift_r(w[q - 1], w[q], 32 - SH + s);
    else
        f = w[0] << (SH - s);
    return f & (0xFFFu << SH);
}

// 8-way replicated codebook: entry e of copy g at word 8e + g, so the copy
// of lane group g = lane % 8 lives in banks {g, g+8, g+16, g+24} and the 4
// lanes of a group only contend among themselves.  128 KB of shared memory.
constexpr int kLutRep = 8;
constexpr int kLutRepShift = 5;
constexpr size_t kLutRepBytes = (size_t)kLutN * kLutRep * sizeof(float);

// All of a thread's codebook loads are issued before its first store, so the
// staging costs one global-memory latency per 8 entries instead of one per
// entry (a CTA of 512..1024 threads stages the table in one round).
__device__ __forceinline__ void stage_lut_rep8(float* lut_s, const float* __restrict__ lut) {
    float4* dst = reinterpret_cast<float4*>(lut_s);
    for (int base = threadIdx.x; base < kLutN; base += 8 * blockDim.x) {
        float v[8];
        #pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = base + i * blockDim.x;
            v[i] = e < kLutN ? __ldg(lut + e) : 0.f;
        }
        #pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = base + i * blockDim.x;
            if (e < kLutN) {
                const float4 q = make_float4(v[i], v[i], v[i], v[i]);
                dst[2 * e] = q;
                dst[2 * e + 1] = q;
            }
        }
    }
}

// Programmatic dependent launch.  A kernel launched with
// launch_pdl() may be placed on the GPU while the previous kernel of its
// stream still runs; pdl_wait() blocks until that kernel has completed and
// its writes are visible, so it comes before the first access to memory
// that kernel may write (activations, outputs, workspace, the status word).
// The packed weights (codes, scales, codebook) are inputs that no kernel of
// this library writes, so a kernel may read them before pdl_wait().
// pdl_release() lets the next such kernel be placed.  Both are no-ops for a
// kernel launched the ordinary way (whose predecessor has then completed).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_release() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Byte offset of this lane's copy inside an entry of the replicated codebook.
__device__ __forceinline__ uint32_t lut_rep_lane_offset() {
    return (threadIdx.x & 7u) << 2;
}

// d += a.lo * b.lo (or .hi * .hi) with bf16 multiplicands and an f32
// accumulator, rounded once: equal to converting both to f32 and fmaf.
__device__ __forceinline__ float fma_bf16_lo(uint32_t a, uint32_t b, float c) {
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, al, bl, %0;\n\t}" : "+f"(c) : "r"(a), "r"(b));
    return c;
}
__device__ __forceinline__ float fma_bf16_hi(uint32_t a, uint32_t b, float c) {
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, ah, bh, %0;\n\t}" : "+f"(c) : "r"(a), "r"(b));
    return c;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ float lut_at(const float* lut_s, uint32_t byte_off) {
    return *reinterpret_cast<const float*>(reinterpret_cast<const char*>(lut_s) + byte_off);
}

// Stage the 4096-entry codebook in shared memory (16 KB, float4 copies).
__device__ __forceinline__ void stage_lut(float* lut_s, const float* __restrict__ lut) {
    const float4* src = reinterpret_cast<const float4*>(lut);
    float4* dst = reinterpret_cast<float4*>(lut_s);
    for (int i = threadIdx.x; i < kLutN / 4; i += blockDim.x) dst[i] = __ldg(src + i);
}

// Streaming loads of code words: read once, so they skip L1 allocation.
__device__ __forceinline__ uint4 ld_stream_v4(const uint32_t* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ uint2 ld_stream_v2(const uint32_t* p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
                 : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ld_stream(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// The K words of one unit at p (16-byte aligned for K=4, 8-byte for K=2).
template <int K>
__device__ __forceinline__ void load_unit(uint32_t* w, const uint32_t* p) {
    if constexpr (K == 4) {
        const uint4 v = ld_stream_v4(p);
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    } else if constexpr (K == 2) {
        const uint2 v = ld_stream_v2(p);
        w[0] = v.x; w[1] = v.y;
    } else {
        #pragma unroll
        for (int j = 0; j < K; ++j) w[j] = ld_stream(p + j);
    }
}

// Lane that holds the first word of the next unit of the same block, when
// the 8 units of a block sit on 8 consecutive lanes (unit 7 wraps to unit 0).
__device__ __forceinline__ int next_unit_lane(int lane) {
    return (lane & ~7) | ((lane + 1) & 7);
}

// Block layout of the codes.  Block b of row r starts at word
// block_col_base(b) + r * block_row_stride: interleave 0 keeps the blocks of a
// row contiguous (row stride (cols/256)*wpb); interleave 2 groups blocks in
// pairs and stores the pair of every row together, base (b/2)*R*2*wpb +
// (b%2)*wpb and row stride 2*wpb (@mlx-bun/inference 1.0.0,
// kernels/trellis/vector-expand.ts and scatter.ts, the INTERLEAVE addressing).
__host__ __device__ __forceinline__ int64_t block_col_base(int64_t b, int64_t rows, int wpb, int interleave) {
    return interleave == 2 ? (b >> 1) * rows * 2 * wpb + (b & 1) * wpb : b * wpb;
}
__host__ __device__ __forceinline__ int64_t block_row_stride(int64_t nblocks, int wpb, int interleave) {
    return interleave == 2 ? (int64_t)2 * wpb : nblocks * wpb;
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t h16) {
    return __uint_as_float(h16 << 16);
}

// silu(g) * u in f32, silu(g) = g / (1 + e^-g): the SwiGLU gate of an MLP
// layer, shared by trellis_silu_mul and the fused gate/up matvec so that the
// two chains give the same bits.
__device__ __forceinline__ float silu_mul_f32(float g, float u) {
    return g / (1.0f + expf(-g)) * u;
}

}  // namespace tcq
