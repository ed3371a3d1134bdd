// trellis_prefill: axis-1 packed matmul for M = 1..32 activation rows on the
// 5th-generation tensor cores, out[m][r] = bf16(sum_c x[m][c] w[r][c]).
//
// Arithmetic as the pages' prefill tile kernel (@mlx-bun/inference 1.0.0,
// kernels/trellis/tiled-prefill.ts): weights decoded to bf16 in the tile,
// contracted with the bf16 activations, fp32 accumulation, bf16 output.
//
// GB300 design (one CTA per 128 weight rows, whole K):
//   - the MMA is D[128 x N] += A[128 x 16] * B[16 x N] with A = decoded
//     weights (rows of the matrix are MMA rows, "swap AB") held in TENSOR
//     MEMORY, B = activations in shared memory (K-major, 128-byte swizzle),
//     D = fp32 accumulator in tensor memory; N = 16 or 32 (M padded);
//   - 8 decoder warps: warp w owns tensor-memory lane quarter w % 4 (32
//     matrix rows, one row per thread) and half w / 4 of each 256-column
//     block (4 units of 32 columns).  A thread streams its row's code words,
//     extracts windows, gathers the codebook from shared memory (8-way
//     replicated, one copy per lane group of 4, against bank conflicts), scales,
//     rounds pairs to bf16x2 and writes them with tcgen05.st straight into
//     the A stage: decoded weights never touch shared memory;
//   - 1 loader warp copies the activation tile of each block into shared
//     memory in the swizzled layout;
//   - 1 MMA warp: one thread waits for a stage, issues 16 tcgen05.mma
//     (K = 16 each) and commits to the stage's "empty" barrier;
//   - 2 stages (A: 2 x 128 tensor-memory columns, B: 2 x N x 512 bytes),
//     mbarriers with bounded waits; after the last block the accumulator is
//     read back with tcgen05.ld by the lane-quarter warps and stored as bf16.
// The K order of a block is the natural column order on both operands.
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace tcq {
namespace {

constexpr int kPfDecWarps = 8;
constexpr int kPfMmaWarp = 8;
constexpr int kPfLoadWarp = 9;
constexpr int kPfThreads = 10 * 32;
constexpr int kPfRows = 128;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kDCol = 256;            // accumulator columns [256, 256 + N)
constexpr uint64_t kWaitLimitNs = 1000000000ull;

template <int NPAD>
struct PfLayout {
    static constexpr int kXStage = NPAD * kBT * 2;        // bytes of one activation stage
    static constexpr int kXChunk = NPAD * 128;            // one 64-column K chunk
    static constexpr int kLutOff = 2 * kXStage;
    static constexpr int kBarOff = kLutOff + (int)kLutRepBytes;
    static constexpr int kBytes = kBarOff + 64;
    static constexpr int kAlloc = kBytes + 1024;          // slack for 1024-byte alignment
};

__device__ __forceinline__ uint4 ld_nc_v4(const uint32_t* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// Words of one half block of one row: 4 units (4K words) and the neighbour.
template <int K>
__device__ __forceinline__ void load_half(uint32_t* w, const uint32_t* blk, int h, bool valid) {
    if (!valid) {
        #pragma unroll
        for (int j = 0; j < 4 * K + 1; ++j) w[j] = 0u;
        return;
    }
    const uint32_t* p = blk + 4 * h * K;
    #pragma unroll
    for (int q = 0; q < K; ++q) {
        const uint4 v = ld_nc_v4(p + 4 * q);
        w[4 * q] = v.x; w[4 * q + 1] = v.y; w[4 * q + 2] = v.z; w[4 * q + 3] = v.w;
    }
    // neighbour of unit 4h+3: unit 4 of the block, or unit 0 (wrap) for h = 1
    w[4 * K] = __ldg(blk + (h == 0 ? 4 * K : 0));
}

template <int K, int NPAD>
__global__ void __launch_bounds__(kPfThreads, 1)
prefill_kernel(const uint16_t* __restrict__ x, int M, const uint32_t* __restrict__ codes,
               const uint16_t* __restrict__ scales, const float* __restrict__ lut,
               int rows, int cols, uint16_t* __restrict__ out, int* __restrict__ status) {
    using Lay = PfLayout<NPAD>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* xs = base;
    float* lut_s = reinterpret_cast<float*>(base + Lay::kLutOff);
    uint64_t* full = reinterpret_cast<uint64_t*>(base + Lay::kBarOff);
    uint64_t* empty = full + 2;
    uint64_t* done = full + 4;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(full + 5);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    stage_lut_rep8(lut_s, lut);
    if (threadIdx.x == 0) {
        tc::mbar_init(&full[0], kPfDecWarps * 32 + 32);
        tc::mbar_init(&full[1], kPfDecWarps * 32 + 32);
        tc::mbar_init(&empty[0], 1);
        tc::mbar_init(&empty[1], 1);
        tc::mbar_init(done, 1);
        *abort_flag = 0;
        tc::mbar_init_fence();
    }
    if (warp == kPfMmaWarp) {
        tc::tmem_alloc(tmem_slot, kTmemCols);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int nblocks = cols / kBT;
    constexpr int wpb = kBT * K / 32;
    const int row0 = blockIdx.x * kPfRows;

    if (warp < kPfDecWarps) {
        // ------------------------------------------------------------ decoders
        const int q = warp & 3, h = warp >> 2;
        const int row = row0 + 32 * q + lane;
        const bool valid = row < rows;
        const float s = valid ? bf16_bits_to_float(__ldg(scales + row)) : 0.f;
        const uint32_t* rowp = codes + (int64_t)(valid ? row : 0) * nblocks * wpb;
        const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
        const uint32_t gofs = lut_rep_lane_offset();
        uint32_t cw[4 * K + 1], nw[4 * K + 1];
        load_half<K>(cw, rowp, h, valid);
        for (int b = 0; b < nblocks; ++b) {
            const int stage = b & 1;
            if (b + 1 < nblocks) load_half<K>(nw, rowp + (int64_t)(b + 1) * wpb, h, valid);
            if (b >= 2 && !tc::mbar_wait(&empty[stage], ((b >> 1) - 1) & 1, abort_flag, kWaitLimitNs)) break;
            __syncwarp();
            tc::tc_fence_after();
            #pragma unroll
            for (int uu = 0; uu < 4; ++uu) {
                const int u = 4 * h + uu;
                uint32_t w[K + 1];
                #pragma unroll
                for (int j = 0; j <= K; ++j) w[j] = cw[uu * K + j];   // neighbour is the next unit's first word
                uint32_t r[16];
                #pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float lo = lut_at(lut_s, win_off_sh<K, kLutRepShift>(w, 31 - 2 * j) | gofs);
                    const float hi = lut_at(lut_s, win_off_sh<K, kLutRepShift>(w, 30 - 2 * j) | gofs);
                    const __nv_bfloat162 p2 = __floats2bfloat162_rn(__fmul_rn(lo, s), __fmul_rn(hi, s));
                    r[j] = valid ? *reinterpret_cast<const uint32_t*>(&p2) : 0u;
                }
                tc::tmem_st16(lane_base + (uint32_t)(stage * 128 + 112 - 16 * u), r);
            }
            tc::tmem_wait_st();
            tc::tc_fence_before();
            tc::mbar_arrive(&full[stage]);
            #pragma unroll
            for (int j = 0; j < 4 * K + 1; ++j) cw[j] = nw[j];
        }
    } else if (warp == kPfLoadWarp) {
        // ------------------------------------------------------------ activation loader
        // 16-byte cp.async copies into the swizzled layout (rows >= M are
        // zero-filled); the warp waits for its own copies, then fences them
        // into the async proxy before arriving.
        const uint32_t xs_base = tc::smem_addr(xs);
        for (int b = 0; b < nblocks; ++b) {
            const int stage = b & 1;
            if (b >= 2 && !tc::mbar_wait(&empty[stage], ((b >> 1) - 1) & 1, abort_flag, kWaitLimitNs)) break;
            __syncwarp();
            const uint32_t st = xs_base + stage * Lay::kXStage;
            #pragma unroll 8
            for (int qd = lane; qd < NPAD * 32; qd += 32) {
                const int n = qd >> 5, cc = qd & 31;
                const int kc = cc >> 3, c = cc & 7;
                const uint32_t dst = st + kc * Lay::kXChunk + n * 128 + ((c ^ (n & 7)) << 4);
                const bool in = n < M;
                const uint16_t* src = in ? x + (int64_t)n * cols + (int64_t)b * kBT + cc * 8 : x;
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
                             :: "r"(dst), "l"(src), "r"(in ? 16 : 0) : "memory");
            }
            asm volatile("cp.async.wait_all;" ::: "memory");
            tc::fence_proxy_async_smem();
            tc::mbar_arrive(&full[stage]);
        }
    } else if (warp == kPfMmaWarp) {
        // ------------------------------------------------------------ MMA issue
        if (lane == 0) {
            constexpr uint32_t idesc = tc::idesc_bf16_f32(128, NPAD);
            const uint32_t xs_base = tc::smem_addr(xs);
            for (int b = 0; b < nblocks; ++b) {
                const int stage = b & 1;
                if (!tc::mbar_wait(&full[stage], (b >> 1) & 1, abort_flag, kWaitLimitNs)) break;
                tc::tc_fence_after();
                #pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const uint32_t a = tmem + (uint32_t)(stage * 128 + 8 * j);
                    const uint64_t bd = tc::sdesc_sw128(
                        xs_base + stage * Lay::kXStage + (j >> 2) * Lay::kXChunk + (j & 3) * 32, 1024);
                    tc::mma_ts(tmem + kDCol, a, bd, idesc, (b | j) != 0 ? 1u : 0u);
                }
                tc::mma_commit(&empty[stage]);
            }
            tc::mma_commit(done);
        }
        __syncwarp();
    }

    // ---------------------------------------------------------------- epilogue
    if (warp < 4) {
        const bool ok = tc::mbar_wait(done, 0, abort_flag, kWaitLimitNs);
        __syncwarp();
        tc::tc_fence_after();
        const int row = row0 + 32 * warp + lane;
        const uint32_t taddr = tmem + ((uint32_t)(32 * warp) << 16) + kDCol;
        #pragma unroll
        for (int c = 0; c < NPAD; c += 16) {
            uint32_t d[16];
            tc::tmem_ld16(taddr + c, d);
            tc::tmem_wait_ld();
            if (ok && !*abort_flag && row < rows) {
                #pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int n = c + j;
                    if (n < M) out[(int64_t)n * rows + row] = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(d[j])));
                }
            }
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == kPfMmaWarp) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
    if (threadIdx.x == 0 && *abort_flag) atomicOr(status, kStatusWaitTimeout);
}

template <int K, int NPAD>
cudaError_t launch_kn(const Packed& p, const uint16_t* x, int M, uint16_t* out, int* status,
                      cudaStream_t stream) {
    const int smem = PfLayout<NPAD>::kAlloc;
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel<K, NPAD>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)((p.rows + kPfRows - 1) / kPfRows);
    prefill_kernel<K, NPAD><<<grid, kPfThreads, smem, stream>>>(x, M, p.codes, p.scales, p.lut,
                                                                (int)p.rows, (int)p.cols, out, status);
    return cudaGetLastError();
}

template <int K>
cudaError_t launch_k(const Packed& p, const uint16_t* x, int M, uint16_t* out, int* status,
                     cudaStream_t stream) {
    if (M <= 16) return launch_kn<K, 16>(p, x, M, out, status, stream);
    return launch_kn<K, 32>(p, x, M, out, status, stream);
}

}  // namespace

cudaError_t launch_prefill(const Packed& p, const uint16_t* x, int M, uint16_t* out,
                           int* status, int sm_count, cudaStream_t stream) {
    (void)sm_count;
    switch (p.k) {
        case 2: return launch_k<2>(p, x, M, out, status, stream);
        case 3: return launch_k<3>(p, x, M, out, status, stream);
        case 4: return launch_k<4>(p, x, M, out, status, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace tcq
