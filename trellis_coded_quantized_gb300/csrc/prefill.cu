// trellis_prefill: axis-1 packed matmul for M = 1..32 activation rows on the
// 5th-generation tensor cores, out[m][r] = bf16(sum_c x[m][c] w[r][c]).
//
// Arithmetic as the pages' prefill tile kernel (@mlx-bun/inference 1.0.0,
// kernels/trellis/tiled-prefill.ts): weights decoded to bf16 in the tile,
// contracted with the bf16 activations, fp32 accumulation, bf16 output.
//
// GB300 design (one CTA per tile of <= 128 weight rows, whole K; with 64..128
// rows per SM the rows are spread evenly over all SMs):
//   - the MMA is D[128 x N] += A[128 x 16] * B[16 x N] with A = decoded
//     weights (rows of the matrix are MMA rows, "swap AB") held in TENSOR
//     MEMORY, B = activations in shared memory (K-major, 128-byte swizzle),
//     D = fp32 accumulator in tensor memory; N = 16 or 32 (M padded);
//   - 1 code-loader thread: per 256-column block one TMA tensor copy of
//     the block of the CTA's rows (32 words per row with the 128-byte
//     swizzle, so that 8 consecutive rows read 8 different 16-byte chunks)
//     into one of 2 shared-memory tiles, completing on the tile's mbarrier;
//     the decoders release a tile as soon as they hold its words, so the
//     copies run up to 2 blocks ahead;
//   - 1 activation-loader thread copies the activation tile of each block
//     with four TMA tensor copies (64 columns x N rows each, the 128-byte
//     swizzle of the MMA's K-major B operand; rows M..N-1 lie outside the
//     tensor and arrive as zeros), whose bytes complete the stage's "full"
//     barrier together with the decoders' arrivals, so the activations need
//     no load/store-pipe copies and no wait in the loader;
//   - 16 decoder warps: warp w owns tensor-memory lane quarter w % 4 (32
//     matrix rows, one row per thread) and quarter w / 4 of each block (2
//     units of 32 columns).  A thread reads its row's words from the tile,
//     extracts windows, gathers the codebook from shared memory (8-way
//     replicated, one copy per lane group of 4, against bank conflicts),
//     scales, rounds pairs to bf16x2 and writes them with tcgen05.st straight
//     into the A stage: decoded weights never touch shared memory;
//   - 1 MMA warp: one thread waits for a stage, issues 16 tcgen05.mma
//     (K = 16 each) and commits to the stage's "empty" barrier;
//   - 3 stages (A: 3 x 128 tensor-memory columns beside the accumulator,
//     B: 3 x N x 512 bytes), mbarriers with bounded waits; after the last
//     block the accumulator is read back with tcgen05.ld by the lane-quarter
//     warps and stored as bf16.
// The K order of a block is the natural column order on both operands.
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace tcq {
namespace {

constexpr int kPfDecWarps = 16;            // 4 lane quarters x 4 block quarters
constexpr int kPfParts = kPfDecWarps / 4;
constexpr int kPfUnits = 8 / kPfParts;      // units of 32 columns per decoder warp and block
constexpr int kPfMmaWarp = kPfDecWarps;
constexpr int kPfLoadWarp = kPfDecWarps + 1;      // activation tiles
constexpr int kPfCodeWarp = kPfDecWarps + 2;      // code tiles
constexpr int kPfThreads = (kPfDecWarps + 3) * 32;
// Stages of the A operand (tensor memory) and the activations, and of the
// code tiles; the macros let a build try other depths.
// Three A stages let the decoders run two blocks ahead of the MMA (M=32:
// 2 us faster at k=2 and 3 on GB300); two code tiles keep the k=4, N=32
// layout within 227 KB of shared memory.
#ifndef TCQ_PF_ASTAGES
#define TCQ_PF_ASTAGES 3
#endif
#ifndef TCQ_PF_CSTAGES
#define TCQ_PF_CSTAGES 2
#endif
constexpr int kPfAStages = TCQ_PF_ASTAGES;
constexpr int kPfCodeStages = TCQ_PF_CSTAGES;
static_assert(kPfAStages == 2 || kPfAStages == 3, "2 or 3 A stages fit beside the accumulator");
constexpr int kPfRows = 128;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kDCol = 256;            // accumulator columns [256, 256 + N)
// tensor-memory column of A stage st: [0, 128), [128, 256), [384, 512)
__host__ __device__ constexpr uint32_t a_col(int st) { return st < 2 ? (uint32_t)st * 128u : 384u; }
// Wall-clock limit of every mbarrier wait (a test build of the library sets
// a shorter one).
#ifndef TCQ_WAIT_LIMIT_NS
#define TCQ_WAIT_LIMIT_NS 1000000000ull
#endif
constexpr uint64_t kWaitLimitNs = TCQ_WAIT_LIMIT_NS;
// After an abort: how long the activation loader waits for its last copies.
constexpr uint64_t kDrainLimitNs = 2000000ull;

#ifdef TCQ_TEST_HOOKS
// test build only (see trellis_test_set_withhold at the end of this file)
__device__ int g_test_withhold;
__device__ __forceinline__ bool test_withhold_arrival() {
    return *reinterpret_cast<volatile int*>(&g_test_withhold) != 0;
}
#endif

template <int K, int NPAD>
struct PfLayout {
    static constexpr int kWpb = kBT * K / 32;              // words of one block
    // bytes per row of a code tile: one 128-byte swizzle row (the TMA box
    // is 32 words wide; past a block's kWpb words it holds the next block's
    // first words, or zeros past the end of the matrix row)
    static constexpr int kPitch = 128;
    static constexpr int kXStage = NPAD * kBT * 2;         // bytes of one activation stage
    static constexpr int kXChunk = NPAD * 128;             // one 64-column K chunk
    static constexpr int kCodeOff = kPfAStages * kXStage;
    static constexpr int kCodeStage = kPfRows * kPitch;
    static constexpr int kBarOff = kCodeOff + kPfCodeStages * kCodeStage;
    static constexpr int kBytes = kBarOff + 128;
    // the codebook copies come first, at the start of the dynamic shared
    // memory (a constant address the gathers fold into their offset); the
    // region above starts at the next 1024-byte boundary
    static constexpr int kAlloc = (int)kLutRepBytes + kBytes + 1024;
};

// Words of the kPfUnits units of one block quarter of row rl from the code
// tile (128-byte rows with the 128-byte swizzle: 16-byte chunk c of row rl
// sits at chunk c ^ (rl & 7)), plus the neighbour word (first word of the
// next unit, unit 0 for the last quarter).  Eight consecutive rows read
// eight different chunks, so a warp's vector loads take the fewest
// wavefronts.
template <int K>
__device__ __forceinline__ uint32_t sw_word_off(int j, int rl) {
    return (uint32_t)((((j >> 2) ^ (rl & 7)) << 4) | ((j & 3) << 2));
}
template <int K>
__device__ __forceinline__ void read_quarter(uint32_t* w, const uint8_t* row, int rl, int part) {
    const int j0 = part * kPfUnits * K;
    if constexpr (K == 3) {
        #pragma unroll
        for (int j = 0; j < kPfUnits * K; j += 2) {
            const uint2 v = *reinterpret_cast<const uint2*>(row + sw_word_off<K>(j0 + j, rl));
            w[j] = v.x; w[j + 1] = v.y;
        }
    } else {
        #pragma unroll
        for (int j = 0; j < kPfUnits * K; j += 4) {
            const uint4 v = *reinterpret_cast<const uint4*>(row + sw_word_off<K>(j0 + j, rl));
            w[j] = v.x; w[j + 1] = v.y; w[j + 2] = v.z; w[j + 3] = v.w;
        }
    }
    const int nb = (part + 1 == kPfParts) ? 0 : (part + 1) * kPfUnits * K;
    w[kPfUnits * K] = *reinterpret_cast<const uint32_t*>(row + sw_word_off<K>(nb, rl));
}

// GU: the gate and up projections of a SwiGLU layer in one launch.  The CTA
// walks the column blocks of its gate rows, then those of the same up rows
// (2 x nblocks blocks through the same pipeline, the codes and scales of the
// second pass from codes_u / scales_u), accumulating into two tensor-memory
// accumulators, and its epilogue writes h = bf16(silu(bf16(gate)) *
// bf16(up)) -- the bits trellis_prefill twice and trellis_silu_mul give.
template <int K, int NPAD, bool GU>
__global__ void __launch_bounds__(kPfThreads, 1)
prefill_kernel(const uint16_t* __restrict__ x, int M, const uint32_t* __restrict__ codes,
               const uint16_t* __restrict__ scales, const uint32_t* __restrict__ codes_u,
               const uint16_t* __restrict__ scales_u, const float* __restrict__ lut,
               int rows, int cols, int interleave, int tile_rows, uint16_t* __restrict__ out,
               int* __restrict__ status, const __grid_constant__ CUtensorMap xmap,
               const __grid_constant__ CUtensorMap cmap, const __grid_constant__ CUtensorMap cmap_u) {
    using Lay = PfLayout<K, NPAD>;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    pdl_release();
    // 1024-byte aligned base, derived by pointer arithmetic on the shared
    // array (an integer round trip would lose the shared address space and
    // turn every table gather into a generic load)
    float* lut_s = reinterpret_cast<float*>(smem_raw);
    uint8_t* base = smem_raw + kLutRepBytes + ((1024u - (tc::smem_addr(smem_raw) & 1023u)) & 1023u);
    uint8_t* xs = base;
    uint8_t* cs = base + Lay::kCodeOff;
    uint64_t* full = reinterpret_cast<uint64_t*>(base + Lay::kBarOff);   // decoders + activations
    uint64_t* empty = full + kPfAStages;                                  // MMA done with a stage
    uint64_t* cfull = empty + kPfAStages;                                 // code tile landed
    uint64_t* cempty = cfull + kPfCodeStages;                             // code tile read
    uint64_t* done = cempty + kPfCodeStages;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // the codebook (a weight input, never written by this library) is staged
    // while the previous kernel of the stream may still run; nothing else is
    // read, written or allocated (tensor memory) before that kernel has
    // completed
    stage_lut_rep8(lut_s, lut);
    pdl_wait();
    if (threadIdx.x == 0) {
        for (int st = 0; st < kPfAStages; ++st) {
            tc::mbar_init(&full[st], kPfDecWarps * 32 + 1);
            tc::mbar_init(&empty[st], 1);
        }
        for (int st = 0; st < kPfCodeStages; ++st) {
            tc::mbar_init(&cfull[st], 1);
            tc::mbar_init(&cempty[st], kPfDecWarps * 32);
        }
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
    const int nbt = GU ? 2 * nblocks : nblocks;      // blocks through the pipeline
    constexpr int wpb = Lay::kWpb;
    // this CTA owns tile_rows (<= 128) rows: the MMA always spans 128 lanes.
    // Its nvalid rows are dealt evenly to the 4 lane quarters (rpq each, the
    // last quarter fewer), so every decoder warp has about the same work;
    // local row q*rpq + i sits in lane 32q + i, and lanes past rpq decode
    // nothing and are not stored.
    const int row0 = blockIdx.x * tile_rows;
    const int nvalid = min(tile_rows, rows - row0);
    const int rpq = (nvalid + 3) >> 2;

    if (warp < kPfDecWarps) {
        // ------------------------------------------------------------ decoders
        const int q = warp & 3, part = warp >> 2;
        const int rl = q * rpq + lane;
        const bool valid = lane < rpq && rl < nvalid;
        const float s_g = valid ? bf16_bits_to_float(__ldg(scales + row0 + rl)) : 0.f;
        const float s_u = GU && valid ? bf16_bits_to_float(__ldg(scales_u + row0 + rl)) : 0.f;
        const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
        const uint32_t gofs = lut_rep_lane_offset();     // this lane's codebook copy
        for (int b = 0; b < nbt; ++b) {
            const float s = GU && b >= nblocks ? s_u : s_g;
            const int stage = b % kPfAStages, use = b / kPfAStages;
            const int cst = b % kPfCodeStages, cuse = b / kPfCodeStages;
            if (!tc::mbar_wait(&cfull[cst], cuse & 1, abort_flag, kWaitLimitNs)) break;
            uint32_t cw[kPfUnits * K + 1];
            read_quarter<K>(cw, cs + cst * Lay::kCodeStage + rl * Lay::kPitch, rl, part);
            tc::mbar_arrive(&cempty[cst]);                 // the code tile may be refilled
            if (b >= kPfAStages && !tc::mbar_wait(&empty[stage], (use - 1) & 1, abort_flag, kWaitLimitNs)) break;
            __syncwarp();
            tc::tc_fence_after();
            #pragma unroll
            for (int uu = 0; uu < kPfUnits; ++uu) {
                const int u = kPfUnits * part + uu;
                uint32_t w[K + 1];
                #pragma unroll
                for (int j = 0; j <= K; ++j) w[j] = cw[uu * K + j];   // neighbour is the next unit's first word
                uint32_t r[16];
                if (valid) {                                // lanes past the CTA's rows issue no gathers
                    // the unit's 32 codebook values first, then the scaling
                    float v[32];
                    #pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = lut_at(lut_s, win_off_sh<K, kLutRepShift>(w, 31 - j) | gofs);
                    #pragma unroll
                    for (int j = 0; j < 16; ++j)
                        r[j] = pack_bf16x2(__fmul_rn(v[2 * j], s), __fmul_rn(v[2 * j + 1], s));
                } else {
                    #pragma unroll
                    for (int j = 0; j < 16; ++j) r[j] = 0u;
                }
                __syncwarp();
                tc::tmem_st16(lane_base + a_col(stage) + (uint32_t)(112 - 16 * u), r);
            }
            tc::tmem_wait_st();
            tc::tc_fence_before();
            tc::mbar_arrive(&full[stage]);
        }
    } else if (warp == kPfCodeWarp) {
        // ------------------------------------------------------------ code loader
        // One thread: per block, one TMA tensor copy of the CTA's rows
        // (32 words each, the 128-byte swizzle) into tile cst, completing on
        // cfull[cst] with its bytes.  Up to kPfCodeStages blocks ahead of
        // the decoders, which release a tile (cempty) as soon as they hold
        // its words in registers.
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&cmap)) : "memory");
            if (GU) asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&cmap_u)) : "memory");
            const uint32_t tile_bytes = (uint32_t)tile_rows * Lay::kPitch;
            int issued = 0;
            for (int b = 0; b < nbt; ++b) {
                const int cst = b % kPfCodeStages, cuse = b / kPfCodeStages;
                if (b >= kPfCodeStages &&
                    !tc::mbar_wait(&cempty[cst], (cuse - 1) & 1, abort_flag, kWaitLimitNs)) break;
#ifdef TCQ_TEST_HOOKS
                // test build only: with the hook set, CTA 0 withholds its
                // first code tile, so the decoders' bounded wait on it runs
                // out and the kernel takes its abort path
                if (b == 0 && blockIdx.x == 0 && test_withhold_arrival()) continue;
#endif
                const bool upm = GU && b >= nblocks;
                const int bb = upm ? b - nblocks : b;
                const uint64_t map = reinterpret_cast<uint64_t>(upm ? &cmap_u : &cmap);
                const uint32_t dst = tc::smem_addr(cs + cst * Lay::kCodeStage);
                const uint32_t bar = tc::smem_addr(&cfull[cst]);
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(bar), "r"(tile_bytes)
                             : "memory");
                if (interleave == 2)
                    asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                                 " [%0], [%1, {%2, %3, %4}], [%5];"
                                 :: "r"(dst), "l"(map), "r"((bb & 1) * wpb), "r"(row0), "r"(bb >> 1), "r"(bar)
                                 : "memory");
                else
                    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                                 " [%0], [%1, {%2, %3}], [%4];"
                                 :: "r"(dst), "l"(map), "r"(bb * wpb), "r"(row0), "r"(bar) : "memory");
                issued = b + 1;
            }
            // no copy may still be in flight when the CTA ends: wait for the
            // last issued tiles' bytes, with a limit of its own
            volatile int keep_waiting = 0;
            for (int b = issued > kPfCodeStages ? issued - kPfCodeStages : 0; b < issued; ++b)
                tc::mbar_wait(&cfull[b % kPfCodeStages], (b / kPfCodeStages) & 1, &keep_waiting, kDrainLimitNs);
        }
        __syncwarp();
    } else if (warp == kPfLoadWarp) {
        // ------------------------------------------------------------ activation loader
        // One thread: per block, four TMA tensor copies of 64 columns x NPAD
        // rows into the stage; their bytes count towards full[stage].
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&xmap)) : "memory");
            const uint32_t xs_base = tc::smem_addr(xs);
            int issued = 0;
            for (int b = 0; b < nbt; ++b) {
                const int stage = b % kPfAStages, use = b / kPfAStages;
                if (b >= kPfAStages && !tc::mbar_wait(&empty[stage], (use - 1) & 1, abort_flag, kWaitLimitNs)) break;
                const int bb = GU && b >= nblocks ? b - nblocks : b;   // column block
                const uint32_t bar = tc::smem_addr(&full[stage]);
                const uint32_t st = xs_base + stage * Lay::kXStage;
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                             :: "r"(bar), "r"(Lay::kXStage) : "memory");
                #pragma unroll
                for (int kc = 0; kc < 4; ++kc)
                    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                                 " [%0], [%1, {%2, %3}], [%4];"
                                 :: "r"(st + kc * Lay::kXChunk), "l"(reinterpret_cast<uint64_t>(&xmap)),
                                    "r"(bb * kBT + kc * 64), "r"(0), "r"(bar) : "memory");
                issued = b + 1;
            }
            // no copy may still be in flight when the CTA ends: after an
            // abort, wait for the last issued stages' barriers with a limit
            // of its own (their phases may also lack the decoders' arrivals,
            // so the limit, far longer than a copy takes, can run out)
            if (*abort_flag) {
                volatile int keep_waiting = 0;
                for (int b = issued > kPfAStages ? issued - kPfAStages : 0; b < issued; ++b)
                    tc::mbar_wait(&full[b % kPfAStages], (b / kPfAStages) & 1, &keep_waiting, kDrainLimitNs);
            }
        }
        __syncwarp();
    } else if (warp == kPfMmaWarp) {
        // ------------------------------------------------------------ MMA issue
        if (lane == 0) {
            constexpr uint32_t idesc = tc::idesc_bf16_f32(128, NPAD);
            const uint32_t xs_base = tc::smem_addr(xs);
            for (int b = 0; b < nbt; ++b) {
                const int stage = b % kPfAStages;
                if (!tc::mbar_wait(&full[stage], (b / kPfAStages) & 1, abort_flag, kWaitLimitNs)) break;
                tc::tc_fence_after();
                const bool upm = GU && b >= nblocks;
                const int bb = upm ? b - nblocks : b;
                const uint32_t dcol = tmem + kDCol + (upm ? (uint32_t)NPAD : 0u);
                #pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const uint32_t a = tmem + a_col(stage) + (uint32_t)(8 * j);
                    const uint64_t bd = tc::sdesc_sw128(
                        xs_base + stage * Lay::kXStage + (j >> 2) * Lay::kXChunk + (j & 3) * 32, 1024);
                    tc::mma_ts(dcol, a, bd, idesc, (bb | j) != 0 ? 1u : 0u);
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
        const int rl = warp * rpq + lane;
        const int row = row0 + rl;
        const uint32_t taddr = tmem + ((uint32_t)(32 * warp) << 16) + kDCol;
        #pragma unroll
        for (int c = 0; c < NPAD; c += 16) {
            uint32_t d[16], du[16];
            tc::tmem_ld16(taddr + c, d);
            if constexpr (GU) tc::tmem_ld16(taddr + NPAD + c, du);
            tc::tmem_wait_ld();
            if (ok && !*abort_flag && lane < rpq && rl < nvalid) {
                #pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int n = c + j;
                    if (n >= M) continue;
                    uint16_t v = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(d[j])));
                    if constexpr (GU) {
                        const uint16_t u = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(du[j])));
                        v = __bfloat16_as_ushort(__float2bfloat16_rn(
                            silu_mul_f32(bf16_bits_to_float(v), bf16_bits_to_float(u))));
                    }
                    out[(int64_t)n * rows + row] = v;
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

// cuTensorMapEncodeTiled, found once through the runtime (no link-time
// dependence on the driver library).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn pf_encode_tiled() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, []() {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
        cudaGetLastError();
    });
    return fn;
}

// The activations x [M][cols] (bf16, 16-byte aligned, cols a multiple of
// 256) with a box of 64 columns by npad rows and the 128-byte swizzle: one
// K chunk of the MMA's B operand per copy; rows past M are filled with zeros.
cudaError_t pf_x_tensor_map(const uint16_t* x, int M, int64_t cols, int npad, CUtensorMap* map) {
    EncodeTiledFn enc = pf_encode_tiled();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)M};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)npad}, estr[2] = {1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<uint16_t*>(x), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// The codes as uint32 words with a box of 32 words (one 128-byte swizzle
// row) by tile_rows rows: interleave 0 is [rows][nb * wpb], interleave 2 is
// [nb / 2][rows][2 * wpb].  Past a block's wpb words the box reads the next
// block's first words, or zeros past the end of the tensor's row.
cudaError_t pf_code_tensor_map(const uint32_t* codes, int64_t rows, int64_t cols, int k, int interleave,
                               int tile_rows, CUtensorMap* map) {
    EncodeTiledFn enc = pf_encode_tiled();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t wpb = (cuuint64_t)(kBT * k / 32), nb = (cuuint64_t)(cols / kBT);
    cuuint64_t dims[3], strides[2];
    const cuuint32_t box[3] = {32, (cuuint32_t)tile_rows, 1}, estr[3] = {1, 1, 1};
    cuuint32_t rank;
    if (interleave == 2) {
        rank = 3;
        dims[0] = 2 * wpb;
        dims[1] = (cuuint64_t)rows;
        dims[2] = nb / 2;
        strides[0] = dims[0] * 4;
        strides[1] = strides[0] * dims[1];
    } else {
        rank = 2;
        dims[0] = nb * wpb;
        dims[1] = (cuuint64_t)rows;
        strides[0] = dims[0] * 4;
    }
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, rank, const_cast<uint32_t*>(codes), dims, strides,
                           box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int K, int NPAD, bool GU>
cudaError_t launch_kn(const Packed& p, const uint32_t* codes_u, const uint16_t* scales_u, const uint16_t* x, int M,
                      uint16_t* out, int* status, int sm_count, cudaStream_t stream) {
    const int smem = PfLayout<K, NPAD>::kAlloc;
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel<K, NPAD, GU>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // Between 64 and 128 rows per SM: spread the rows over all SMs (the decode
    // is the work, so CTAs with fewer rows finish sooner); else 128-row tiles.
    int tile_rows = kPfRows;
    if (sm_count > 0 && p.rows > (int64_t)64 * sm_count && p.rows <= (int64_t)kPfRows * sm_count)
        tile_rows = (int)((p.rows + sm_count - 1) / sm_count);
    const unsigned grid = (unsigned)((p.rows + tile_rows - 1) / tile_rows);
    alignas(64) CUtensorMap xmap, cmap, cmap_u;
    e = pf_x_tensor_map(x, M, p.cols, NPAD, &xmap);
    if (e != cudaSuccess) return e;
    e = pf_code_tensor_map(p.codes, p.rows, p.cols, K, p.interleave, tile_rows, &cmap);
    if (e != cudaSuccess) return e;
    cmap_u = cmap;
    if (GU) {
        e = pf_code_tensor_map(codes_u, p.rows, p.cols, K, p.interleave, tile_rows, &cmap_u);
        if (e != cudaSuccess) return e;
    }
    e = launch_pdl(prefill_kernel<K, NPAD, GU>, dim3(grid), dim3(kPfThreads), (size_t)smem, stream, x, M, p.codes,
                   p.scales, codes_u, scales_u, p.lut, (int)p.rows, (int)p.cols, p.interleave, tile_rows, out, status,
                   xmap, cmap, cmap_u);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int K, bool GU>
cudaError_t launch_k(const Packed& p, const uint32_t* codes_u, const uint16_t* scales_u, const uint16_t* x, int M,
                     uint16_t* out, int* status, int sm_count, cudaStream_t stream) {
    if (M <= 16) return launch_kn<K, 16, GU>(p, codes_u, scales_u, x, M, out, status, sm_count, stream);
    return launch_kn<K, 32, GU>(p, codes_u, scales_u, x, M, out, status, sm_count, stream);
}

template <bool GU>
cudaError_t launch_any(const Packed& p, const uint32_t* codes_u, const uint16_t* scales_u, const uint16_t* x, int M,
                       uint16_t* out, int* status, int sm_count, cudaStream_t stream) {
    switch (p.k) {
        case 2: return launch_k<2, GU>(p, codes_u, scales_u, x, M, out, status, sm_count, stream);
        case 3: return launch_k<3, GU>(p, codes_u, scales_u, x, M, out, status, sm_count, stream);
        case 4: return launch_k<4, GU>(p, codes_u, scales_u, x, M, out, status, sm_count, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_prefill(const Packed& p, const uint16_t* x, int M, uint16_t* out,
                           int* status, int sm_count, cudaStream_t stream) {
    return launch_any<false>(p, nullptr, nullptr, x, M, out, status, sm_count, stream);
}

cudaError_t launch_gate_up_prefill(const Packed& gate, const uint32_t* up_codes, const uint16_t* up_scales,
                                   const uint16_t* x, int M, uint16_t* h, int* status, int sm_count,
                                   cudaStream_t stream) {
    return launch_any<true>(gate, up_codes, up_scales, x, M, h, status, sm_count, stream);
}

}  // namespace tcq

#ifdef TCQ_TEST_HOOKS
// Test build only, not part of the C ABI: nonzero makes the prefill's code
// loader withhold one mbarrier arrival (lane 0 of CTA 0, first code tile) so
// that the decoders' bounded wait runs out.  Returns the cudaError_t of the
// copy to the device flag.
extern "C" int trellis_test_set_withhold(int on) {
    return (int)cudaMemcpyToSymbol(tcq::g_test_withhold, &on, sizeof on);
}
#endif
