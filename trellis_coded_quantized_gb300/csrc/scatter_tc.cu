// trellis_scatter on the 5th-generation tensor cores (rounded contract,
// 3..32 activation rows): out[m][c] = bf16(sum_r x[m][r] w[r][c]) through
// fp32 split partials P[m][s][c] (@mlx-bun/inference 1.0.0,
// kernels/trellis/scatter.ts: split ranges, the [M, SPLITS, C] float
// partials and their sum over the split axis; splitk-prefill.ts computes the
// same partials with 8x8 simdgroup MMAs on weights decoded into threadgroup
// memory).
//
// The MMA is D[c][m] += W^T[c][r] X^T[r][m]: output columns are the MMA
// rows (tensor-memory lanes), the input rows of the split are K, the
// activation rows (padded to N = 16 or 32) are N.
//   - A (decoded weights) is written straight into TENSOR MEMORY with the
//     16x256b store shape, so the MMA reads only the small B operand from
//     shared memory, where the codebook gathers already take the bandwidth.
//     That shape fills 16 lanes of a warp's 32-lane quarter; the other 16
//     lanes are left out, so an M = 128 MMA carries 64 output columns and a
//     256-column block is four "regions" of 64 columns.  In a region a thread
//     (g = lane / 4, c = lane % 4) of quarter q fills lanes 32q+g and
//     32q+g+8 with K rows 4c..4c+3; it owns the 8 consecutive columns
//     64q + 8g .. +7 of the block, region r holding columns 64q + 8g + 2r
//     (lane 32q+g) and 64q + 8g + 2r + 1 (lane 32q+g+8).  The rows of D past
//     lane 16 of a quarter are never read;
//   - B (activations x[m][r0 .. r0+63]) is K-major with the 128-byte swizzle;
//   - a loader warp fills a ring of 8 slots (7 at N = 32), each the bundle of one stage:
//     its code words (64 rows of one block, 128 bytes each), its 64 row
//     scales and B, all by TMA tensor copies on one mbarrier, up to 8 stages
//     ahead.  The copies bypass the load/store pipe that the codebook
//     gathers keep busy (per-thread cp.async copies there took microseconds
//     to land).  Rows whose first index is not a multiple of 8 fall back to
//     plain copies for the scales and B;
//   - D (fp32) lives in tensor memory, two buffers of 4 regions x N columns,
//     so the epilogue of one item overlaps the MMAs of the next.
// A stage is up to 64 rows (4 K steps) of one item (one split, one block of
// 256 columns).  Persistent CTAs, one per SM, take equal runs of K steps
// over all items (splitk_schedule.cuh); a CTA that starts inside an item
// leaves its share in a fix-up slot that the split reduction adds in CTA
// order.
//
// Warps: 16 decoders (warp w: lane quarter w % 4, K step w / 4 of the stage;
// a thread decodes 8 windows of each of its 4 rows from 3 words of the code
// tile), 4 epilogue warps (lane quarters 0..3), 4 MMA warps (region r each),
// 1 loader.  One thread issues an MMA only every 60-100 cycles whatever its
// shape, so the 16 MMAs of a stage go out from four threads at once.
// The barriers are few on purpose: each wait costs a few hundred cycles even
// when the phase is already complete.  Every mbarrier wait is bounded (1 s); a wait that
// gives up sets the CTA's abort flag and the device status word, and the
// kernel returns without further output.
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "splitk_schedule.cuh"
#include "tc.cuh"

namespace tcq {
namespace {

constexpr int kStDecWarps = 16;                 // warps 16..19: epilogue, lane quarters 0..3
constexpr int kStMmaWarp = 20;                  // warps 20..23: MMA issue, one region each
constexpr int kStActWarp = 24;
constexpr int kStThreads = 25 * 32;
constexpr int kStRows = 64;                     // rows (K) of a stage: 4 MMA steps of 16
constexpr int kStSteps = kStRows / 16;
constexpr int kStStages = 3;                    // stages of decoded weights (A, tensor memory)
constexpr int kStPitch = 128;                   // bytes per row of a code tile
constexpr int kStCBytes = kStRows * kStPitch;   // one code tile (8 KB)
// Per code slot, written by the loader with the tile: the stage's 64 row
// scales (bf16) and a descriptor: take, valid rows, whether another stage
// follows.
constexpr int kStSclBytes = kStRows * 2;
constexpr uint32_t kStTmemCols = 512;
// A stages at [128, 512): 4 regions x 32 columns each; D buffers at [0, 128):
// two of 4 regions x 16 columns, or one of 4 x 32
constexpr uint32_t kStACol = kStTmemCols - kStStages * 128;
__host__ __device__ constexpr int st_dbufs(int npad) { return 4 * npad * 2 <= (int)kStACol ? 2 : 1; }
constexpr uint64_t kStWaitNs = 1000000000ull;

template <int NPAD>
struct StLayout {
    // slots of the TMA ring (code tile, scales and activations of a stage):
    // the loader refills a slot once the MMAs of its stage are done, and a
    // stage's copies take microseconds from HBM, so the ring runs as deep as
    // shared memory allows (8 slots against 4: 3% faster at M = 4..32)
    static constexpr int kCStages = NPAD <= 16 ? 8 : 7;
    static constexpr int kB = NPAD * 128;       // activations of one stage: NPAD rows x 64 K
    static constexpr int kCOff = 0;             // code tiles: 1024-byte aligned for the swizzled TMA
    static constexpr int kBOff = kCOff + kCStages * kStCBytes;
    // per code slot: the stage's 64 row scales (TMA destination: 128-byte
    // aligned, here 1024) and its 16-byte descriptor
    static constexpr int kSclOff = kBOff + kCStages * kB;
    static constexpr int kInfoOff = kSclOff + kCStages * kStSclBytes;
    static constexpr int kLutOff = (kInfoOff + kCStages * 16 + 1023) / 1024 * 1024;
    static constexpr int kBarOff = kLutOff + (int)kLutRepBytes;
    // the mbarriers (at most 2 x 3 + 2 x 8 + 5), the tensor-memory address
    // and the abort flag
    static constexpr int kBarBytes = 320;
    static constexpr int kBytes = kBarOff + kBarBytes;
    static constexpr int kAlloc = kBytes + 1024;    // slack for 1024-byte alignment
};

// One stage of the CTA's run: up to kStSteps steps of one item.
struct Stage {
    int s, b;          // split, block of 256 columns
    int k, take, n;    // first step within the item, steps taken, steps of the item
    int64_t r_begin;   // first input row
    int valid;         // rows of the stage inside the split (<= 16 * take)
    bool first;        // first stage of this item in the CTA
    bool last;         // last stage of this item in the CTA
};

// Walks the CTA's run stage by stage.  Only the start is located by
// division; after that the position advances by additions, so the per-stage
// bookkeeping costs every thread a few instructions.
struct Cursor {
    int64_t x, xe;     // next step, end of the run
    int s, b, k, n;    // item and step within it of x, steps of that item
    bool fresh;        // no stage taken yet
};

__device__ __forceinline__ void cursor_init(const SplitSchedule& sc, Cursor& c, int64_t xb, int64_t xe) {
    c.x = xb;
    c.xe = xe;
    c.s = c.b = c.k = c.n = 0;
    if (xb < xe) sc.locate(xb, c.s, c.b, c.k, c.n);
    c.fresh = true;
}

__device__ __forceinline__ bool next_stage(const SplitSchedule& sc, Cursor& c, Stage& st) {
    if (c.x >= c.xe) return false;
    st.s = c.s;
    st.b = c.b;
    st.k = c.k;
    st.n = c.n;
    int take = c.n - c.k;
    if (take > kStSteps) take = kStSteps;
    if ((int64_t)take > c.xe - c.x) take = (int)(c.xe - c.x);
    st.take = take;
    st.first = c.k == 0 || c.fresh;
    st.last = c.k + take == c.n || c.x + take == c.xe;
    st.r_begin = sc.row0(st.s) + 16 * (int64_t)st.k;
    const int64_t v = sc.row1(st.s) - st.r_begin;
    st.valid = (int)(v < 16 * take ? v : 16 * take);
    c.fresh = false;
    c.x += take;
    c.k += take;
    if (c.k == c.n) {                  // next item: next block, then next split
        c.k = 0;
        if (++c.b == sc.NB) {
            c.b = 0;
            ++c.s;
            c.n = sc.steps(c.s);       // past the last non-empty split x has reached xe
        }
    }
    return true;
}

// Byte offset of word w of row r in a code tile written by the TMA with the
// 128-byte swizzle (tile 1024-byte aligned): the 16-byte chunk index of the
// row is XOR-ed with r mod 8.
__device__ __forceinline__ uint32_t ctile_off(int r, int w) {
    return (uint32_t)r * kStPitch + ((((uint32_t)w >> 2) ^ ((uint32_t)r & 7u)) << 4) + ((uint32_t)w & 3u) * 4u;
}

// tcgen05.st of 4 registers per thread in the 16x256b shape: thread (g, c)
// writes lanes g and g+8 of the 16 lanes at taddr, columns 2c and 2c+1.
__device__ __forceinline__ void tmem_st_16x256b(uint32_t taddr, uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3) {
    asm volatile("tcgen05.st.sync.aligned.16x256b.x1.b32 [%0], {%1, %2, %3, %4};"
                 :: "r"(taddr), "r"(r0), "r"(r1), "r"(r2), "r"(r3) : "memory");
}

template <int K, int NPAD>
__global__ void __launch_bounds__(kStThreads, 1)
scatter_tc_kernel(const uint16_t* __restrict__ x, int M, const uint32_t* __restrict__ codes,
                  const uint16_t* __restrict__ scales, const float* __restrict__ lut,
                  int C, int interleave, SplitSchedule sc, float* __restrict__ partial,
                  float* __restrict__ fix, int* __restrict__ status, const __grid_constant__ CUtensorMap tmap,
                  const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap smap, int tma_x) {
    using Lay = StLayout<NPAD>;
    constexpr int kDBuf = st_dbufs(NPAD);
    constexpr int kCS = Lay::kCStages;
    static_assert(kDBuf * 4 * NPAD <= (int)kStACol, "D buffers overlap the A stages");
    extern __shared__ uint8_t smem_raw[];
    pdl_release();
    uint8_t* base = smem_raw + ((1024u - (tc::smem_addr(smem_raw) & 1023u)) & 1023u);
    float* lut_s = reinterpret_cast<float*>(base + Lay::kLutOff);
    // Per stage of A (tensor memory): afull -- all decoders wrote it;
    // aempty -- the MMAs that read it are done.  Per slot (codes, scales and
    // activations of one stage, one TMA bundle): cfull -- landed; sempty --
    // the stage's MMAs are done, which is after every decoder read the slot.
    uint64_t* afull = reinterpret_cast<uint64_t*>(base + Lay::kBarOff);
    uint64_t* aempty = afull + kStStages;
    uint64_t* cfull = aempty + kStStages;
    uint64_t* sempty = cfull + kCS;
    uint64_t* dfull = sempty + kCS;                                 // an item's D complete
    uint64_t* dempty = dfull + 2;                                          // epilogue done with D
    uint64_t* done = dempty + 2;                                           // every MMA complete
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    static_assert((2 * kStStages + 2 * kCS + 5) * 8 + 8 <= Lay::kBarBytes, "barrier area too small");
    // every TMA destination: tiles 1024-byte aligned (128-byte swizzle), the
    // scales 128-byte aligned
    static_assert(Lay::kCOff % 1024 == 0 && kStCBytes % 1024 == 0 && Lay::kBOff % 1024 == 0 && Lay::kB % 1024 == 0,
                  "swizzled TMA destinations must be 1024-byte aligned");
    static_assert(Lay::kSclOff % 128 == 0 && kStSclBytes % 128 == 0, "TMA destinations must be 128-byte aligned");

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // the codebook (a weight input, never written by this library) is staged
    // while the previous kernel of the stream may still run; nothing else is
    // read, written or allocated (tensor memory) before that kernel has
    // completed
    stage_lut_rep8(lut_s, lut);
    pdl_wait();
    if (threadIdx.x == 0) {
        for (int i = 0; i < kStStages; ++i) {
            tc::mbar_init(&afull[i], kStDecWarps * 32);
            tc::mbar_init(&aempty[i], 4);
        }
        for (int i = 0; i < kCS; ++i) {
            tc::mbar_init(&cfull[i], 1);
            tc::mbar_init(&sempty[i], 4);
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&dfull[i], 4);
            tc::mbar_init(&dempty[i], 4);
        }
        tc::mbar_init(done, 4);
        *abort_flag = 0;
        tc::mbar_init_fence();
    }
    if (warp == kStMmaWarp) {
        tc::tmem_alloc(tmem_slot, kStTmemCols);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int64_t xb = sc.start(blockIdx.x), xe = sc.start(blockIdx.x + 1);
    const uint32_t s_base = tc::smem_addr(base);
    const uint32_t b_base = s_base + Lay::kBOff;
    const uint32_t c_base = s_base + Lay::kCOff;
    const int64_t R = sc.R;
    constexpr int wpb = kBT * K / 32;

    if (warp < kStDecWarps) {
        // ------------------------------------------------------------ decoders
        const int q = warp & 3, ks = warp >> 2;
        const int g = lane >> 2, c = lane & 3;
        // shared address of this lane's codebook copy (entry e at +32 e)
        const uint32_t lut_sa = tc::smem_addr(lut_s) + lut_rep_lane_offset();
        // columns t0 .. t0+7 of the block; the window of column t0+e starts at
        // bit (255 - t0 - e) k = S + (7 - e) k, S = (248 - t0) k
        const int t0 = 64 * q + 8 * g;
        const int S = (248 - t0) * K;
        const int wi = S >> 5;
        const uint32_t off = (uint32_t)(S & 31);
        const int w1i = wi + 1 < wpb ? wi + 1 : wi + 1 - wpb;
        const int w2i = wi + 2 < wpb ? wi + 2 : wi + 2 - wpb;
        // this thread's rows of the stage: 16 ks + 4c + i, i = 0..3.  Held
        // words slot i carries row 4c + (i ^ sw): threads c = 2, 3 load their
        // rows in the order 2, 3, 0, 1, so that in every word load the four c
        // of a warp read tile rows whose 128-byte swizzle phases (row mod 8)
        // differ by 2, 4 or 6 and no two of them meet in a bank (rows 8
        // apart, the same phase, would).  The decode puts the rows back in
        // order.
        const int row0 = 16 * ks + 4 * c;
        const int sw = c & 2;
        const int widx[3] = {wi, w1i, w2i};
        // Byte offset of word widx[t] in tile row row0 + j, j = 0..3, is
        // (wofs[t] ^ (j << 4)) + (j << 7): row0 is a multiple of 4, so the
        // row's swizzle phase is (row0 & 7) | j and j only flips chunk bits.
        uint32_t wofs[3];
        #pragma unroll
        for (int t = 0; t < 3; ++t) wofs[t] = ctile_off(row0, widx[t]);
        const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
        const uint32_t info_base = s_base + Lay::kInfoOff;
        const uint32_t scl_base = s_base + Lay::kSclOff;
        // What a decoder thread takes from code slot cs once it has landed:
        // the stage's take / valid / more, this thread's 4 scales (bf16
        // pairs) and the 3 words of each of its 4 rows.  The slot is released
        // right after.
        struct Held { int take, valid, more; uint32_t s01, s23; uint32_t wv[4][3]; };
        auto take_slot = [&](int cs, Held& h) {
            const uint32_t info = info_base + (uint32_t)cs * 16u;
            uint32_t d0, d1, d2, d3, s01, s23;
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(d0), "=r"(d1), "=r"(d2), "=r"(d3) : "r"(info));
            asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(s01), "=r"(s23)
                         : "r"(scl_base + (uint32_t)cs * kStSclBytes + 2u * (uint32_t)row0));
            (void)d3;
            h.take = (int)d0;
            h.valid = (int)d1;
            h.more = (int)d2;
            h.s01 = s01;
            h.s23 = s23;
            const uint32_t tile = c_base + (uint32_t)cs * kStCBytes;
            #pragma unroll
            for (int i = 0; i < 4; ++i) {
                #pragma unroll
                for (int t = 0; t < 3; ++t) {
                    uint32_t v;
                    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v)
                                 : "r"(tile + ((wofs[t] ^ ((uint32_t)(i ^ sw) << 4)) + ((uint32_t)(i ^ sw) << 7))));
                    h.wv[i][t] = v;
                }
            }
        };
        Held h0, h1;
        bool have = xb < xe;
        if (have) {
            if (!__all_sync(0xffffffffu, tc::mbar_wait(&cfull[0], 0, abort_flag, kStWaitNs))) have = false;
            else take_slot(0, h0);
        }
        for (int j = 0; have; ++j) {
            const int as = j % kStStages;
            const bool more = h0.more != 0;
            // the next stage's slot, read while this stage is decoded
            if (more) {
                const int cn = (j + 1) % kCS;
                if (!__all_sync(0xffffffffu, tc::mbar_wait(&cfull[cn], ((j + 1) / kCS) & 1, abort_flag, kStWaitNs)))
                    break;
                take_slot(cn, h1);
            }
            const bool active = ks < h0.take;
            uint32_t pk[16];
            if (active) {
                // bits [S, S + 64) of each row, back in row order: the window
                // of column t0+e at bit (7-e) k
                uint32_t wl[4][2], ww[4][2];
                #pragma unroll
                for (int i = 0; i < 4; ++i) {
                    wl[i][0] = __funnelshift_r(h0.wv[i][0], h0.wv[i][1], off);
                    wl[i][1] = __funnelshift_r(h0.wv[i][1], h0.wv[i][2], off);
                }
                #pragma unroll
                for (int i = 0; i < 4; ++i) {
                    ww[i][0] = sw ? wl[i ^ 2][0] : wl[i][0];
                    ww[i][1] = sw ? wl[i ^ 2][1] : wl[i][1];
                }
                // rows past the split enter the MMA as zeros (zero scale; the
                // codebook entries are finite)
                float sv[4];
                #pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t pr = i < 2 ? h0.s01 : h0.s23;
                    sv[i] = row0 + i >= h0.valid ? 0.f : bf16_bits_to_float((i & 1) ? pr >> 16 : pr & 0xffffu);
                }
                // All 32 codebook gathers are issued before the first is used:
                // under a busy load pipe one round trip takes hundreds of
                // cycles, and a thread that waits on a few gathers at a time
                // pays it several times per stage.
                uint32_t vb[4][8];
                #pragma unroll
                for (int i = 0; i < 4; ++i) {
                    #pragma unroll
                    for (int e = 0; e < 8; ++e)
                        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(vb[i][e])
                                     : "r"(lut_sa + win_off_sh<K, kLutRepShift>(ww[i], 7 - e)));
                }
                // region r: lane g <- column t0+2r, lane g+8 <- column t0+2r+1;
                // registers (rows 4c, 4c+1) and (rows 4c+2, 4c+3) of each
                auto wgt = [&](int i, int e) { return __fmul_rn(__uint_as_float(vb[i][e]), sv[i]); };
                #pragma unroll
                for (int r = 0; r < 4; ++r) {
                    pk[4 * r + 0] = pack_bf16x2(wgt(0, 2 * r), wgt(1, 2 * r));
                    pk[4 * r + 1] = pack_bf16x2(wgt(2, 2 * r), wgt(3, 2 * r));
                    pk[4 * r + 2] = pack_bf16x2(wgt(0, 2 * r + 1), wgt(1, 2 * r + 1));
                    pk[4 * r + 3] = pack_bf16x2(wgt(2, 2 * r + 1), wgt(3, 2 * r + 1));
                }
            }
            // the warp leaves together: a wait that gave up in one lane ends the loop in all
            if (j >= kStStages &&
                !__all_sync(0xffffffffu, tc::mbar_wait(&aempty[as], ((j / kStStages) - 1) & 1, abort_flag, kStWaitNs)))
                break;
            if (active) {
                tc::tc_fence_after();
                #pragma unroll
                for (int r = 0; r < 4; ++r)
                    tmem_st_16x256b(lane_base + kStACol + (uint32_t)(as * 128 + r * 32 + ks * 8),
                                    pk[4 * r + 0], pk[4 * r + 1], pk[4 * r + 2], pk[4 * r + 3]);
                tc::tmem_wait_st();
            }
            tc::tc_fence_before();
            tc::mbar_arrive(&afull[as]);
            h0 = h1;
            have = more;
        }
    } else if (warp == kStActWarp) {
        // ------------------------------------------------------------ loader
        // One bundle per slot: the stage's code tile (rows r_begin .. +63 of
        // block b, 32 words from the block's first; rows past the matrix and
        // words past its row arrive as zeros), its 64 row scales, and the
        // activation tile x[0 .. NPAD)[r_begin .. +64) (K-major, 128-byte
        // swizzle; rows past M and past the matrix as zeros, rows past the
        // split meet zero weights).  Slot j % kCS was last used by stage j - kCS.
        const uint64_t tmap_ptr = reinterpret_cast<uint64_t>(&tmap);
        if (lane == 0) asm volatile("prefetch.tensormap [%0];" :: "l"(tmap_ptr) : "memory");
        Cursor cur;
        cursor_init(sc, cur, xb, xe);
        Stage st;
        for (int j = 0; next_stage(sc, cur, st); ++j) {
            const int cs = j % kCS;
            if (j >= kCS && !tc::warp_wait(&sempty[cs], ((j / kCS) - 1) & 1, abort_flag, kStWaitNs)) break;
            const uint32_t bar = tc::smem_addr(&cfull[cs]);
            const uint32_t bs = b_base + (uint32_t)cs * Lay::kB;
            if (!tma_x) {
                // scales and activations with plain copies (rows that do not
                // start on a 16-byte boundary), complete before the arrival
                const int r2 = 2 * lane;
                const uint32_t lo = r2 < st.valid ? (uint32_t)__ldg(scales + st.r_begin + r2) : 0u;
                const uint32_t hi = r2 + 1 < st.valid ? (uint32_t)__ldg(scales + st.r_begin + r2 + 1) : 0u;
                reinterpret_cast<uint32_t*>(base + Lay::kSclOff + cs * kStSclBytes)[lane] = lo | (hi << 16);
                #pragma unroll 1
                for (int idx = lane; idx < NPAD * 8; idx += 32) {
                    const int n = idx >> 3, c8 = idx & 7;
                    const uint32_t dst = bs + (uint32_t)n * 128u + ((uint32_t)(c8 ^ (n & 7)) << 4);
                    int cnt = st.valid - 8 * c8;
                    cnt = cnt < 0 ? 0 : cnt > 8 ? 8 : cnt;
                    const int64_t e = (int64_t)n * R + st.r_begin + 8 * c8;
                    uint32_t v[4] = {0u, 0u, 0u, 0u};
                    if (n < M && cnt > 0) {
                        #pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const uint32_t l16 = 2 * q < cnt ? (uint32_t)__ldg(x + e + 2 * q) : 0u;
                            const uint32_t h16 = 2 * q + 1 < cnt ? (uint32_t)__ldg(x + e + 2 * q + 1) : 0u;
                            v[q] = l16 | (h16 << 16);
                        }
                    }
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                                 :: "r"(dst), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]) : "memory");
                }
                tc::fence_proxy_async_smem();
            }
            if (lane == 0) {
                int* d = reinterpret_cast<int*>(base + Lay::kInfoOff + cs * 16);
                d[0] = st.take;
                d[1] = st.valid;
                d[2] = cur.x < cur.xe ? 1 : 0;
                d[3] = 0;
            }
            __syncwarp();
            if (lane == 0) {
                const uint32_t dst = c_base + (uint32_t)cs * kStCBytes;
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                             :: "r"(bar), "r"(kStCBytes + (tma_x ? kStSclBytes + Lay::kB : 0)) : "memory");
                if (tma_x) {
                    asm volatile("cp.async.bulk.tensor.1d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                                 " [%0], [%1, {%2}], [%3];"
                                 :: "r"(s_base + (uint32_t)(Lay::kSclOff + cs * kStSclBytes)),
                                    "l"(reinterpret_cast<uint64_t>(&smap)), "r"((int)st.r_begin), "r"(bar) : "memory");
                    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                                 " [%0], [%1, {%2, %3}], [%4];"
                                 :: "r"(bs), "l"(reinterpret_cast<uint64_t>(&xmap)), "r"((int)st.r_begin), "r"(0),
                                    "r"(bar) : "memory");
                }
                if (interleave == 2) {
                    asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                                 " [%0], [%1, {%2, %3, %4}], [%5];"
                                 :: "r"(dst), "l"(tmap_ptr), "r"((st.b & 1) * wpb), "r"((int)st.r_begin), "r"(st.b >> 1),
                                    "r"(bar) : "memory");
                } else {
                    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                                 " [%0], [%1, {%2, %3}], [%4];"
                                 :: "r"(dst), "l"(tmap_ptr), "r"(st.b * wpb), "r"((int)st.r_begin), "r"(bar) : "memory");
                }
            }
            __syncwarp();
        }
    } else if (warp >= kStMmaWarp) {
        // ------------------------------------------------------------ MMA issue
        // Warp 20 + r issues region r of every stage.  One wait per stage:
        // the decoders arrive on afull after they took the stage's slot, so
        // the slot's activations have landed too.  One commit of each of the
        // four warps frees the A stage, one the slot.
        if (lane == 0) {
            const int r = warp - kStMmaWarp;
            constexpr uint32_t idesc = tc::idesc_bf16_f32(128, NPAD);
            Cursor cur;
            cursor_init(sc, cur, xb, xe);
            Stage st;
            int ic = -1;
            for (int j = 0; next_stage(sc, cur, st); ++j) {
                if (st.first) {
                    ++ic;
                    if (ic >= kDBuf &&
                        !tc::mbar_wait(&dempty[ic % kDBuf], ((ic / kDBuf) - 1) & 1, abort_flag, kStWaitNs))
                        break;
                }
                const int as = j % kStStages, cs = j % kCS;
                if (!tc::mbar_wait(&afull[as], (j / kStStages) & 1, abort_flag, kStWaitNs)) break;
                tc::tc_fence_after();
                const uint32_t d = tmem + (uint32_t)((ic % kDBuf) * (4 * NPAD) + r * NPAD);
                const uint32_t a = tmem + kStACol + (uint32_t)(as * 128 + r * 32);
                // K step kk: 32 bytes further along the swizzled rows (the
                // descriptor's address field counts 16-byte units)
                const uint64_t bd = tc::sdesc_sw128(b_base + (uint32_t)cs * Lay::kB, 1024u);
                for (int kk = 0; kk < st.take; ++kk)
                    tc::mma_ts(d, a + (uint32_t)(kk * 8), bd + (uint64_t)(2 * kk), idesc,
                               (st.first && kk == 0) ? 0u : 1u);
                tc::mma_commit(&aempty[as]);
                tc::mma_commit(&sempty[cs]);
                if (st.last) tc::mma_commit(&dfull[ic % kDBuf]);
            }
            tc::mma_commit(done);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;
        const int g = lane & 7, h = (lane >> 3) & 1;
        Cursor cur;
        cursor_init(sc, cur, xb, xe);
        Stage st;
        int ic = -1;
        bool from_zero = false;
        while (next_stage(sc, cur, st)) {
            if (st.first) {
                ++ic;
                from_zero = st.k == 0;
            }
            if (!st.last) continue;
            const int d = ic % kDBuf;
            if (!tc::warp_wait(&dfull[d], (ic / kDBuf) & 1, abort_flag, kStWaitNs)) break;
            tc::tc_fence_after();
            // the CTA that holds the item's first step writes the partial
            // itself; a CTA that starts inside an item (only ever its first
            // item) writes its share to its own fix-up slot
            float* dstb = from_zero ? partial + (int64_t)st.s * C + (int64_t)st.b * kBT
                                    : fix + ((int64_t)blockIdx.x * M) * kBT;
            const int64_t mstride = from_zero ? (int64_t)sc.S * C : (int64_t)kBT;
            // 16 activation rows at a time
            #pragma unroll 1
            for (int r = 0; r < 4; ++r) {
                #pragma unroll
                for (int m0 = 0; m0 < NPAD; m0 += 16) {
                    uint32_t v[16];
                    tc::tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)d * (4 * NPAD) + (uint32_t)(r * NPAD + m0), v);
                    tc::tmem_wait_ld();
                    if (lane < 16) {           // lanes 16..31 of the quarter carry no column
                        float* dst = dstb + 64 * q + 8 * g + 2 * r + h + m0 * mstride;
                        #pragma unroll
                        for (int m = 0; m < 16; ++m) {
                            if (m0 + m < M) *dst = __uint_as_float(v[m]);
                            dst += mstride;
                        }
                    }
                }
            }
            tc::tc_fence_before();
            tc::warp_arrive(&dempty[d]);
        }
    }

    __syncthreads();
    if (warp == kStMmaWarp) {
        // no MMA of the four issuing warps may still write tensor memory
        // when it is released
        tc::mbar_wait(done, 0, abort_flag, kStWaitNs);
        __syncwarp();
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, kStTmemCols);
    }
    if (threadIdx.x == 0 && *abort_flag) atomicOr(status, kStatusWaitTimeout);
}

// out[m][c] = bf16( sum_s P[m][s][c] ).  The CTA that holds an item's first
// step has written its share of P to the workspace; when the item runs on
// into later CTAs, their fix-up slots are added to it here in CTA order and
// the sum is stored back; P of an empty split is zero.  A CTA covers
// 4 * (256 / groups) columns of one activation row with `groups` groups of
// 256 / groups threads (groups: the power of two at or below min(S, 32),
// at least 4 so that a CTA stays within one 256-column block; few threads
// idle for want of a split); group g takes a contiguous run of splits in
// order, then the runs are added in order.
__host__ __device__ inline int tc_rd_groups(int S) {
    int g = 4;
    while (g * 2 <= S && g * 2 <= 32) g *= 2;
    return g;
}

template <bool F32OUT>
__global__ void __launch_bounds__(256)
tc_split_reduce_kernel(float* __restrict__ partial, const float* __restrict__ fix, SplitSchedule sc,
                       int M, int C, void* __restrict__ out_) {
    __shared__ float4 red[256];
    pdl_wait();
    pdl_release();
    const int S = sc.S;
    const int groups = tc_rd_groups(S);
    const int ct = 256 / groups;                    // float4 columns per CTA
    const int m = blockIdx.y;
    const int grp = threadIdx.x / ct, ci = threadIdx.x - grp * ct;
    const int col = (blockIdx.x * ct + ci) * 4;
    const int b = col >> 8, cl = col & 255;
    const int per = (S + groups - 1) / groups;
    const int s0 = grp * per, s1 = min(S, s0 + per);
    const bool sm32 = sc.small();
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = s0; s < s1; ++s) {
        float4* pp = reinterpret_cast<float4*>(partial + ((int64_t)m * S + s) * C + col);
        const int n = sc.steps(s);
        float4 p = make_float4(0.f, 0.f, 0.f, 0.f);
        if (n == 0) {
            *pp = p;
        } else {
            const int64_t x0 = (int64_t)sc.NB * sc.prefix(s) + (int64_t)b * n;
            const int g1 = sm32 ? sc.cta_of32((uint32_t)x0) : sc.cta_of(x0);
            const int g2 = sm32 ? sc.cta_of32((uint32_t)(x0 + n - 1)) : sc.cta_of(x0 + n - 1);
            p = *pp;
            if (g2 > g1) {
                for (int g = g1 + 1; g <= g2; ++g) {
                    const bool empty = sm32 ? sc.start32(g) == sc.start32(g + 1) : sc.start(g) == sc.start(g + 1);
                    if (empty) continue;                                // a CTA with no steps
                    const float4 v = *reinterpret_cast<const float4*>(fix + ((int64_t)g * M + m) * kBT + cl);
                    p.x += v.x; p.y += v.y; p.z += v.z; p.w += v.w;
                }
                *pp = p;
            }
        }
        a.x += p.x; a.y += p.y; a.z += p.z; a.w += p.w;
    }
    red[threadIdx.x] = a;
    __syncthreads();
    if (grp == 0) {
        float4 t = red[ci];
        for (int g = 1; g < groups; ++g) {
            const float4 v = red[g * ct + ci];
            t.x += v.x; t.y += v.y; t.z += v.z; t.w += v.w;
        }
        if constexpr (F32OUT) {
            *reinterpret_cast<float4*>(static_cast<float*>(out_) + (int64_t)m * C + col) = t;
        } else {
            __nv_bfloat162 lo = __floats2bfloat162_rn(t.x, t.y);
            __nv_bfloat162 hi = __floats2bfloat162_rn(t.z, t.w);
            uint2 o;
            o.x = *reinterpret_cast<uint32_t*>(&lo);
            o.y = *reinterpret_cast<uint32_t*>(&hi);
            *reinterpret_cast<uint2*>(static_cast<uint16_t*>(out_) + (int64_t)m * C + col) = o;
        }
    }
}

// cuTensorMapEncodeTiled, found once through the runtime (no link-time
// dependence on the driver library).
using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_tiled() {
    static std::once_flag once;
    static EncodeTiled fn = nullptr;
    std::call_once(once, []() {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(f);
        cudaGetLastError();
    });
    return fn;
}

// The codes as a tensor of uint32 words: interleave 0 is [rows][words of a
// row]; interleave 2 is [block pairs][rows][2 * wpb].  The box is 32 words
// (128 bytes, one swizzle row) by 64 rows.
cudaError_t code_tensor_map(const Packed& p, CUtensorMap* map) {
    EncodeTiled enc = encode_tiled();
    if (!enc) return cudaErrorNotSupported;
    const int wpb = kBT * p.k / 32;
    const cuuint64_t nb = (cuuint64_t)(p.cols / kBT);
    cuuint64_t dims[3], strides[2];
    cuuint32_t box[3] = {32, (cuuint32_t)kStRows, 1}, estr[3] = {1, 1, 1};
    cuuint32_t rank;
    if (p.interleave == 2) {
        rank = 3;
        dims[0] = 2 * (cuuint64_t)wpb;
        dims[1] = (cuuint64_t)p.rows;
        dims[2] = nb / 2;
        strides[0] = dims[0] * 4;
        strides[1] = strides[0] * dims[1];
    } else {
        rank = 2;
        dims[0] = nb * (cuuint64_t)wpb;
        dims[1] = (cuuint64_t)p.rows;
        strides[0] = dims[0] * 4;
    }
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, rank, const_cast<uint32_t*>(p.codes), dims, strides, box,
                           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// The activations x [M][R] (bf16) with a box of 64 input rows by npad
// activation rows and the 128-byte swizzle, which is the MMA's K-major B
// layout; and the scales [R] (bf16) with a box of 64.
cudaError_t act_tensor_maps(const Packed& p, const uint16_t* x, int M, int npad, CUtensorMap* xmap,
                            CUtensorMap* smap) {
    EncodeTiled enc = encode_tiled();
    if (!enc) return cudaErrorNotSupported;
    const cuuint32_t estr[2] = {1, 1};
    const cuuint64_t xd[2] = {(cuuint64_t)p.rows, (cuuint64_t)M};
    const cuuint64_t xs[1] = {(cuuint64_t)p.rows * 2};
    const cuuint32_t xb[2] = {(cuuint32_t)kStRows, (cuuint32_t)npad};
    CUresult r = enc(xmap, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<uint16_t*>(x), xd, xs, xb, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    const cuuint64_t sd[1] = {(cuuint64_t)p.rows};
    const cuuint32_t sb[1] = {(cuuint32_t)kStRows};
    const cuuint64_t ss[1] = {(cuuint64_t)p.rows * 2};   // not read for a rank-1 tensor
    r = enc(smap, CU_TENSOR_MAP_DATA_TYPE_UINT16, 1, const_cast<uint16_t*>(p.scales), sd, ss, sb, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int K, int NPAD>
cudaError_t launch_kn(const Packed& p, const uint16_t* x, int M, const SplitSchedule& sc, float* partial,
                      float* fix, int* status, const CUtensorMap& map, cudaStream_t stream) {
    const int smem = StLayout<NPAD>::kAlloc;
    cudaError_t e = cudaFuncSetAttribute(scatter_tc_kernel<K, NPAD>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // TMA for the activations and scales when every stage's first row is a
    // multiple of 8 (16 bytes of bf16) and x, scales and rows allow it
    const bool tma_x = p.rows % 8 == 0 && sc.rp % 8 == 0 && (reinterpret_cast<uintptr_t>(x) & 15u) == 0 &&
                       (reinterpret_cast<uintptr_t>(p.scales) & 15u) == 0;
    alignas(64) CUtensorMap xmap, smap;
    if (tma_x) {
        e = act_tensor_maps(p, x, M, NPAD, &xmap, &smap);
        if (e != cudaSuccess) return e;
    } else {
        xmap = map;                    // unused
        smap = map;
    }
    return launch_pdl(scatter_tc_kernel<K, NPAD>, dim3((unsigned)sc.G), dim3(kStThreads), (size_t)smem, stream, x, M,
                      p.codes, p.scales, p.lut, (int)p.cols, p.interleave, sc, partial, fix, status, map, xmap,
                      smap, tma_x ? 1 : 0);
}

template <int K>
cudaError_t launch_k(const Packed& p, const uint16_t* x, int M, const SplitSchedule& sc, float* partial,
                     float* fix, int* status, const CUtensorMap& map, cudaStream_t stream) {
    if (M <= 16) return launch_kn<K, 16>(p, x, M, sc, partial, fix, status, map, stream);
    return launch_kn<K, 32>(p, x, M, sc, partial, fix, status, map, stream);
}

}  // namespace

cudaError_t launch_scatter_tc(const Packed& p, const uint16_t* x, int M, int splits, float* partial,
                              float* fix, void* out, bool out_f32, int* status, int sm_count,
                              cudaStream_t stream) {
    const int64_t C = p.cols;
    SplitSchedule sc = SplitSchedule::make(p.rows, splits, C, 1);
    int64_t G = sm_count < kScatterTcMaxCtas ? sm_count : kScatterTcMaxCtas;
    if (G > sc.T) G = sc.T;
    if (G < 1) G = 1;
    sc.G = (int)G;
    alignas(64) CUtensorMap map;
    cudaError_t e = code_tensor_map(p, &map);
    if (e != cudaSuccess) return e;
    switch (p.k) {
        case 2: e = launch_k<2>(p, x, M, sc, partial, fix, status, map, stream); break;
        case 3: e = launch_k<3>(p, x, M, sc, partial, fix, status, map, stream); break;
        case 4: e = launch_k<4>(p, x, M, sc, partial, fix, status, map, stream); break;
        default: return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return e;
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // C is a multiple of 256 and a CTA covers 32..256 columns
    const dim3 rgrid((unsigned)(C / (4 * (256 / tc_rd_groups(splits)))), (unsigned)M);
    e = out_f32 ? launch_pdl(tc_split_reduce_kernel<true>, rgrid, dim3(256), 0,
                             stream, partial, static_cast<const float*>(fix), sc, M, (int)C, out)
                : launch_pdl(tc_split_reduce_kernel<false>, rgrid, dim3(256), 0,
                             stream, partial, static_cast<const float*>(fix), sc, M, (int)C, out);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace tcq
