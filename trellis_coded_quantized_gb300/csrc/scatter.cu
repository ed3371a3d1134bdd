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
//   - more than 4 activation rows are processed in passes of up to 4;
//   - the unrounded contract (scatter.ts, balanced scatter kernels: the f32
//     product of codebook value and scale, no bf16 rounding) folds the row's
//     scale into the activations, x[m][r] * scale[r] once per row, and
//     contracts the codebook values with them in f32.
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace tcq {
namespace {

// Row warps per column range: 4 with one activation row, else 2; warps per
// CTA at most 20 (one activation row) or 10 (the accumulators of 2..4 rows
// need the larger register share).
__host__ __device__ constexpr int sc_row_warps(int mb) { return mb == 1 ? 4 : 2; }
__host__ __device__ constexpr int sc_max_warps(int mb) { return mb == 1 ? 20 : 10; }

template <int K, int MB, bool UNR>
__global__ void __launch_bounds__(sc_max_warps(MB) * 32, 1)
scatter_kernel(const uint16_t* __restrict__ x, int m0, const uint32_t* __restrict__ codes,
               const uint16_t* __restrict__ scales, const float* __restrict__ lut,
               int R, int C, int splits, int rp, int nur, int nurb, int interleave,
               float* __restrict__ partial) {
    constexpr int RW = sc_row_warps(MB);
    extern __shared__ __align__(16) float smem[];
    float* lut_s = smem;                                // 8-way replicated codebook
    float* red = smem + kLutN * kLutRep;                // [RW-1][nurb][MB][32 cols][32 lanes]
    stage_lut_rep8(lut_s, lut);                         // a weight input: before the wait
    pdl_wait();                                         // x, and the partials the last reduction read
    __syncthreads();
    // let the split reduction be scheduled now (it waits for this grid's
    // completion before reading anything)
    pdl_release();

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
        if constexpr (UNR) {
            float xs[MB];                               // x[m][r] * scale[r]
            #pragma unroll
            for (int m = 0; m < MB; ++m) xs[m] = bf16_bits_to_float(__ldg(x + (int64_t)(m0 + m) * R + r)) * sr;
            #pragma unroll
            for (int i = 0; i < 32; i += 2) {
                const float v0 = lut_at(lut_s, win_off_sh<K, kLutRepShift>(w, i) | gofs);
                const float v1 = lut_at(lut_s, win_off_sh<K, kLutRepShift>(w, i + 1) | gofs);
                #pragma unroll
                for (int m = 0; m < MB; ++m) {
                    acc[m][i] = fmaf(v0, xs[m], acc[m][i]);
                    acc[m][i + 1] = fmaf(v1, xs[m], acc[m][i + 1]);
                }
            }
        } else {
            uint32_t xx[MB];                            // x[m][r] in both halves
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

template <bool F32OUT, int B>
__global__ void __launch_bounds__(256)
split_reduce_kernel(const float* __restrict__ partial, int splits, int C, void* __restrict__ out_) {
    __shared__ float4 red[kRdGroups][kRdCols / 4];
    // launched as a programmatic dependent of the scatter: wait until that
    // grid has completed and its partials are visible (a no-op otherwise)
    pdl_wait();
    pdl_release();
    const int m = blockIdx.y;
    const int cq = blockIdx.x * (kRdCols / 4) + (threadIdx.x & 7);   // float4 column index
    const int grp = threadIdx.x >> 3;
    const int per = (splits + kRdGroups - 1) / kRdGroups;
    const int s0 = grp * per, s1 = min(splits, s0 + per);
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    const float4* p = reinterpret_cast<const float4*>(partial + (int64_t)m * splits * C) + cq;
    const int64_t stride = C / 4;
    // the run's loads issued B at a time (one L2 round trip for up to B
    // splits), then added in split order
    for (int s = s0; s < s1; s += B) {
        float4 v[B];
        #pragma unroll
        for (int j = 0; j < B; ++j)
            if (s + j < s1) v[j] = __ldg(p + (int64_t)(s + j) * stride);
        #pragma unroll
        for (int j = 0; j < B; ++j)
            if (s + j < s1) { a.x += v[j].x; a.y += v[j].y; a.z += v[j].z; a.w += v[j].w; }
    }
    red[grp][threadIdx.x & 7] = a;
    __syncthreads();
    if (grp == 0) {
        float4 t = red[0][threadIdx.x];
        for (int g = 1; g < kRdGroups; ++g) {
            const float4 v = red[g][threadIdx.x];
            t.x += v.x; t.y += v.y; t.z += v.z; t.w += v.w;
        }
        if constexpr (F32OUT) {
            reinterpret_cast<float4*>(out_)[(int64_t)m * (C / 4) + cq] = t;
        } else {
            __nv_bfloat162 lo = __floats2bfloat162_rn(t.x, t.y);
            __nv_bfloat162 hi = __floats2bfloat162_rn(t.z, t.w);
            uint2 o;
            o.x = *reinterpret_cast<uint32_t*>(&lo);
            o.y = *reinterpret_cast<uint32_t*>(&hi);
            *reinterpret_cast<uint2*>(static_cast<uint16_t*>(out_) + (int64_t)m * C + cq * 4) = o;
        }
    }
}

template <int K, int MB, bool UNR>
cudaError_t launch_pass(const Packed& p, const uint16_t* x, int m0, int splits, int rp, int nur,
                        float* partial, cudaStream_t stream) {
    constexpr int RW = sc_row_warps(MB);
    const int nurb = nur < sc_max_warps(MB) / RW ? nur : sc_max_warps(MB) / RW;
    const int nblk = (nur + nurb - 1) / nurb;
    const size_t smem = kLutRepBytes + (size_t)(RW - 1) * nurb * MB * 1024 * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(scatter_kernel<K, MB, UNR>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)(splits * nblk);
    e = launch_pdl(scatter_kernel<K, MB, UNR>, dim3(grid), dim3(nurb * RW * 32), smem, stream, x, m0, p.codes,
                   p.scales, p.lut, (int)p.rows, (int)p.cols, splits, rp, nur, nurb, p.interleave, partial);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int K, bool UNR>
cudaError_t launch_k(const Packed& p, const uint16_t* x, int M, int splits, float* partial,
                     cudaStream_t stream) {
    const int rp = (int)((p.rows + splits - 1) / splits);
    const int units = (int)(p.cols / 32);
    const int nur = (units + 31) / 32;
    for (int m0 = 0; m0 < M; m0 += 4) {
        const int mb = M - m0 < 4 ? M - m0 : 4;
        cudaError_t e;
        switch (mb) {
            case 1: e = launch_pass<K, 1, UNR>(p, x, m0, splits, rp, nur, partial, stream); break;
            case 2: e = launch_pass<K, 2, UNR>(p, x, m0, splits, rp, nur, partial, stream); break;
            case 3: e = launch_pass<K, 3, UNR>(p, x, m0, splits, rp, nur, partial, stream); break;
            default: e = launch_pass<K, 4, UNR>(p, x, m0, splits, rp, nur, partial, stream); break;
        }
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

// ---------------------------------------------------------------------------
// Axis-0 scatter for 3..32 activation rows on the tensor cores (mma.sync
// m16n8k16, bf16 x bf16 -> f32): D[col][m] += W^T[col][r] * X^T[r][m], the
// output columns are the MMA rows and the input rows of the split are K
// (the split-K prefill of splitk-prefill.ts computes the same partials with
// 8x8 simdgroup MMAs).  A warp owns 128-column tiles of its split; lane
// (g, c) = (lane / 4, lane % 4) owns the 16 consecutive columns 16g..16g+15
// of the tile, i.e. 16 consecutive windows of each row, and the rows
// 2c, 2c+1, 2c+8, 2c+9 of every 16-row step.  Its A fragment of m-tile mt
// takes columns 2mt (MMA row g) and 2mt+1 (row g+8), so the decoded weights
// go straight from the codebook into fragment registers; B is read from x
// as K-adjacent pairs.  Each weight is decoded once for all M rows.
// ---------------------------------------------------------------------------
namespace {

__device__ __forceinline__ void mma_bf16_16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
                 "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__host__ __device__ constexpr int smma_warps(int nt) { return nt == 1 ? 20 : nt == 2 ? 10 : 8; }

// XS: the split's activations (bf16 [NT*8][xpitch], rows past the split and
// activation rows past M zero) and scales (f32 [rp16]) are staged in shared
// memory once per CTA, so the B operands and scales of a step are
// conflict-free shared loads (xpitch/2 words = 4 mod 32: lanes (g, c) hit
// banks 4g + c) instead of global loads that touch 8 lines each.
// UNR: the unrounded contract.  The f32 weight w = lut * scale is carried as
// three bf16 terms, hi = bf16(w), mid = bf16(w - hi), lo = bf16(w - hi -
// mid) (each difference exact in f32), contracted by three MMAs: the weight
// is kept to 24 significant bits, as in the f32 product.
template <int K, int NT, bool XS, bool UNR>
__global__ void __launch_bounds__(smma_warps(NT) * 32, 1)
scatter_mma_kernel(const uint16_t* __restrict__ x, int M, const uint32_t* __restrict__ codes,
                   const uint16_t* __restrict__ scales, const float* __restrict__ lut,
                   int R, int C, int splits, int rp, int interleave, int xpitch, int rp16,
                   float* __restrict__ partial) {
    extern __shared__ __align__(16) float smem[];
    float* lut_s = smem;                                // 8-way replicated codebook
    stage_lut_rep8(lut_s, lut);                         // a weight input: before the wait
    pdl_wait();

    constexpr int wpb = kBT * K / 32;
    // per warp: 2 chunks of 16 rows x (4k + 2 used) words of the tile's half
    // block; the row pitch (20 words for k=3, 4k+4 else) is 4 or 12 mod 16, so
    // the 4 rows a warp reads at once start 8 banks apart
    constexpr int kPitchW = K == 3 ? 20 : 4 * K + 4;
    constexpr int kChunkW = 16 * kPitchW;
    const int s = blockIdx.x;
    const int r0 = s * rp;
    const int r1 = min(R, r0 + rp);
    const int nsteps = (max(r1 - r0, 0) + 15) / 16;
    uint32_t* xs32 = reinterpret_cast<uint32_t*>(smem + kLutN * kLutRep) + smma_warps(NT) * 2 * kChunkW;
    float* ss = reinterpret_cast<float*>(xs32 + NT * 8 * (xpitch >> 1));
    if constexpr (XS) {
        const int nr = max(r1 - r0, 0);
        const int hp = xpitch >> 1;
        for (int i = threadIdx.x; i < NT * 8 * hp; i += blockDim.x) {
            const int m = i / hp, rr = 2 * (i - m * hp);
            uint32_t v = 0u;
            if (m < M) {
                const uint16_t* xr = x + (int64_t)m * R + r0;
                const uint32_t lo16 = rr < nr ? __ldg(xr + rr) : 0u;
                const uint32_t hi16 = rr + 1 < nr ? __ldg(xr + rr + 1) : 0u;
                v = lo16 | (hi16 << 16);
            }
            xs32[i] = v;
        }
        for (int i = threadIdx.x; i < rp16; i += blockDim.x)
            ss[i] = i < nr ? bf16_bits_to_float(__ldg(scales + r0 + i)) : 0.f;
    }
    __syncthreads();
    pdl_release();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const uint32_t gofs = lut_rep_lane_offset();
    const int64_t rs = block_row_stride(C / kBT, wpb, interleave);
    const int ntiles = C / 128;

    for (int ct = warp; ct < ntiles; ct += smma_warps(NT)) {
        const int b = ct >> 1, h = ct & 1;
        // bits of the 16 windows of this lane: [lo, lo + 15k + 12) of the block
        const int lo = (240 - 128 * h - 16 * g) * K;
        const int wl = lo >> 5, sh = lo & 31;
        const uint32_t* blk = codes + block_col_base(b, R, wpb, interleave);
        float acc[8][NT][4];
        #pragma unroll
        for (int mt = 0; mt < 8; ++mt)
            #pragma unroll
            for (int nt = 0; nt < NT; ++nt)
                #pragma unroll
                for (int e = 0; e < 4; ++e) acc[mt][nt][e] = 0.f;

        // The tile's words of a row: the half block [4k(1-h), 4k(1-h) + 4k) and
        // the two words after it in the block (wrapping to words 0, 1 for
        // h = 0) -- every window of the 128 columns lies inside them.
        uint32_t* cbuf = reinterpret_cast<uint32_t*>(smem + kLutN * kLutRep) + warp * 2 * kChunkW;
        const int span0 = 4 * K * (1 - h);
        const int ext0 = (span0 + 4 * K) % wpb;
        const int lw = wl - span0;                      // this lane's first word in a chunk row
        auto stage = [&](int ks, int buf) {
            uint32_t* dst = cbuf + buf * kChunkW;
            for (int idx = lane; idx < 16 * (K + 1); idx += 32) {
                const int rr = idx / (K + 1), part = idx - rr * (K + 1);
                const int r = r0 + 16 * ks + rr;
                if (r >= r1) continue;
                const uint32_t* rowp = blk + (int64_t)r * rs;
                const uint32_t sa = tc::smem_addr(dst + rr * kPitchW + 4 * part);
                if (part < K)
                    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(sa), "l"(rowp + span0 + 4 * part) : "memory");
                else
                    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" :: "r"(sa), "l"(rowp + ext0) : "memory");
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
        };
        // scales and B operands of a step, one step ahead of their use
        struct Step { float sq[4]; uint32_t bf[NT][2]; };
        auto fetch = [&](int ks, Step& st) {
            if constexpr (XS) {
                #pragma unroll
                for (int q = 0; q < 4; ++q) st.sq[q] = ss[16 * ks + 2 * c + (q & 1) + 8 * (q >> 1)];
                #pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    #pragma unroll
                    for (int hh = 0; hh < 2; ++hh)
                        st.bf[nt][hh] = xs32[(8 * nt + g) * (xpitch >> 1) + 8 * ks + c + 4 * hh];
                return;
            }
            #pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int r = r0 + 16 * ks + 2 * c + (q & 1) + 8 * (q >> 1);
                st.sq[q] = r < r1 ? bf16_bits_to_float(__ldg(scales + r)) : 0.f;
            }
            // B: x[m][r], x[m][r+1] for r = 16ks + 2c (+8); rows past the split read as zero
            #pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int m = 8 * nt + g;
                st.bf[nt][0] = st.bf[nt][1] = 0u;
                if (m < M) {
                    const uint16_t* xr = x + (int64_t)m * R;
                    #pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int ra = r0 + 16 * ks + 2 * c + 8 * hh;
                        // one 4-byte load when the pair starts on an even element of x
                        if (((((int64_t)m * R + ra) & 1) == 0) && ra + 1 < r1) {
                            st.bf[nt][hh] = __ldg(reinterpret_cast<const uint32_t*>(xr + ra));
                        } else {
                            const uint32_t lo = ra < r1 ? __ldg(xr + ra) : 0u;
                            const uint32_t hi = ra + 1 < r1 ? __ldg(xr + ra + 1) : 0u;
                            st.bf[nt][hh] = lo | (hi << 16);
                        }
                    }
                }
            }
        };
        // the step loop unrolled by two: the operands of step ks+1 are
        // fetched into the other Step instead of being copied at the end of
        // the step (M=16: 2%, M=32: 5% faster on GB300)
        Step sa, sb;
        auto one_step = [&](int ks, Step& cur, Step& nxt) {
            if (ks + 1 < nsteps) {
                stage(ks + 1, (ks + 1) & 1);
                fetch(ks + 1, nxt);
                asm volatile("cp.async.wait_group 1;" ::: "memory");
            } else {
                asm volatile("cp.async.wait_group 0;" ::: "memory");
            }
            __syncwarp();
            const uint32_t* ch = cbuf + (ks & 1) * kChunkW;
            uint32_t wq[4][3];
            #pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t* rw = ch + (2 * c + (q & 1) + 8 * (q >> 1)) * kPitchW + lw;
                const uint32_t w0 = rw[0], w1 = rw[1], w2 = rw[2];
                // bit lo of the block becomes bit 0
                wq[q][0] = __funnelshift_r(w0, w1, sh);
                wq[q][1] = __funnelshift_r(w1, w2, sh);
                wq[q][2] = w2 >> sh;
            }
            const float* sq = cur.sq;
            #pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                // column j = 2mt (MMA row g) and j = 2mt+1 (row g+8); window of
                // column j sits at bit (15 - j) * k of the shifted words
                float v[4][2];
                #pragma unroll
                for (int q = 0; q < 4; ++q) {
                    v[q][0] = lut_at(lut_s, win_off_sh<K, kLutRepShift>(wq[q], 15 - 2 * mt) | gofs);
                    v[q][1] = lut_at(lut_s, win_off_sh<K, kLutRepShift>(wq[q], 14 - 2 * mt) | gofs);
                }
                if constexpr (UNR) {
                    // fragment register e holds (lo half, hi half) = (w[q0][j], w[q1][j])
                    float wl[4], wh[4];
                    #pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int q0 = 2 * (e >> 1), j = e & 1;
                        wl[e] = __fmul_rn(v[q0][j], sq[q0]);
                        wh[e] = __fmul_rn(v[q0 + 1][j], sq[q0 + 1]);
                    }
                    #pragma unroll
                    for (int term = 0; term < 3; ++term) {
                        uint32_t a[4];
                        #pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            a[e] = pack_bf16x2(wl[e], wh[e]);
                            wl[e] = __fsub_rn(wl[e], __uint_as_float(a[e] << 16));
                            wh[e] = __fsub_rn(wh[e], __uint_as_float(a[e] & 0xffff0000u));
                        }
                        #pragma unroll
                        for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(acc[mt][nt], a, cur.bf[nt][0], cur.bf[nt][1]);
                    }
                } else {
                    uint32_t a[4];
                    a[0] = pack_bf16x2(__fmul_rn(v[0][0], sq[0]), __fmul_rn(v[1][0], sq[1]));
                    a[1] = pack_bf16x2(__fmul_rn(v[0][1], sq[0]), __fmul_rn(v[1][1], sq[1]));
                    a[2] = pack_bf16x2(__fmul_rn(v[2][0], sq[2]), __fmul_rn(v[3][0], sq[3]));
                    a[3] = pack_bf16x2(__fmul_rn(v[2][1], sq[2]), __fmul_rn(v[3][1], sq[3]));
                    #pragma unroll
                    for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(acc[mt][nt], a, cur.bf[nt][0], cur.bf[nt][1]);
                }
            }
            // all lanes are done with this chunk before it is refilled
            __syncwarp();
        };
        if (nsteps > 0) { stage(0, 0); fetch(0, sa); }
        for (int ks = 0; ks < nsteps; ks += 2) {
            one_step(ks, sa, sb);
            if (ks + 1 < nsteps) one_step(ks + 1, sb, sa);
        }
        // D[row][n]: rows g / g+8 are columns 2mt / 2mt+1, n = 2c, 2c+1 are tokens
        const int64_t cbase = (int64_t)b * kBT + 128 * h + 16 * g;
        #pragma unroll
        for (int mt = 0; mt < 8; ++mt)
            #pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int m = 8 * nt + 2 * c;
                const int64_t col = cbase + 2 * mt;
                if (m < M)
                    *reinterpret_cast<float2*>(partial + ((int64_t)m * splits + s) * C + col) =
                        make_float2(acc[mt][nt][0], acc[mt][nt][2]);
                if (m + 1 < M)
                    *reinterpret_cast<float2*>(partial + ((int64_t)(m + 1) * splits + s) * C + col) =
                        make_float2(acc[mt][nt][1], acc[mt][nt][3]);
            }
    }
}

template <int K, int NT, bool XS, bool UNR>
cudaError_t launch_mma_xs(const Packed& p, const uint16_t* x, int M, int splits, int rp, int xpitch, int rp16,
                          size_t smem, float* partial, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(scatter_mma_kernel<K, NT, XS, UNR>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(scatter_mma_kernel<K, NT, XS, UNR>, dim3((unsigned)splits), dim3(smma_warps(NT) * 32), smem, stream,
                   x, M, p.codes, p.scales, p.lut, (int)p.rows, (int)p.cols, splits, rp, p.interleave, xpitch, rp16,
                   partial);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Activations and scales of a split go to shared memory when they take at
// most this many bytes (row splits of up to ~600 rows at M = 32); longer
// splits read them from global memory.
constexpr size_t kXsBudget = 40960;

template <int K, int NT, bool UNR>
cudaError_t launch_mma_nt(const Packed& p, const uint16_t* x, int M, int splits, float* partial,
                          cudaStream_t stream) {
    const int rp = (int)((p.rows + splits - 1) / splits);
    const int rp16 = (rp + 15) / 16 * 16;
    const int xpitch = rp16 + (((8 - rp16) % 64) + 64) % 64;     // xpitch / 2 words = 4 mod 32
    const size_t xs_bytes = (size_t)NT * 8 * xpitch * 2 + (size_t)rp16 * 4;
    const size_t base = kLutRepBytes + (size_t)smma_warps(NT) * 2 * 16 * (K == 3 ? 20 : 4 * K + 4) * sizeof(uint32_t);
    if (xs_bytes <= kXsBudget)
        return launch_mma_xs<K, NT, true, UNR>(p, x, M, splits, rp, xpitch, rp16, base + xs_bytes, partial, stream);
    return launch_mma_xs<K, NT, false, UNR>(p, x, M, splits, rp, 0, rp16, base, partial, stream);
}

template <int K, bool UNR>
cudaError_t launch_mma(const Packed& p, const uint16_t* x, int M, int splits, float* partial,
                       cudaStream_t stream) {
    if (M <= 8) return launch_mma_nt<K, 1, UNR>(p, x, M, splits, partial, stream);
    if (M <= 16) return launch_mma_nt<K, 2, UNR>(p, x, M, splits, partial, stream);
    return launch_mma_nt<K, 4, UNR>(p, x, M, splits, partial, stream);
}

}  // namespace


// Fewest activation rows that take the tensor-core scatter (GB300, 17408 x
// 5120, k=3, back to back: M=2 FMA 47.7 / tensor 54.6 us, M=3 61.4 / 56.0,
// M=4 65.9 / 57.6).
#ifndef TCQ_MMA_MIN_ROWS
#define TCQ_MMA_MIN_ROWS 3
#endif
constexpr int kMmaMinRows = TCQ_MMA_MIN_ROWS;

cudaError_t launch_scatter(const Packed& p, const uint16_t* x, int M, int splits,
                           float* partial, float* fix, void* out, bool out_f32, int* status, int sm_count,
                           cudaStream_t stream) {
    // 3 and more activation rows, rounded contract, fewer than 128 splits:
    // the tcgen05 kernel, whose stream-K schedule fills every SM whatever the
    // split count.  From 128 splits one mma.sync CTA per split fills the SMs
    // as well and has no per-item overhead (17408 x 5120, k=3, back to back:
    // M=4 at 128 splits 56.5 us against 70.9 on tcgen05; M=16 at 128 splits
    // 79.3 against 86.1; M=16 at 8 splits 57.1 on tcgen05 against 893).
    if (scatter_uses_tc(M, p.unrounded) && splits < kScatterTcMaxSplits)
        return launch_scatter_tc(p, x, M, splits, partial, fix, out, out_f32, status, sm_count, stream);
    cudaError_t e;
    // up to 2 activation rows: FMA kernel, each decoded weight feeding every
    // row; 3 and more: one pass on the tensor cores (under the unrounded
    // contract with each f32 weight as three bf16 terms)
    const bool fma = M < kMmaMinRows;
    switch (p.k * 2 + (p.unrounded ? 1 : 0)) {
        case 4: e = fma ? launch_k<2, false>(p, x, M, splits, partial, stream) : launch_mma<2, false>(p, x, M, splits, partial, stream); break;
        case 5: e = fma ? launch_k<2, true>(p, x, M, splits, partial, stream) : launch_mma<2, true>(p, x, M, splits, partial, stream); break;
        case 6: e = fma ? launch_k<3, false>(p, x, M, splits, partial, stream) : launch_mma<3, false>(p, x, M, splits, partial, stream); break;
        case 7: e = fma ? launch_k<3, true>(p, x, M, splits, partial, stream) : launch_mma<3, true>(p, x, M, splits, partial, stream); break;
        case 8: e = fma ? launch_k<4, false>(p, x, M, splits, partial, stream) : launch_mma<4, false>(p, x, M, splits, partial, stream); break;
        case 9: e = fma ? launch_k<4, true>(p, x, M, splits, partial, stream) : launch_mma<4, true>(p, x, M, splits, partial, stream); break;
        default: return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return e;
    const int C = (int)p.cols;
    // programmatic dependent launch: the reduction's CTAs are placed while
    // the last scatter pass still runs and start reading when it completes
    // With at most two CTAs per SM (M = 1) each thread issues its run's
    // loads 8 at a time; larger grids keep a split per load and 8 CTAs per
    // SM in flight (the 8-wide form needs twice the registers).
    const dim3 rgrid((unsigned)(C / kRdCols), (unsigned)M);
    const bool wide = (int64_t)rgrid.x * rgrid.y <= 2 * (int64_t)sm_count;
    if (out_f32)
        e = wide ? launch_pdl(split_reduce_kernel<true, 8>, rgrid, dim3(256), 0, stream,
                              static_cast<const float*>(partial), splits, C, out)
                 : launch_pdl(split_reduce_kernel<true, 1>, rgrid, dim3(256), 0, stream,
                              static_cast<const float*>(partial), splits, C, out);
    else
        e = wide ? launch_pdl(split_reduce_kernel<false, 8>, rgrid, dim3(256), 0, stream,
                              static_cast<const float*>(partial), splits, C, out)
                 : launch_pdl(split_reduce_kernel<false, 1>, rgrid, dim3(256), 0, stream,
                              static_cast<const float*>(partial), splits, C, out);
    if (e != cudaSuccess) return e;
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
// keeps the fp32 split partials, and the fix-up slots of the tensor-core
// path, in a fixed array in device memory that the library itself declares,
// so the call needs no allocation at all.  The driver reserves the array
// when the library's scatter code is first used on a GPU (lazy module
// loading), and it stays reserved on every GPU that used it until the
// process exits.
// ---------------------------------------------------------------------------
#include "trellis.h"

#include <mutex>

namespace {

// 16 MiB of partials (M * splits * cols <= 4,194,304), then 5 MiB for the
// fix-up slots of the tensor-core path at up to 32 activation rows
constexpr size_t kNoAllocPartialFloats = size_t(1) << 22;
constexpr size_t kNoAllocScratchFloats =
    kNoAllocPartialFloats + (size_t)tcq::kScatterTcMaxCtas * 32 * 256;
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
    // invalid arguments give 0 here and are reported by trellis_scatter
    const size_t need = trellis_scatter_workspace_bytes(g, M, splits);
    if (need > 0 && (size_t)M *
                        (size_t)tcq::scatter_splits(g->rows, g->cols, M, splits,
                                                    (g->flags & TRELLIS_FLAG_UNROUNDED) != 0) *
                        (size_t)g->cols >
                        kNoAllocPartialFloats)
        return TRELLIS_ERR_WORKSPACE;
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
    // Every partial and fix-up slot the reduction reads is written by this
    // same call (empty splits store zeros), so nothing in the scratch has to
    // be cleared first.  The partials fit the first 16 MiB, so the fix-up
    // slots that trellis_scatter places right after them fit the array.
    return trellis_scatter(x, M, codes, scales, lut, g, splits, g_scratch_ptr[dev],
                           kNoAllocScratchFloats * sizeof(float), out, stream);
}
