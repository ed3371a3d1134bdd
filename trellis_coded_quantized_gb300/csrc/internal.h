// Launchers behind the C ABI (host side, C++ linkage).  Arguments are
// validated by the ABI layer before any of these is called.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace tcq {

struct Packed {              // one packed matrix
    const uint32_t* codes;   // [rows, (cols/256)*wpb]
    const uint16_t* scales;  // bf16 [rows]
    const float* lut;        // f32 [4096]
    int64_t rows, cols;
    int k;                   // bits per symbol
    int interleave;          // 0: contiguous blocks; 2: blocks paired across rows
    bool unrounded;          // weight lut*scale not rounded to bf16
};

cudaError_t launch_expand(const Packed& p, uint16_t* w_out, uint16_t* win_out,
                          int sm_count, cudaStream_t stream);

// M = 1, axis 1: out[r] = sum_c x[c] w[r][c]
cudaError_t launch_matvec(const Packed& p, const uint16_t* x, uint16_t* out,
                          int sm_count, cudaStream_t stream);

// M = 1, axis 1, the gate and up projections of one SwiGLU layer (same
// geometry and codebook): h[r] = bf16(silu(bf16(gate_r)) * bf16(up_r))
cudaError_t launch_gate_up_matvec(const Packed& gate, const uint32_t* up_codes, const uint16_t* up_scales,
                                  const uint16_t* x, uint16_t* h, int sm_count, cudaStream_t stream);

// axis 1, M in 1..32, tensor cores
cudaError_t launch_prefill(const Packed& p, const uint16_t* x, int M, uint16_t* out,
                           int* status, int sm_count, cudaStream_t stream);
// The gate and up projections (same geometry, codebook of `gate`) at
// M = 1..32 in one launch: h[m][r] = bf16(silu(gate[m][r]) * up[m][r]).
cudaError_t launch_gate_up_prefill(const Packed& gate, const uint32_t* up_codes, const uint16_t* up_scales,
                                   const uint16_t* x, int M, uint16_t* h, int* status, int sm_count,
                                   cudaStream_t stream);

// axis 0: partials [M, splits, cols] then the split reduction into out [M, cols]
// out is bf16 [M, cols], or with out_f32 the unrounded f32 sums [M, cols]
cudaError_t launch_scatter(const Packed& p, const uint16_t* x, int M, int splits,
                           float* partial, float* fix, void* out, bool out_f32, int* status, int sm_count,
                           cudaStream_t stream);

// axis 0 on the tensor cores (rounded contract, 3..32 rows): partials
// [M, splits, cols] and fix-up slots fix [kScatterTcMaxCtas, M, 256], then
// the split reduction
cudaError_t launch_scatter_tc(const Packed& p, const uint16_t* x, int M, int splits, float* partial,
                              float* fix, void* out, bool out_f32, int* status, int sm_count,
                              cudaStream_t stream);

// Most CTAs of the tensor-core scatter (its fix-up space is sized for them;
// GB300 has 152 SMs).
constexpr int kScatterTcMaxCtas = 160;
// Fewest activation rows that take the tensor-core scatter, and the split
// count from which the mma.sync kernel (one CTA per split) takes over from
// the tcgen05 one.
constexpr int kScatterTcMinRows = 3;
constexpr int kScatterTcMaxSplits = 128;
// Whether a scatter call takes the tensor-core path (and its fix-up space).
inline bool scatter_uses_tc(int M, bool unrounded) { return !unrounded && M >= kScatterTcMinRows; }
// Floats of fix-up space the scatter needs besides the partials.
inline int64_t scatter_fix_floats(int M, bool unrounded) {
    return scatter_uses_tc(M, unrounded) ? (int64_t)kScatterTcMaxCtas * M * 256 : 0;
}

cudaError_t launch_rmsnorm(const uint16_t* x, int64_t M, int64_t D, float eps,
                           uint16_t* out, cudaStream_t stream);
cudaError_t launch_silu_mul(const uint16_t* g, const uint16_t* u, int64_t n,
                            uint16_t* out, cudaStream_t stream);
cudaError_t launch_round_bf16(const float* in, int64_t n, uint16_t* out, cudaStream_t stream);
cudaError_t launch_gather_probe(const float* lut, int blocks, int iters, int replicas, float* sink,
                                cudaStream_t stream);

// Largest input width the matvec kernel accepts (one 32-column unit per thread).
constexpr int64_t kMatvecMaxCols = 640 * 32;

// Split count of the scatter.  An explicit count is taken as given.  The
// default:
//   - 128 for up to 4 activation rows (scatter.ts, SCATTER_SPLITS);
//   - 128 at every M under the unrounded contract.  That contract is the one
//     of scatter.ts's balanced scatter kernels, which run SCATTER_SPLITS
//     ranges; the rule below belongs to the rounded split-K prefill.  Its
//     kernel from 3 rows runs one CTA per split, so 8 splits would leave all
//     but 8 SMs idle;
//   - otherwise, from 5 rows, the rule of the split-K launcher
//     (splitk-prefill.ts): tiles of 32 activation rows and 32 output
//     columns, 16-row K tiles, ratio = max(1, floor(K tiles / (row tiles *
//     column tiles))) and splits = min(32, max(2, the power of two at or
//     above ratio)).  At 17408 x 5120 that is 8.
// The rows of split s are [s*rp, min(rows, (s+1)*rp)) with rp =
// ceil(rows/splits) for every count.
inline int scatter_splits(int64_t rows, int64_t cols, int M, int splits, bool unrounded) {
    if (splits != 0) return splits;
    if (M <= 4 || unrounded) return 128;
    const int64_t tiles_m = (M + 31) / 32;
    const int64_t tiles_n = (cols + 31) / 32;
    const int64_t tiles_k = rows / 16;
    int64_t ratio = tiles_k / (tiles_m * tiles_n);
    if (ratio < 1) ratio = 1;
    int64_t p2 = 1;
    while (p2 < ratio) p2 <<= 1;
    return (int)(p2 < 2 ? 2 : p2 > 32 ? 32 : p2);
}

// Status codes a kernel may record in the device status word.
constexpr int kStatusWaitTimeout = 1;

// TurboQuant packed K/V decode (turboquant.cu).  Element types of the scale
// and zero arrays (the values of trellis_dtype).
constexpr int kDtF32 = 0, kDtF16 = 1, kDtBF16 = 2;
struct KvArgs {
    const uint8_t* kp;      // [rows, D*kbits/8]
    const void* ks;         // [rows, D/kg]
    const void* kz;         // [rows, D/kg]
    const uint8_t* vp;      // [rows, D*vbits/8]
    const void* vs;         // [rows, D/vg]
    const float* centroids; // [1 << vbits]
    int64_t rows;
    int D, kbits, vbits, kg, vg;
    int ks_dt, kz_dt, vs_dt;
    int v_bf16;             // values out as bf16 (else f32)
    void* k_out;            // bf16 [rows, D]
    void* v_out;            // f32 or bf16 [rows, D]
};
cudaError_t launch_kv_decode(const KvArgs& a, int sm_count, cudaStream_t stream);
// D = 256, kbits 8, vbits 3, groups of 32, bf16 values after the inverse
// rotation with signs[256].
cudaError_t launch_kv_inverse256(const KvArgs& a, const float* signs, int sm_count, cudaStream_t stream);

}  // namespace tcq
