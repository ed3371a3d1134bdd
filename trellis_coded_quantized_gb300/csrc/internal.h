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

// axis 0: partials [M, splits, cols] then the split reduction into out [M, cols]
cudaError_t launch_scatter(const Packed& p, const uint16_t* x, int M, int splits,
                           float* partial, uint16_t* out, int sm_count, cudaStream_t stream);

cudaError_t launch_rmsnorm(const uint16_t* x, int64_t M, int64_t D, float eps,
                           uint16_t* out, cudaStream_t stream);
cudaError_t launch_silu_mul(const uint16_t* g, const uint16_t* u, int64_t n,
                            uint16_t* out, cudaStream_t stream);
cudaError_t launch_gather_probe(const float* lut, int blocks, int iters, int replicas, float* sink,
                                cudaStream_t stream);

// Largest input width the matvec kernel accepts (one 32-column unit per thread).
constexpr int64_t kMatvecMaxCols = 640 * 32;

// Status codes a kernel may record in the device status word.
constexpr int kStatusWaitTimeout = 1;

}  // namespace tcq
