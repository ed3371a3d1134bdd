/*
 * trellis.h -- C ABI of libtrellis: the packed trellis-coded weight matmul on
 * one NVIDIA GB300 GPU (sm_103a).
 *
 * The method (pages: @mlx-bun/inference 1.0.0 diff, the kernels/trellis TypeScript files).
 * A weight matrix of `rows` x `cols` is stored only as packed codes: each row
 * is cut into blocks of BT = 256 columns, and each block is a circular
 * bitstring of BT*k bits (k = 2, 3 or 4 bits per symbol) held in
 * wpb = BT*k/32 uint32 words, least significant bit first.  Column t of a
 * block reads the L = 12-bit window that starts at bit (BT-1-t)*k and wraps
 * from the end of the block to its first word (tiled-prefill.ts, prefill tile
 * kernel).  The window indexes a 4096-entry f32 codebook, the value is
 * multiplied by the row's bf16 scale in f32 and rounded to bf16; the decoded
 * weights are contracted with bf16 activations, accumulated in fp32, and the
 * result is rounded to bf16.
 *
 * Conventions of every entry point:
 *   - All array arguments are DEVICE pointers of the current CUDA device
 *     (cudaSetDevice before the call).  bf16 arrays are IEEE bfloat16 bit
 *     patterns (uint16), row-major.  The caller owns and allocates every
 *     buffer, inputs, outputs and workspace; the library allocates no memory
 *     and keeps no pointer after the call returns.  One exception:
 *     trellis_scatter_noalloc keeps its scratch in a fixed 21 MiB device
 *     array that the library itself declares (see there).
 *   - `stream` is a cudaStream_t (NULL: the legacy default stream).  Work is
 *     only enqueued: the call never synchronises.  Results are valid once
 *     the stream has reached the work.
 *   - A call returns TRELLIS_OK when its kernels were enqueued.  Any bad
 *     argument returns an error status before anything is enqueued; no
 *     kernel traps or asserts.  Kernel-side waits are bounded: a wait that
 *     gives up records a code readable with trellis_device_status().
 *   - codes are rows*(cols/256)*wpb uint32 words in the geometry's block
 *     layout (see trellis_geometry).  scales are
 *     bf16 [rows].  lut is f32 [4096].  codes, x and lut must be 16-byte
 *     aligned; so must out and workspace of the scatter.
 */
#ifndef TRELLIS_H
#define TRELLIS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Geometry of one packed matrix (the pages' TrellisGeometry: axis, T, L, k,
 * rows, cols, blockInterleave).
 *   axis 1: rows are output features, cols are input features
 *           (out[m][r] = sum_c x[m][c] w[r][c]; tiled-prefill.ts).
 *   axis 0: rows are input features, cols are output features
 *           (out[m][c] = sum_r x[m][r] w[r][c]; scatter.ts).
 *   bt must be 256, L must be 12, k in {2, 3, 4}, rows >= 1,
 *   cols a positive multiple of 256.
 *   interleave 0: the blocks of a row are contiguous; block b of row r
 *                 starts at word (r*(cols/256) + b)*wpb.
 *   interleave 2: blocks are grouped in pairs and the pair of every row is
 *                 stored together; block b of row r starts at word
 *                 (b/2)*rows*2*wpb + r*2*wpb + (b%2)*wpb (vector-expand.ts
 *                 and scatter.ts, INTERLEAVE).  cols must then be a multiple
 *                 of 512.  Same number of words as interleave 0.
 *   flags: 0, or TRELLIS_FLAG_UNROUNDED.  Any other bit is
 *                 TRELLIS_ERR_GEOMETRY.
 */
typedef struct trellis_geometry {
    int32_t axis;
    int32_t bt;
    int32_t L;
    int32_t k;
    int64_t rows;
    int64_t cols;
    int32_t interleave;
    int32_t flags;
} trellis_geometry;

/*
 * The pages' second numerical contract (scatter.ts, the balanced scatter
 * kernels; tiled-prefill.ts names the default matvec's unrounded code value
 * as a different contract): the weight lut[win] * scale[r] enters the
 * contraction in f32 WITHOUT the bf16 rounding.  The kernels apply the scale
 * once per row -- to the row sum on axis 1, to the activation x[m][r] on
 * axis 0 -- which equals the per-weight f32 product up to f32 rounding.
 * Taken by trellis_matvec, trellis_gate_up_matvec and trellis_scatter (and
 * trellis_scatter_noalloc; from 3 activation rows the scatter's tensor-core
 * path carries each f32 weight as three bf16 terms, hi + mid + lo, which
 * keep its 24 significant bits).
 * trellis_prefill and trellis_expand return TRELLIS_ERR_GEOMETRY for it:
 * their tensor-core operands and their output are the rounded bf16 weight.
 */
#define TRELLIS_FLAG_UNROUNDED 1

typedef enum trellis_status {
    TRELLIS_OK = 0,
    TRELLIS_ERR_NULL = 1,       /* a required pointer is NULL */
    TRELLIS_ERR_GEOMETRY = 2,   /* bt, L, k, interleave, rows or cols unsupported */
    TRELLIS_ERR_SHAPE = 3,      /* M or a size out of range, or axis wrong for the call */
    TRELLIS_ERR_ALIGN = 4,      /* codes, x or workspace not 16-byte aligned */
    TRELLIS_ERR_WORKSPACE = 5,  /* workspace smaller than trellis_scatter_workspace_bytes() */
    TRELLIS_ERR_DEVICE = 6,     /* no usable device, or not compute capability 10.3 */
    TRELLIS_ERR_LAUNCH = 7      /* a kernel launch failed (cudaGetLastError) */
} trellis_status;

/*
 * M = 1 decode matvec, axis 1 (the pages' default packed matvec is named but
 * not shown; its arithmetic follows the prefill tile kernel of
 * tiled-prefill.ts and the shuffle reduction of wide-prefill.ts).
 *   x     bf16 [cols]            activations
 *   out   bf16 [rows]            out[r] = bf16( sum_c x[c] w[r][c] ), fp32 accumulation
 * Requires g->axis == 1 and cols <= 20480.
 */
trellis_status trellis_matvec(const void* x, const uint32_t* codes, const void* scales,
                              const float* lut, const trellis_geometry* g,
                              void* out, void* stream);

/*
 * The gate and up projections of one SwiGLU MLP layer at M = 1 in one
 * launch, with the SiLU gate applied on the way out (the pages' MLP input
 * is the RMSNorm output, tiled-prefill.ts; the fused chain is this
 * library's).  Both matrices have geometry g (axis 1: rows = intermediate
 * width, cols = hidden width) and share the codebook lut.
 *   x            bf16 [cols]
 *   gate_codes, up_codes, gate_scales, up_scales: the two packed matrices
 *   h_out        bf16 [rows]     h[r] = bf16( silu(gate_r) * up_r ), where
 *                gate_r = bf16( sum_c x[c] w_gate[r][c] ) and up_r likewise
 *                (exactly what trellis_matvec and trellis_silu_mul give),
 *                silu(v) = v / (1 + e^-v) in fp32
 * Requires g->axis == 1 and cols <= 20480; takes TRELLIS_FLAG_UNROUNDED.
 * Codes must be 16-byte aligned.
 */
trellis_status trellis_gate_up_matvec(const void* x, const uint32_t* gate_codes, const void* gate_scales,
                                      const uint32_t* up_codes, const void* up_scales, const float* lut,
                                      const trellis_geometry* g, void* h_out, void* stream);

/*
 * Axis-1 prefill for 1 <= M <= 32 activation rows (tiled-prefill.ts,
 * prefill tile kernel; the pages gate it to M = 5..32).  The decoded bf16
 * weight tile is contracted on the tensor cores (tcgen05, fp32 accumulation
 * in tensor memory).
 *   x     bf16 [M, cols]
 *   out   bf16 [M, rows]         out[m][r] = bf16( sum_c x[m][c] w[r][c] )
 * Requires g->axis == 1.
 */
trellis_status trellis_prefill(const void* x, int32_t M, const uint32_t* codes,
                               const void* scales, const float* lut,
                               const trellis_geometry* g, void* out, void* stream);

/*
 * The gate and up projections of one SwiGLU MLP layer at 1 <= M <= 32 in
 * one launch, with the SiLU gate applied on the way out (the pages' MLP
 * input is the RMSNorm output, tiled-prefill.ts; the fused chain is this
 * library's).  Both matrices have geometry g (axis 1: rows = intermediate
 * width, cols = hidden width) and share the codebook lut.
 *   x            bf16 [M, cols], 16-byte aligned
 *   gate_codes, up_codes (16-byte aligned), gate_scales, up_scales: the two
 *                packed matrices
 *   h_out        bf16 [M, rows]  h[m][r] = bf16( silu(gate[m][r]) * up[m][r] ),
 *                gate and up each what trellis_prefill gives, silu(v) =
 *                v / (1 + e^-v) in fp32: bit for bit trellis_prefill twice
 *                followed by trellis_silu_mul
 * Requires g->axis == 1; the rounded contract only (TRELLIS_FLAG_UNROUNDED
 * is TRELLIS_ERR_GEOMETRY, as for trellis_prefill).
 */
trellis_status trellis_gate_up_prefill(const void* x, int32_t M, const uint32_t* gate_codes,
                                       const void* gate_scales, const uint32_t* up_codes,
                                       const void* up_scales, const float* lut,
                                       const trellis_geometry* g, void* h_out, void* stream);

/*
 * Axis-0 scatter for 1 <= M <= 32 activation rows (scatter.ts: scatter
 * kernels, launch and the sum over splits).  The rows are cut into `splits`
 * ranges of rp = ceil(rows/splits) rows; range s covers
 * [s*rp, min(rows, (s+1)*rp)) and may be empty.  fp32 partial sums go to
 * workspace [M, splits, cols] and a second kernel sums them over the split
 * axis in split order and rounds to bf16.
 *   x          bf16 [M, rows], 16-byte aligned
 *   splits     1..1024, or 0 for the default: 128 when M <= 4 (scatter.ts,
 *              SCATTER_SPLITS), and 128 at every M under
 *              TRELLIS_FLAG_UNROUNDED (the contract of scatter.ts's
 *              balanced scatter kernels, which run SCATTER_SPLITS ranges;
 *              its kernel from 3 rows takes one CTA per split), else the
 *              split count of the split-K
 *              launcher (splitk-prefill.ts): with tilesM = ceil(M/32),
 *              tilesN = ceil(cols/32), tilesK = floor(rows/16) and
 *              ratio = max(1, floor(tilesK / (tilesM*tilesN))), the power of
 *              two at or above ratio, clamped to [2, 32] (8 at 17408 x 5120).
 *              Speed: the rounded contract from 3 rows with fewer than 128
 *              splits takes the tensor-core path, which spreads any split
 *              count over every SM.  Every other case (up to 2 rows, 128 or
 *              more splits, the unrounded contract) runs one CTA per split
 *              (up to 2 rows: per split and 5120 columns), so fewer splits
 *              than SMs leave SMs idle.
 *   workspace  f32, at least trellis_scatter_workspace_bytes(g, M, splits) bytes,
 *              16-byte aligned; contents on entry do not matter.  On return
 *              it holds the partials P[m][s][c] (empty ranges hold zeros).
 *   out        bf16 [M, cols], 16-byte aligned
 *              out[m][c] = bf16( sum_r x[m][r] w[r][c] )
 * Requires g->axis == 0.
 */
trellis_status trellis_scatter(const void* x, int32_t M, const uint32_t* codes,
                               const void* scales, const float* lut,
                               const trellis_geometry* g, int32_t splits,
                               float* workspace, size_t workspace_bytes,
                               void* out, void* stream);

/*
 * trellis_scatter with the split sums left unrounded: out is f32 [M, cols],
 * out[m][c] = sum over the splits of P[m][s][c], in the same order as
 * trellis_scatter, which rounds exactly this value to bf16.  For a caller
 * that still adds other partial sums before the rounding -- the rows of the
 * same matrix held by other GPUs (the split-K sum over splits of scatter.ts
 * and splitk-prefill.ts, continued across devices): all-reduce the f32
 * outputs, then trellis_round_bf16.  Same arguments, rules and workspace as
 * trellis_scatter; out must be 16-byte aligned.
 */
trellis_status trellis_scatter_f32(const void* x, int32_t M, const uint32_t* codes,
                                   const void* scales, const float* lut,
                                   const trellis_geometry* g, int32_t splits,
                                   float* workspace, size_t workspace_bytes,
                                   float* out, void* stream);

/*
 * out[i] = bf16( in[i] ), round to nearest even: the output rounding of the
 * packed matmul (tiled-prefill.ts and scatter.ts, the final cast to T), for
 * sums finished outside the library.  in f32 [n], out bf16 [n], n >= 1.
 */
trellis_status trellis_round_bf16(const float* in, int64_t n, void* out, void* stream);

/*
 * trellis_scatter without a caller-provided workspace.  The pages have no
 * counterpart: this exists for callers that cannot allocate device memory,
 * such as plugin interfaces that pass in only input and output buffers, or
 * serving loops that must not call cudaMalloc because it can synchronise the
 * device.  Same arguments and result as trellis_scatter minus the workspace;
 * the fp32 split partials (and the fix-up slots of the tensor-core path) go
 * to a 21 MiB array of device memory that the library declares itself: 16
 * MiB of partials and 5 MiB of fix-up space (reserved on every GPU that
 * uses it until the process exits).
 *   - x and out must be 16-byte aligned, as for trellis_scatter;
 *   - M * splits * cols must be at most 4,194,304 (splits 0 is resolved as
 *     for trellis_scatter), else TRELLIS_ERR_WORKSPACE and nothing is
 *     enqueued;
 *   - allocates nothing; the first call on a device looks up the array's
 *     device address (cudaGetSymbolAddress).  With CUDA's lazy module
 *     loading the driver reserves the array when the library's scatter code
 *     is first used on that device -- the first trellis_scatter or
 *     trellis_scatter_noalloc call -- and that first use may synchronise.
 *     So make one such call on each device before any stream capture or any
 *     region where device allocation is not allowed;
 *   - all calls share the one array: calls that overlap on the GPU (other
 *     streams, other host threads) race and must be serialised by the caller.
 */
trellis_status trellis_scatter_noalloc(const void* x, int32_t M, const uint32_t* codes,
                                       const void* scales, const float* lut,
                                       const trellis_geometry* g, int32_t splits,
                                       void* out, void* stream);

/*
 * Bytes of workspace trellis_scatter needs, with splits 0 resolved as
 * trellis_scatter does; 0 for invalid arguments:
 *   - the fp32 partials [M, splits, cols] of the scatter launch (scatter.ts,
 *     the [M, SPLITS, C] float partial output): M * splits * cols * 4;
 *   - from 3 activation rows under the rounded contract (the tensor-core
 *     path), after them, fix-up slots for the split reduction: 160 * M * 256
 *     floats, M * 163840 bytes.  Its CTAs take equal runs of 16-row K steps
 *     across the splits; a CTA that starts inside a split leaves its share of
 *     that split's partial in its slot.
 */
size_t trellis_scatter_workspace_bytes(const trellis_geometry* g, int32_t M, int32_t splits);

/*
 * Verification export: decode the whole matrix (vector-expand.ts, expand
 * kernel).  Never needed on the matmul path.
 *   w_out    bf16 [rows, cols]    w[r][c] = bf16( f32( lut[win] * scale[r] ) )
 *   win_out  uint16 [rows, cols]  the window of each weight; may be NULL
 * Either axis.
 */
trellis_status trellis_expand(const uint32_t* codes, const void* scales, const float* lut,
                              const trellis_geometry* g, void* w_out, uint16_t* win_out,
                              void* stream);

/*
 * Glue of a SwiGLU MLP layer built from the packed matmuls (not a step of
 * the method; the pages only say the prefill input is the RMSNorm output).
 *   trellis_rmsnorm:  out[m][d] = bf16( x[m][d] / sqrt(mean_d x[m][d]^2 + eps) ),
 *                     unit gain, fp32 arithmetic; x, out bf16 [M, D], D <= 65536.
 *   trellis_silu_mul: out[i] = bf16( silu(g[i]) * u[i] ), fp32 arithmetic;
 *                     g, u, out bf16 [n].
 */
trellis_status trellis_rmsnorm(const void* x, int64_t M, int64_t D, float eps,
                               void* out, void* stream);
trellis_status trellis_silu_mul(const void* g, const void* u, int64_t n,
                                void* out, void* stream);

/*
 * TurboQuant packed K/V cache decode (@mlx-bun/inference 1.0.0,
 * kernels/turboquant/decode.ts, joint K/V decode kernel; inverse.ts, the
 * decode with the inverse 256-point rotation).  A second packed-decode
 * workload beside the trellis matmul; it shares no code path with it.
 *
 * The cache is `rows` positions (B * H * N of the pages' [B, H, N, D]
 * arrays), every array row-major and contiguous:
 *   key_codes     u8  [rows, D*key_bits/8]   code of column c at bit offset
 *                 c*key_bits of the row's bytes, low bits first, reaching
 *                 into the next byte when it straddles two; an 8-bit code is
 *                 a signed byte (int8)
 *   key_scales, key_zeros   [rows, D/key_group] of their trellis_dtype
 *   value_codes   u8  [rows, D*value_bits/8]  same bit layout, unsigned
 *   value_scales  [rows, D/value_group] of its trellis_dtype
 *   centroids     f32 [1 << value_bits]
 *   keys_out      bf16 [rows, D]   bf16( (f32(code) + f32(zero)) * f32(scale) ),
 *                 the zero added before scaling, both in f32
 *   values_out    f32 or bf16 [rows, D]   f32(centroids[code]) * f32(scale),
 *                 rounded to bf16 when value_out_bf16 (the pages' deferred
 *                 rotation)
 * key_codes, value_codes, keys_out and values_out must be 16-byte aligned;
 * scales and zeros aligned to their element; the codes and scales are read
 * after the previous kernel of the stream completed, the centroids (and the
 * signs below) before -- they are constant tables.
 */
typedef enum trellis_dtype {
    TRELLIS_DT_F32 = 0,
    TRELLIS_DT_F16 = 1,
    TRELLIS_DT_BF16 = 2
} trellis_dtype;

typedef struct trellis_kv_geometry {
    int64_t rows;                /* >= 1 */
    int32_t head_dim;            /* D: 64, 128, 256 or 512 */
    int32_t key_bits;            /* 2, 4, 5 or 8 */
    int32_t value_bits;          /* 2, 3, 4, 5 or 8 */
    int32_t key_group;           /* columns per key scale and zero: 32 or 64 */
    int32_t value_group;         /* columns per value scale: 32 or 64 */
    int32_t key_scale_dtype;     /* trellis_dtype */
    int32_t key_zero_dtype;      /* trellis_dtype */
    int32_t value_scale_dtype;   /* trellis_dtype */
    int32_t value_out_bf16;      /* 0: f32 values, 1: bf16 values */
} trellis_kv_geometry;

/* Joint decode of keys and values.  A field outside the sets above is
 * TRELLIS_ERR_GEOMETRY. */
trellis_status trellis_kv_decode(const uint8_t* key_codes, const void* key_scales, const void* key_zeros,
                                 const uint8_t* value_codes, const void* value_scales, const float* centroids,
                                 const trellis_kv_geometry* g, void* keys_out, void* values_out, void* stream);

/* The decode followed by the inverse rotation of every value row: with v
 * the decoded f32 values of a row, values_out[c] =
 * bf16( (H v)[c] * (1/16) * signs[c] ), H the 256-point Walsh-Hadamard
 * matrix ((-1)^popcount(c & j)), computed by butterflies over the column
 * bits 0..7 in that order (each a + b, a - b in f32, as the page's two
 * radix-16 passes).  Requires head_dim 256, key_bits 8, value_bits 3, both
 * groups 32 and value_out_bf16 = 1 (the pages' regime; any scale dtype is
 * taken).  signs: f32 [256]. */
trellis_status trellis_kv_decode_inverse256(const uint8_t* key_codes, const void* key_scales, const void* key_zeros,
                                            const uint8_t* value_codes, const void* value_scales,
                                            const float* centroids, const float* signs,
                                            const trellis_kv_geometry* g, void* keys_out, void* values_out,
                                            void* stream);

/*
 * Measurement aid: `iters` rounds of 8 random 4-byte gathers per thread from
 * a 4096-entry f32 table held in shared memory, on `blocks` CTAs of 1024
 * threads; one float per thread goes to sink (f32 [blocks*1024]) so nothing
 * is optimised away.  Timed with events it gives the shared-memory gather
 * rate that bounds the decode.  replicas 1: one table; 4 or 8: copies of the
 * table interleaved so that lane group lane % replicas reads only its own
 * banks (entry e of copy g at word replicas*e + g).
 */
trellis_status trellis_gather_probe(const float* lut, int32_t blocks, int32_t iters, int32_t replicas,
                                    float* sink, void* stream);

/*
 * Device-side status of the last kernels on the current device: 0 when no
 * bounded wait gave up.  Copies one word with cudaMemcpy (synchronising the
 * device) into *status and clears it.  Returns TRELLIS_ERR_NULL or
 * TRELLIS_ERR_DEVICE on failure.
 */
trellis_status trellis_device_status(int32_t* status);

/*
 * Static English text for a status; never NULL.  The pages report an
 * unsupported geometry by throwing with a message (tiled-prefill.ts and
 * splitk-prefill.ts, launchers); this library returns the status and this
 * text describes it.
 */
const char* trellis_strerror(trellis_status status);

#ifdef __cplusplus
}
#endif

#endif /* TRELLIS_H */
