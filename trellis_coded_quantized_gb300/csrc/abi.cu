// The C ABI of libtrellis: argument validation (before anything is enqueued),
// per-device facts, and dispatch to the launchers.  See include/trellis.h for
// the contract of every entry point.
#include "trellis.h"
#include "internal.h"

#include <climits>
#include <initializer_list>
#include <mutex>

namespace {

__device__ int g_device_status;   // recorded by kernels whose bounded waits gave up

constexpr int kMaxDevices = 64;

struct DeviceFacts {
    trellis_status st;   // TRELLIS_OK when the device is usable
    int sm_count;
    int* status;         // device address of g_device_status on this device
};

DeviceFacts g_facts[kMaxDevices];
std::once_flag g_once[kMaxDevices];

trellis_status current_device(const DeviceFacts** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return TRELLIS_ERR_DEVICE;
    }
    std::call_once(g_once[dev], [dev]() {
        DeviceFacts f{TRELLIS_ERR_DEVICE, 0, nullptr};
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, dev) == cudaSuccess && prop.major == 10 && prop.minor == 3) {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_device_status) == cudaSuccess) {
                f.st = TRELLIS_OK;
                f.sm_count = prop.multiProcessorCount;
                f.status = static_cast<int*>(p);
            }
        }
        cudaGetLastError();
        g_facts[dev] = f;
    });
    *out = &g_facts[dev];
    return g_facts[dev].st;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// axis: the axis the call requires (-1: either); unrounded_ok: whether the
// call takes TRELLIS_FLAG_UNROUNDED
trellis_status check_geometry(const trellis_geometry* g, int axis, bool unrounded_ok) {
    if (!g) return TRELLIS_ERR_NULL;
    if ((g->flags & ~TRELLIS_FLAG_UNROUNDED) != 0) return TRELLIS_ERR_GEOMETRY;
    if ((g->flags & TRELLIS_FLAG_UNROUNDED) && !unrounded_ok) return TRELLIS_ERR_GEOMETRY;
    if (g->bt != 256 || g->L != 12 || g->k < 2 || g->k > 4 || (g->interleave != 0 && g->interleave != 2))
        return TRELLIS_ERR_GEOMETRY;
    if (g->axis != 0 && g->axis != 1) return TRELLIS_ERR_GEOMETRY;
    if (g->rows < 1 || g->rows > INT_MAX / 2 || g->cols < 256 || g->cols % 256 != 0 ||
        g->cols > INT_MAX / 2)
        return TRELLIS_ERR_GEOMETRY;
    if (g->interleave == 2 && (g->cols / 256) % 2 != 0) return TRELLIS_ERR_GEOMETRY;
    if (axis >= 0 && g->axis != axis) return TRELLIS_ERR_SHAPE;
    return TRELLIS_OK;
}

tcq::Packed packed(const uint32_t* codes, const void* scales, const float* lut,
                   const trellis_geometry* g) {
    return tcq::Packed{codes, static_cast<const uint16_t*>(scales), lut, g->rows, g->cols, g->k, g->interleave,
                       (g->flags & TRELLIS_FLAG_UNROUNDED) != 0};
}

trellis_status launched(cudaError_t e) {
    if (e != cudaSuccess) {
        cudaGetLastError();
        return TRELLIS_ERR_LAUNCH;
    }
    return TRELLIS_OK;
}

// The checks and the launch shared by trellis_scatter and trellis_scatter_f32.
trellis_status scatter_common(const void* x, int32_t M, const uint32_t* codes, const void* scales,
                              const float* lut, const trellis_geometry* g, int32_t splits, float* workspace,
                              size_t workspace_bytes, void* out, bool out_f32, void* stream) {
    if (!x || !codes || !scales || !lut || !g || !out || !workspace) return TRELLIS_ERR_NULL;
    trellis_status st = check_geometry(g, 0, true);
    if (st != TRELLIS_OK) return st;
    if (M < 1 || M > 32 || splits < 0 || splits > 1024) return TRELLIS_ERR_SHAPE;
    const int s = tcq::scatter_splits(g->rows, g->cols, M, splits, (g->flags & TRELLIS_FLAG_UNROUNDED) != 0);
    if (!aligned16(x) || !aligned16(codes) || !aligned16(lut) || !aligned16(workspace) ||
        !aligned16(out))
        return TRELLIS_ERR_ALIGN;
    if (workspace_bytes < trellis_scatter_workspace_bytes(g, M, splits)) return TRELLIS_ERR_WORKSPACE;
    const DeviceFacts* d;
    if ((st = current_device(&d)) != TRELLIS_OK) return st;
    // the fix-up slots of the tensor-core path follow the partials
    float* fix = workspace + (int64_t)M * s * g->cols;
    return launched(tcq::launch_scatter(packed(codes, scales, lut, g), static_cast<const uint16_t*>(x), M, s,
                                        workspace, fix, out, out_f32, d->status, d->sm_count,
                                        static_cast<cudaStream_t>(stream)));
}

bool one_of(int v, std::initializer_list<int> set) {
    for (int x : set)
        if (v == x) return true;
    return false;
}
bool aligned_to(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
size_t dt_size(int dt) { return dt == tcq::kDtF32 ? 4 : 2; }

trellis_status check_kv(const uint8_t* kp, const void* ks, const void* kz, const uint8_t* vp, const void* vs,
                        const float* centroids, const trellis_kv_geometry* g, void* k_out, void* v_out) {
    if (!kp || !ks || !kz || !vp || !vs || !centroids || !g || !k_out || !v_out) return TRELLIS_ERR_NULL;
    if (g->rows < 1 || !one_of(g->head_dim, {64, 128, 256, 512}) || !one_of(g->key_bits, {2, 4, 5, 8}) ||
        !one_of(g->value_bits, {2, 3, 4, 5, 8}) || !one_of(g->key_group, {32, 64}) ||
        !one_of(g->value_group, {32, 64}) || !one_of(g->key_scale_dtype, {0, 1, 2}) ||
        !one_of(g->key_zero_dtype, {0, 1, 2}) || !one_of(g->value_scale_dtype, {0, 1, 2}) ||
        !one_of(g->value_out_bf16, {0, 1}) || g->rows > ((int64_t)1 << 40) / g->head_dim)
        return TRELLIS_ERR_GEOMETRY;
    if (!aligned16(kp) || !aligned16(vp) || !aligned16(k_out) || !aligned16(v_out) || !aligned_to(centroids, 4) ||
        !aligned_to(ks, dt_size(g->key_scale_dtype)) || !aligned_to(kz, dt_size(g->key_zero_dtype)) ||
        !aligned_to(vs, dt_size(g->value_scale_dtype)))
        return TRELLIS_ERR_ALIGN;
    return TRELLIS_OK;
}

tcq::KvArgs kv_args(const uint8_t* kp, const void* ks, const void* kz, const uint8_t* vp, const void* vs,
                    const float* centroids, const trellis_kv_geometry* g, void* k_out, void* v_out) {
    return tcq::KvArgs{kp, ks, kz, vp, vs, centroids, g->rows, g->head_dim, g->key_bits, g->value_bits,
                       g->key_group, g->value_group, g->key_scale_dtype, g->key_zero_dtype, g->value_scale_dtype,
                       g->value_out_bf16, k_out, v_out};
}
}  // namespace

extern "C" {

trellis_status trellis_matvec(const void* x, const uint32_t* codes, const void* scales,
                              const float* lut, const trellis_geometry* g,
                              void* out, void* stream) {
    if (!x || !codes || !scales || !lut || !g || !out) return TRELLIS_ERR_NULL;
    trellis_status st = check_geometry(g, 1, true);
    if (st != TRELLIS_OK) return st;
    if (g->cols > tcq::kMatvecMaxCols) return TRELLIS_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(codes) || !aligned16(lut)) return TRELLIS_ERR_ALIGN;
    const DeviceFacts* d;
    if ((st = current_device(&d)) != TRELLIS_OK) return st;
    return launched(tcq::launch_matvec(packed(codes, scales, lut, g), static_cast<const uint16_t*>(x),
                                       static_cast<uint16_t*>(out), d->sm_count,
                                       static_cast<cudaStream_t>(stream)));
}

trellis_status trellis_gate_up_matvec(const void* x, const uint32_t* gate_codes, const void* gate_scales,
                                     const uint32_t* up_codes, const void* up_scales, const float* lut,
                                     const trellis_geometry* g, void* h_out, void* stream) {
    if (!x || !gate_codes || !gate_scales || !up_codes || !up_scales || !lut || !g || !h_out)
        return TRELLIS_ERR_NULL;
    trellis_status st = check_geometry(g, 1, true);
    if (st != TRELLIS_OK) return st;
    if (g->cols > tcq::kMatvecMaxCols) return TRELLIS_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(gate_codes) || !aligned16(up_codes) || !aligned16(lut)) return TRELLIS_ERR_ALIGN;
    const DeviceFacts* d;
    if ((st = current_device(&d)) != TRELLIS_OK) return st;
    return launched(tcq::launch_gate_up_matvec(packed(gate_codes, gate_scales, lut, g), up_codes,
                                               static_cast<const uint16_t*>(up_scales),
                                               static_cast<const uint16_t*>(x), static_cast<uint16_t*>(h_out),
                                               d->sm_count, static_cast<cudaStream_t>(stream)));
}

trellis_status trellis_prefill(const void* x, int32_t M, const uint32_t* codes,
                               const void* scales, const float* lut,
                               const trellis_geometry* g, void* out, void* stream) {
    if (!x || !codes || !scales || !lut || !g || !out) return TRELLIS_ERR_NULL;
    trellis_status st = check_geometry(g, 1, false);
    if (st != TRELLIS_OK) return st;
    if (M < 1 || M > 32) return TRELLIS_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(codes) || !aligned16(lut)) return TRELLIS_ERR_ALIGN;
    const DeviceFacts* d;
    if ((st = current_device(&d)) != TRELLIS_OK) return st;
    return launched(tcq::launch_prefill(packed(codes, scales, lut, g), static_cast<const uint16_t*>(x), M,
                                        static_cast<uint16_t*>(out), d->status, d->sm_count,
                                        static_cast<cudaStream_t>(stream)));
}

trellis_status trellis_gate_up_prefill(const void* x, int32_t M, const uint32_t* gate_codes,
                                      const void* gate_scales, const uint32_t* up_codes, const void* up_scales,
                                      const float* lut, const trellis_geometry* g, void* h_out, void* stream) {
    if (!x || !gate_codes || !gate_scales || !up_codes || !up_scales || !lut || !g || !h_out)
        return TRELLIS_ERR_NULL;
    trellis_status st = check_geometry(g, 1, false);
    if (st != TRELLIS_OK) return st;
    if (M < 1 || M > 32) return TRELLIS_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(gate_codes) || !aligned16(up_codes) || !aligned16(lut)) return TRELLIS_ERR_ALIGN;
    const DeviceFacts* d;
    if ((st = current_device(&d)) != TRELLIS_OK) return st;
    return launched(tcq::launch_gate_up_prefill(packed(gate_codes, gate_scales, lut, g), up_codes,
                                                static_cast<const uint16_t*>(up_scales),
                                                static_cast<const uint16_t*>(x), M, static_cast<uint16_t*>(h_out),
                                                d->status, d->sm_count, static_cast<cudaStream_t>(stream)));
}

trellis_status trellis_kv_decode(const uint8_t* key_codes, const void* key_scales, const void* key_zeros,
                                 const uint8_t* value_codes, const void* value_scales, const float* centroids,
                                 const trellis_kv_geometry* g, void* keys_out, void* values_out, void* stream) {
    trellis_status st = check_kv(key_codes, key_scales, key_zeros, value_codes, value_scales, centroids, g,
                                 keys_out, values_out);
    if (st != TRELLIS_OK) return st;
    const DeviceFacts* d;
    if ((st = current_device(&d)) != TRELLIS_OK) return st;
    return launched(tcq::launch_kv_decode(kv_args(key_codes, key_scales, key_zeros, value_codes, value_scales,
                                                  centroids, g, keys_out, values_out),
                                          d->sm_count, static_cast<cudaStream_t>(stream)));
}

trellis_status trellis_kv_decode_inverse256(const uint8_t* key_codes, const void* key_scales, const void* key_zeros,
                                            const uint8_t* value_codes, const void* value_scales,
                                            const float* centroids, const float* signs,
                                            const trellis_kv_geometry* g, void* keys_out, void* values_out,
                                            void* stream) {
    if (!signs) return TRELLIS_ERR_NULL;
    trellis_status st = check_kv(key_codes, key_scales, key_zeros, value_codes, value_scales, centroids, g,
                                 keys_out, values_out);
    if (st != TRELLIS_OK) return st;
    if (g->head_dim != 256 || g->key_bits != 8 || g->value_bits != 3 || g->key_group != 32 ||
        g->value_group != 32 || g->value_out_bf16 != 1)
        return TRELLIS_ERR_GEOMETRY;
    if (!aligned_to(signs, 4)) return TRELLIS_ERR_ALIGN;
    const DeviceFacts* d;
    if ((st = current_device(&d)) != TRELLIS_OK) return st;
    return launched(tcq::launch_kv_inverse256(kv_args(key_codes, key_scales, key_zeros, value_codes, value_scales,
                                                      centroids, g, keys_out, values_out),
                                              signs, d->sm_count, static_cast<cudaStream_t>(stream)));
}

size_t trellis_scatter_workspace_bytes(const trellis_geometry* g, int32_t M, int32_t splits) {
    if (check_geometry(g, -1, true) != TRELLIS_OK || M < 1 || M > 32 || splits < 0 || splits > 1024) return 0;
    const bool unr = (g->flags & TRELLIS_FLAG_UNROUNDED) != 0;
    return ((size_t)M * (size_t)tcq::scatter_splits(g->rows, g->cols, M, splits, unr) * (size_t)g->cols +
            (size_t)tcq::scatter_fix_floats(M, unr)) * sizeof(float);
}

trellis_status trellis_scatter(const void* x, int32_t M, const uint32_t* codes,
                               const void* scales, const float* lut,
                               const trellis_geometry* g, int32_t splits,
                               float* workspace, size_t workspace_bytes,
                               void* out, void* stream) {
    return scatter_common(x, M, codes, scales, lut, g, splits, workspace, workspace_bytes, out, false, stream);
}

trellis_status trellis_scatter_f32(const void* x, int32_t M, const uint32_t* codes,
                                   const void* scales, const float* lut,
                                   const trellis_geometry* g, int32_t splits,
                                   float* workspace, size_t workspace_bytes,
                                   float* out, void* stream) {
    return scatter_common(x, M, codes, scales, lut, g, splits, workspace, workspace_bytes, out, true, stream);
}

trellis_status trellis_round_bf16(const float* in, int64_t n, void* out, void* stream) {
    if (!in || !out) return TRELLIS_ERR_NULL;
    if (n < 1) return TRELLIS_ERR_SHAPE;
    const DeviceFacts* d;
    trellis_status st;
    if ((st = current_device(&d)) != TRELLIS_OK) return st;
    return launched(tcq::launch_round_bf16(in, n, static_cast<uint16_t*>(out), static_cast<cudaStream_t>(stream)));
}

trellis_status trellis_expand(const uint32_t* codes, const void* scales, const float* lut,
                              const trellis_geometry* g, void* w_out, uint16_t* win_out,
                              void* stream) {
    if (!codes || !scales || !lut || !g || !w_out) return TRELLIS_ERR_NULL;
    trellis_status st = check_geometry(g, -1, false);
    if (st != TRELLIS_OK) return st;
    if (!aligned16(codes) || !aligned16(lut) || !aligned16(w_out) || (win_out && !aligned16(win_out)))
        return TRELLIS_ERR_ALIGN;
    const DeviceFacts* d;
    if ((st = current_device(&d)) != TRELLIS_OK) return st;
    return launched(tcq::launch_expand(packed(codes, scales, lut, g), static_cast<uint16_t*>(w_out), win_out,
                                       d->sm_count, static_cast<cudaStream_t>(stream)));
}

trellis_status trellis_rmsnorm(const void* x, int64_t M, int64_t D, float eps,
                               void* out, void* stream) {
    if (!x || !out) return TRELLIS_ERR_NULL;
    if (M < 1 || M > INT_MAX || D < 1 || D > 65536 || !(eps >= 0.0f)) return TRELLIS_ERR_SHAPE;
    const DeviceFacts* d;
    trellis_status st;
    if ((st = current_device(&d)) != TRELLIS_OK) return st;
    return launched(tcq::launch_rmsnorm(static_cast<const uint16_t*>(x), M, D, eps,
                                        static_cast<uint16_t*>(out), static_cast<cudaStream_t>(stream)));
}

trellis_status trellis_silu_mul(const void* g, const void* u, int64_t n, void* out, void* stream) {
    if (!g || !u || !out) return TRELLIS_ERR_NULL;
    if (n < 1) return TRELLIS_ERR_SHAPE;
    const DeviceFacts* d;
    trellis_status st;
    if ((st = current_device(&d)) != TRELLIS_OK) return st;
    return launched(tcq::launch_silu_mul(static_cast<const uint16_t*>(g), static_cast<const uint16_t*>(u), n,
                                         static_cast<uint16_t*>(out), static_cast<cudaStream_t>(stream)));
}

trellis_status trellis_gather_probe(const float* lut, int32_t blocks, int32_t iters, int32_t replicas,
                                    float* sink, void* stream) {
    if (!lut || !sink) return TRELLIS_ERR_NULL;
    if (blocks < 1 || blocks > 65536 || iters < 1) return TRELLIS_ERR_SHAPE;
    if (replicas != 1 && replicas != 4 && replicas != 8) return TRELLIS_ERR_SHAPE;
    if (!aligned16(lut)) return TRELLIS_ERR_ALIGN;
    const DeviceFacts* d;
    trellis_status st;
    if ((st = current_device(&d)) != TRELLIS_OK) return st;
    return launched(tcq::launch_gather_probe(lut, blocks, iters, replicas, sink, static_cast<cudaStream_t>(stream)));
}

trellis_status trellis_device_status(int32_t* status) {
    if (!status) return TRELLIS_ERR_NULL;
    const DeviceFacts* d;
    trellis_status st;
    if ((st = current_device(&d)) != TRELLIS_OK) return st;
    int v = 0;
    const int zero = 0;
    if (cudaMemcpy(&v, d->status, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(d->status, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaGetLastError();
        return TRELLIS_ERR_DEVICE;
    }
    *status = v;
    return TRELLIS_OK;
}

const char* trellis_strerror(trellis_status status) {
    switch (status) {
        case TRELLIS_OK: return "ok";
        case TRELLIS_ERR_NULL: return "a required pointer is NULL";
        case TRELLIS_ERR_GEOMETRY: return "unsupported geometry (bt must be 256, L 12, k 2..4, interleave 0 or 2, cols a multiple of 256 (512 for interleave 2), flags 0 or TRELLIS_FLAG_UNROUNDED where the call takes it)";
        case TRELLIS_ERR_SHAPE: return "size out of range or axis wrong for this entry point";
        case TRELLIS_ERR_ALIGN: return "a buffer is not 16-byte aligned";
        case TRELLIS_ERR_WORKSPACE: return "workspace smaller than trellis_scatter_workspace_bytes()";
        case TRELLIS_ERR_DEVICE: return "no usable CUDA device of compute capability 10.3";
        case TRELLIS_ERR_LAUNCH: return "a kernel launch failed";
    }
    return "unknown trellis status";
}

}  // extern "C"
