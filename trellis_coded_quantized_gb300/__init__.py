"""GB300-native packed trellis-coded weight matmul.

Python binding of libtrellis (C ABI: include/trellis.h).  Each function has
the name of the C entry point it calls and only marshals arguments: PyTorch
CUDA tensors in, device pointers out; every step of the computation runs in
the library's CUDA kernels.  bf16 tensors may be torch.bfloat16 or int16 /
uint16 holding bf16 bit patterns.

A packed matrix is described by ``geometry(axis, rows, cols, k)``
(``interleave=2`` for the paired-block layout, ``unrounded=True`` for the
contract without the bf16 rounding of the weight):
  axis 1: rows are output features, cols input features (x [M, cols] -> [M, rows])
  axis 0: rows are input features, cols output features (x [M, rows] -> [M, cols])
codes uint32 (int32 storage) [rows, (cols/256)*256*k/32], scales bf16 [rows],
lut float32 [4096].
"""
from __future__ import annotations

import ctypes

from . import _lib

BT = 256
L = 12
DEFAULT_SPLITS = 128


class TrellisError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _lib.load().trellis_strerror(status).decode()
        super().__init__(f"{where}: {_lib.STATUS.get(status, status)}: {msg}")


FLAG_UNROUNDED = 1   # TRELLIS_FLAG_UNROUNDED: weight lut*scale kept in f32, not rounded to bf16


def geometry(axis: int, rows: int, cols: int, k: int, interleave: int = 0,
             unrounded: bool = False) -> _lib.Geometry:
    return _lib.Geometry(axis, BT, L, k, rows, cols, interleave, FLAG_UNROUNDED if unrounded else 0)


def words_per_row(cols: int, k: int) -> int:
    return (cols // BT) * (BT * k // 32)


def _check(status: int, where: str) -> None:
    if status != 0:
        raise TrellisError(status, where)


def _torch():
    import torch
    return torch


def _dev(t, name: str, dtypes, shape=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return ctypes.c_void_p(t.data_ptr())


def _bf16_types():
    torch = _torch()
    return (torch.bfloat16, torch.int16) + ((torch.uint16,) if hasattr(torch, "uint16") else ())


def _code_types():
    torch = _torch()
    return (torch.int32,) + ((torch.uint32,) if hasattr(torch, "uint32") else ())


def _stream(stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _packed(codes, scales, lut, g):
    torch = _torch()
    return (_dev(codes, "codes", _code_types(), (g.rows, words_per_row(g.cols, g.k))),
            _dev(scales, "scales", _bf16_types(), (g.rows,)),
            _dev(lut, "lut", (torch.float32,), (1 << L,)))


def _out(out, shape, like):
    torch = _torch()
    if out is None:
        out = torch.empty(shape, dtype=torch.bfloat16, device=like.device)
    return out


def trellis_matvec(x, codes, scales, lut, g, out=None, stream=None):
    """M = 1, axis 1: x bf16 [cols] (or [1, cols]) -> out bf16 [rows]."""
    c, s, t = _packed(codes, scales, lut, g)
    xp = _dev(x, "x", _bf16_types())
    if x.numel() != g.cols:
        raise ValueError("x must hold cols elements")
    out = _out(out, (g.rows,), x)
    op = _dev(out, "out", _bf16_types())
    if out.numel() != g.rows:
        raise ValueError("out must hold rows elements")
    _check(_lib.load().trellis_matvec(xp, c, s, t, ctypes.byref(g), op, _stream(stream)), "trellis_matvec")
    return out


def trellis_gate_up_matvec(x, gate_codes, gate_scales, up_codes, up_scales, lut, g, out=None, stream=None):
    """M = 1, gate and up projections of one SwiGLU layer (geometry g, one
    codebook): x bf16 [cols] -> h bf16 [rows], h = bf16(silu(gate) * up)."""
    cg, sg, t = _packed(gate_codes, gate_scales, lut, g)
    cu, su, _ = _packed(up_codes, up_scales, lut, g)
    xp = _dev(x, "x", _bf16_types())
    if x.numel() != g.cols:
        raise ValueError("x must hold cols elements")
    out = _out(out, (g.rows,), x)
    op = _dev(out, "out", _bf16_types())
    if out.numel() != g.rows:
        raise ValueError("out must hold rows elements")
    _check(_lib.load().trellis_gate_up_matvec(xp, cg, sg, cu, su, t, ctypes.byref(g), op, _stream(stream)),
           "trellis_gate_up_matvec")
    return out


def trellis_prefill(x, codes, scales, lut, g, out=None, stream=None):
    """Axis 1, 1 <= M <= 32: x bf16 [M, cols] -> out bf16 [M, rows]."""
    c, s, t = _packed(codes, scales, lut, g)
    M = x.shape[0]
    xp = _dev(x, "x", _bf16_types(), (M, g.cols))
    out = _out(out, (M, g.rows), x)
    op = _dev(out, "out", _bf16_types(), (M, g.rows))
    _check(_lib.load().trellis_prefill(xp, M, c, s, t, ctypes.byref(g), op, _stream(stream)), "trellis_prefill")
    return out


def trellis_gate_up_prefill(x, gate_codes, gate_scales, up_codes, up_scales, lut, g, out=None, stream=None):
    """Axis 1, 1 <= M <= 32, gate and up projections of one SwiGLU layer
    (geometry g, one codebook) in one launch: x bf16 [M, cols] -> h bf16
    [M, rows], h = bf16(silu(gate) * up), bit for bit two trellis_prefill
    calls and trellis_silu_mul."""
    cg, sg, t = _packed(gate_codes, gate_scales, lut, g)
    cu, su, _ = _packed(up_codes, up_scales, lut, g)
    M = x.shape[0]
    xp = _dev(x, "x", _bf16_types(), (M, g.cols))
    out = _out(out, (M, g.rows), x)
    op = _dev(out, "out", _bf16_types(), (M, g.rows))
    _check(_lib.load().trellis_gate_up_prefill(xp, M, cg, sg, cu, su, t, ctypes.byref(g), op, _stream(stream)),
           "trellis_gate_up_prefill")
    return out


DT_F32, DT_F16, DT_BF16 = 0, 1, 2      # trellis_dtype


def kv_geometry(rows: int, head_dim: int, key_bits: int, value_bits: int, key_group: int = 32,
                value_group: int = 32, key_scale_dtype: int = DT_F16, key_zero_dtype: int = DT_F16,
                value_scale_dtype: int = DT_F16, value_out_bf16: bool = False) -> _lib.KvGeometry:
    """Shape of a packed TurboQuant K/V cache of `rows` positions (B*H*N)."""
    return _lib.KvGeometry(rows, head_dim, key_bits, value_bits, key_group, value_group, key_scale_dtype,
                           key_zero_dtype, value_scale_dtype, 1 if value_out_bf16 else 0)


def _scale_types(dt):
    torch = _torch()
    return (torch.float32,) if dt == DT_F32 else (torch.float16,) if dt == DT_F16 else _bf16_types()


def _kv_inputs(key_codes, key_scales, key_zeros, value_codes, value_scales, centroids, g):
    torch = _torch()
    u8 = (torch.uint8, torch.int8)
    D = g.head_dim
    return (_dev(key_codes, "key_codes", u8, (g.rows, D * g.key_bits // 8)),
            _dev(key_scales, "key_scales", _scale_types(g.key_scale_dtype), (g.rows, D // g.key_group)),
            _dev(key_zeros, "key_zeros", _scale_types(g.key_zero_dtype), (g.rows, D // g.key_group)),
            _dev(value_codes, "value_codes", u8, (g.rows, D * g.value_bits // 8)),
            _dev(value_scales, "value_scales", _scale_types(g.value_scale_dtype), (g.rows, D // g.value_group)),
            _dev(centroids, "centroids", (torch.float32,), (1 << g.value_bits,)))


def _kv_outputs(keys_out, values_out, g, like):
    torch = _torch()
    shape = (g.rows, g.head_dim)
    if keys_out is None:
        keys_out = torch.empty(shape, dtype=torch.bfloat16, device=like.device)
    if values_out is None:
        values_out = torch.empty(shape, dtype=torch.bfloat16 if g.value_out_bf16 else torch.float32,
                                 device=like.device)
    vt = _bf16_types() if g.value_out_bf16 else (torch.float32,)
    return keys_out, values_out, _dev(keys_out, "keys_out", _bf16_types(), shape), _dev(values_out, "values_out",
                                                                                         vt, shape)


def trellis_kv_decode(key_codes, key_scales, key_zeros, value_codes, value_scales, centroids, g,
                      keys_out=None, values_out=None, stream=None):
    """TurboQuant joint K/V decode: packed [rows, D*bits/8] uint8 codes,
    per-group scales/zeros, f32 centroids -> (bf16 keys [rows, D], f32 or
    bf16 values [rows, D])."""
    ins = _kv_inputs(key_codes, key_scales, key_zeros, value_codes, value_scales, centroids, g)
    keys_out, values_out, kp, vp = _kv_outputs(keys_out, values_out, g, key_codes)
    _check(_lib.load().trellis_kv_decode(*ins, ctypes.byref(g), kp, vp, _stream(stream)), "trellis_kv_decode")
    return keys_out, values_out


def trellis_kv_decode_inverse256(key_codes, key_scales, key_zeros, value_codes, value_scales, centroids, signs, g,
                                 keys_out=None, values_out=None, stream=None):
    """The decode at D = 256, 8-bit keys, 3-bit values, groups of 32, with
    the inverse Walsh-Hadamard rotation of the values (x 1/16, x signs):
    (bf16 keys, bf16 values)."""
    torch = _torch()
    ins = _kv_inputs(key_codes, key_scales, key_zeros, value_codes, value_scales, centroids, g)
    sp = _dev(signs, "signs", (torch.float32,), (256,))
    keys_out, values_out, kp, vp = _kv_outputs(keys_out, values_out, g, key_codes)
    _check(_lib.load().trellis_kv_decode_inverse256(*ins, sp, ctypes.byref(g), kp, vp, _stream(stream)),
           "trellis_kv_decode_inverse256")
    return keys_out, values_out


def trellis_scatter_workspace_bytes(g, M: int, splits: int = 0) -> int:
    return int(_lib.load().trellis_scatter_workspace_bytes(ctypes.byref(g), M, splits))


def trellis_scatter(x, codes, scales, lut, g, splits: int = 0, workspace=None, out=None, stream=None):
    """Axis 0, 1 <= M <= 32: x bf16 [M, rows] -> out bf16 [M, cols] via fp32
    split partials in `workspace` (float32, allocated here when None)."""
    torch = _torch()
    c, s, t = _packed(codes, scales, lut, g)
    M = x.shape[0]
    xp = _dev(x, "x", _bf16_types(), (M, g.rows))
    need = trellis_scatter_workspace_bytes(g, M, splits)
    if workspace is None:
        workspace = torch.empty(max(need, 4) // 4, dtype=torch.float32, device=x.device)
    wp = _dev(workspace, "workspace", (torch.float32,))
    out = _out(out, (M, g.cols), x)
    op = _dev(out, "out", _bf16_types(), (M, g.cols))
    _check(_lib.load().trellis_scatter(xp, M, c, s, t, ctypes.byref(g), splits, wp,
                                       workspace.numel() * 4, op, _stream(stream)), "trellis_scatter")
    return out


def trellis_scatter_f32(x, codes, scales, lut, g, splits: int = 0, workspace=None, out=None, stream=None):
    """trellis_scatter with the split sums left in f32: x bf16 [M, rows] ->
    out float32 [M, cols], not rounded (to be summed with other devices'
    partial sums, then rounded by trellis_round_bf16)."""
    torch = _torch()
    c, s, t = _packed(codes, scales, lut, g)
    M = x.shape[0]
    xp = _dev(x, "x", _bf16_types(), (M, g.rows))
    need = trellis_scatter_workspace_bytes(g, M, splits)
    if workspace is None:
        workspace = torch.empty(max(need, 4) // 4, dtype=torch.float32, device=x.device)
    wp = _dev(workspace, "workspace", (torch.float32,))
    if out is None:
        out = torch.empty((M, g.cols), dtype=torch.float32, device=x.device)
    op = _dev(out, "out", (torch.float32,), (M, g.cols))
    _check(_lib.load().trellis_scatter_f32(xp, M, c, s, t, ctypes.byref(g), splits, wp,
                                           workspace.numel() * 4, op, _stream(stream)), "trellis_scatter_f32")
    return out


def trellis_round_bf16(x, out=None, stream=None):
    """float32 tensor -> bf16 tensor of the same shape, round to nearest even."""
    torch = _torch()
    xp = _dev(x, "x", (torch.float32,))
    out = _out(out, tuple(x.shape), x)
    op = _dev(out, "out", _bf16_types(), tuple(x.shape))
    _check(_lib.load().trellis_round_bf16(xp, x.numel(), op, _stream(stream)), "trellis_round_bf16")
    return out


def trellis_scatter_noalloc(x, codes, scales, lut, g, splits: int = 0, out=None, stream=None):
    """Axis 0 like trellis_scatter, for callers that cannot allocate device
    memory: the split partials live in the library's own 21 MiB device array
    (16 MiB of partials, 5 MiB of fix-up slots), so M * splits * cols may be
    at most 4,194,304.  Allocates nothing when
    `out` is given.  Calls that overlap on the GPU share that array and race."""
    c, s, t = _packed(codes, scales, lut, g)
    M = x.shape[0]
    xp = _dev(x, "x", _bf16_types(), (M, g.rows))
    out = _out(out, (M, g.cols), x)
    op = _dev(out, "out", _bf16_types(), (M, g.cols))
    _check(_lib.load().trellis_scatter_noalloc(xp, M, c, s, t, ctypes.byref(g), splits, op, _stream(stream)),
           "trellis_scatter_noalloc")
    return out


def trellis_expand(codes, scales, lut, g, w_out=None, win_out=None, with_windows=False, stream=None):
    """Decode the packed matrix: w bf16 [rows, cols] (and windows int16 [rows, cols])."""
    torch = _torch()
    c, s, t = _packed(codes, scales, lut, g)
    if w_out is None:
        w_out = torch.empty((g.rows, g.cols), dtype=torch.bfloat16, device=codes.device)
    wp = _dev(w_out, "w_out", _bf16_types(), (g.rows, g.cols))
    if win_out is None and with_windows:
        win_out = torch.empty((g.rows, g.cols), dtype=torch.int16, device=codes.device)
    vp = None if win_out is None else _dev(win_out, "win_out", _bf16_types(), (g.rows, g.cols))
    _check(_lib.load().trellis_expand(c, s, t, ctypes.byref(g), wp, vp, _stream(stream)), "trellis_expand")
    return (w_out, win_out) if win_out is not None else w_out


def trellis_rmsnorm(x, eps: float = 1e-6, out=None, stream=None):
    M, D = x.shape
    xp = _dev(x, "x", _bf16_types(), (M, D))
    out = _out(out, (M, D), x)
    op = _dev(out, "out", _bf16_types(), (M, D))
    _check(_lib.load().trellis_rmsnorm(xp, M, D, eps, op, _stream(stream)), "trellis_rmsnorm")
    return out


def trellis_silu_mul(g_, u, out=None, stream=None):
    gp = _dev(g_, "g", _bf16_types())
    up = _dev(u, "u", _bf16_types(), tuple(g_.shape))
    out = _out(out, tuple(g_.shape), g_)
    op = _dev(out, "out", _bf16_types(), tuple(g_.shape))
    _check(_lib.load().trellis_silu_mul(gp, up, g_.numel(), op, _stream(stream)), "trellis_silu_mul")
    return out


def trellis_gather_probe(lut, blocks: int, iters: int, replicas: int = 1, sink=None, stream=None):
    torch = _torch()
    lp = _dev(lut, "lut", (torch.float32,), (1 << L,))
    if sink is None:
        sink = torch.empty(blocks * 1024, dtype=torch.float32, device=lut.device)
    sp = _dev(sink, "sink", (torch.float32,), (blocks * 1024,))
    _check(_lib.load().trellis_gather_probe(lp, blocks, iters, replicas, sp, _stream(stream)),
           "trellis_gather_probe")
    return sink


def trellis_device_status() -> int:
    v = ctypes.c_int32(0)
    _check(_lib.load().trellis_device_status(ctypes.byref(v)), "trellis_device_status")
    return int(v.value)


def trellis_strerror(status: int) -> str:
    return _lib.load().trellis_strerror(status).decode()
