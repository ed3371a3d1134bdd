"""ctypes view of libtrellis (include/trellis.h).  Loading fails loudly: there
is no fallback implementation of any entry point."""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libtrellis.so")

# the entry points declared in include/trellis.h
EXPORTS = (
    "trellis_matvec", "trellis_gate_up_matvec", "trellis_prefill", "trellis_gate_up_prefill", "trellis_scatter", "trellis_scatter_f32",
    "trellis_round_bf16", "trellis_scatter_noalloc",
    "trellis_scatter_workspace_bytes",
    "trellis_expand", "trellis_rmsnorm", "trellis_silu_mul", "trellis_kv_decode", "trellis_kv_decode_inverse256",
    "trellis_gather_probe",
    "trellis_device_status", "trellis_strerror",
)

STATUS = {
    0: "TRELLIS_OK", 1: "TRELLIS_ERR_NULL", 2: "TRELLIS_ERR_GEOMETRY", 3: "TRELLIS_ERR_SHAPE",
    4: "TRELLIS_ERR_ALIGN", 5: "TRELLIS_ERR_WORKSPACE", 6: "TRELLIS_ERR_DEVICE", 7: "TRELLIS_ERR_LAUNCH",
}


class Geometry(ctypes.Structure):
    _fields_ = [("axis", ctypes.c_int32), ("bt", ctypes.c_int32), ("L", ctypes.c_int32),
                ("k", ctypes.c_int32), ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                ("interleave", ctypes.c_int32), ("flags", ctypes.c_int32)]


class KvGeometry(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_int64), ("head_dim", ctypes.c_int32), ("key_bits", ctypes.c_int32),
                ("value_bits", ctypes.c_int32), ("key_group", ctypes.c_int32), ("value_group", ctypes.c_int32),
                ("key_scale_dtype", ctypes.c_int32), ("key_zero_dtype", ctypes.c_int32),
                ("value_scale_dtype", ctypes.c_int32), ("value_out_bf16", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


def bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    """Declare the C signatures of the entry points on a loaded library."""
    P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    G = ctypes.POINTER(Geometry)
    KG = ctypes.POINTER(KvGeometry)
    sig = {
        "trellis_matvec": ([P, P, P, P, G, P, P], I32),
        "trellis_gate_up_matvec": ([P, P, P, P, P, P, G, P, P], I32),
        "trellis_prefill": ([P, I32, P, P, P, G, P, P], I32),
        "trellis_gate_up_prefill": ([P, I32, P, P, P, P, P, G, P, P], I32),
        "trellis_scatter": ([P, I32, P, P, P, G, I32, P, SZ, P, P], I32),
        "trellis_scatter_f32": ([P, I32, P, P, P, G, I32, P, SZ, P, P], I32),
        "trellis_round_bf16": ([P, I64, P, P], I32),
        "trellis_scatter_noalloc": ([P, I32, P, P, P, G, I32, P, P], I32),
        "trellis_scatter_workspace_bytes": ([G, I32, I32], SZ),
        "trellis_expand": ([P, P, P, G, P, P, P], I32),
        "trellis_rmsnorm": ([P, I64, I64, ctypes.c_float, P, P], I32),
        "trellis_silu_mul": ([P, P, I64, P, P], I32),
        "trellis_kv_decode": ([P, P, P, P, P, P, KG, P, P, P], I32),
        "trellis_kv_decode_inverse256": ([P, P, P, P, P, P, P, KG, P, P, P], I32),
        "trellis_gather_probe": ([P, I32, I32, I32, P, P], I32),
        "trellis_device_status": ([ctypes.POINTER(I32)], I32),
        "trellis_strerror": ([I32], ctypes.c_char_p),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    return lib


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libtrellis.so and declare its signatures; raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise ImportError(f"libtrellis is not built ({path} missing): run __graft_entry__.build()")
        _lib = bind(ctypes.CDLL(path))
        return _lib
