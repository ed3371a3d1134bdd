"""TurboQuant packed K/V decode on the GPU against the oracle
(oracle/turboquant.py), through the C ABI.

The decode arithmetic is fixed by the pages in f32 (zero added before the
scale, one multiply for the values), so keys and un-rotated values must equal
the oracle bit for bit.  The rotated values are compared with the oracle's
float64 transform within the bound derived in the oracle (half a bf16 unit
plus the f32 butterfly error).  Sizes: small and ragged row counts, every
head dim, code width, group and scale dtype, and the pages' measured regime
(B1 H4, N = 8192, D = 256, 8-bit keys, 3-bit values, f16, groups of 32).
"""
import numpy as np
import pytest
import torch

import trellis_coded_quantized_gb300 as tcq
from trellis_coded_quantized_gb300 import synth
from oracle import turboquant as tq
from conftest import has_gpu

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not has_gpu(), reason="needs a CUDA GPU")]

DT = {"f32": tcq.DT_F32, "f16": tcq.DT_F16, "bf16": tcq.DT_BF16}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from trellis_coded_quantized_gb300 import build
    build.build()


def _t(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda()
    return torch.from_numpy(a).cuda()


def _run(c, value_out_bf16, inverse=False):
    g = tcq.kv_geometry(c["rows"], c["D"], c["key_bits"], c["value_bits"], c["key_group"], c["value_group"],
                        *(DT[d] for d in c["dtypes"]), value_out_bf16=value_out_bf16)
    args = [_t(c[n]) for n in ("kp", "ks", "kz", "vp", "vs", "centroids")]
    if inverse:
        k, v = tcq.trellis_kv_decode_inverse256(*args, _t(c["signs"]), g)
    else:
        k, v = tcq.trellis_kv_decode(*args, g)
    torch.cuda.synchronize()
    kh = k.view(torch.int16).cpu().numpy().view(np.uint16)
    vh = v.view(torch.int16).cpu().numpy().view(np.uint16) if value_out_bf16 else v.cpu().numpy()
    return kh, vh


def _oracle(c):
    kdt, zdt, vdt = c["dtypes"]
    k = tq.decode_keys(c["kp"], c["ks"], c["kz"], c["key_bits"], c["D"], c["key_group"], kdt, zdt)
    v = tq.decode_values(c["vp"], c["vs"], c["centroids"], c["value_bits"], c["D"], c["value_group"], vdt)
    return k, v


@pytest.mark.parametrize("rows,D,kb,vb,kg,vg,dtypes,vbf", [
    (1, 64, 2, 2, 32, 32, ("f16", "f16", "f16"), False),
    (37, 128, 4, 3, 64, 32, ("bf16", "f32", "f16"), False),
    (300, 256, 5, 5, 32, 64, ("f32", "f32", "f32"), True),
    (129, 512, 8, 4, 64, 64, ("f16", "bf16", "bf16"), False),
    (1000, 256, 8, 3, 32, 32, ("f16", "f16", "f16"), True),
    (77, 64, 5, 8, 32, 32, ("bf16", "bf16", "f16"), True),
    (4 * 8192, 256, 8, 3, 32, 32, ("f16", "f16", "f16"), False),   # B1 H4 N8192
])
def test_kv_decode_matches_oracle(rows, D, kb, vb, kg, vg, dtypes, vbf):
    c = synth.kv_cache(rows + D + kb, rows, D, kb, vb, kg, vg, dtypes)
    k, v = _run(c, vbf)
    ko, vo = _oracle(c)
    assert np.array_equal(k, ko), f"{int((k != ko).sum())} keys differ"
    if vbf:
        assert np.array_equal(v, tq.bf16_rne(vo)), "bf16 values differ"
    else:
        assert np.array_equal(v.view(np.uint32), vo.view(np.uint32)), "f32 values differ"


@pytest.mark.parametrize("rows,dtype", [(1, "f16"), (19, "bf16"), (333, "f32"), (4 * 8192, "f16")])
def test_kv_inverse256_matches_oracle(rows, dtype):
    c = synth.kv_cache(rows + 5, rows, 256, 8, 3, 32, 32, (dtype, dtype, dtype))
    k, v = _run(c, True, inverse=True)
    ko, vo = _oracle(c)
    assert np.array_equal(k, ko)
    exact = tq.inverse_rotation(vo, c["signs"])
    bound = tq.rotation_error_bound(vo, c["signs"])
    ok = tq.rotated_within_bound(v, exact, bound)
    assert ok.all(), f"{int((~ok).sum())} rotated values outside the bound"
    # nearly all land on the rounding of the exact value
    assert (v == tq.bf16_rne(exact.astype(np.float32))).mean() > 0.99


def test_kv_errors():
    c = synth.kv_cache(3, 8, 256, 8, 3)
    args = [_t(c[n]) for n in ("kp", "ks", "kz", "vp", "vs", "centroids")]
    bad = tcq.kv_geometry(8, 256, 8, 3, value_out_bf16=False)
    with pytest.raises(tcq.TrellisError) as e:     # the inverse needs bf16 values
        tcq.trellis_kv_decode_inverse256(*args, _t(c["signs"]), bad)
    assert e.value.status == 2
    g = tcq.kv_geometry(8, 256, 6, 3)
    from trellis_coded_quantized_gb300 import _lib
    lib = _lib.load()
    import ctypes
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    kout = torch.empty((8, 256), dtype=torch.bfloat16, device="cuda")
    vout = torch.empty((8, 256), dtype=torch.float32, device="cuda")
    assert lib.trellis_kv_decode(*(P(a) for a in args), ctypes.byref(g), P(kout), P(vout), None) == 2
