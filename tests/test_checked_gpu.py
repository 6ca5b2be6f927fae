"""The bounds-checked build (libqdecode_attn_checked.so, compiled with QDA_BOUNDS_CHECK) on awkward shapes.

In that build every copy range, stage offset, query row and partial slot the split and merge kernels compute is
checked before use; a failed check sets bit 4 of the device status and skips the access (no trap). The cases below
(ragged and one-row sequences, forced split counts up to one range per 8 rows, multi-query and compat calls, every
head dimension) must leave the status clean and still match the oracle."""
import ctypes

import numpy as np
import pytest
import torch

import oracle as O
import attention_quantized_kv_split_gb300 as qda
from attention_quantized_kv_split_gb300 import _lib, build, synth

from harness import TOL, TORCH_DT, small_case, upload_cache

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    handle = ctypes.CDLL(build.build(checked=True))
    for name, (res, args) in _lib.SIGNATURES.items():
        fn = getattr(handle, name)
        fn.restype = res
        fn.argtypes = args
    yield handle
    handle.qdecode_attn_debug_force_splits(0)


def status(L):
    v = ctypes.c_uint()
    assert L.qdecode_attn_device_status(ctypes.byref(v)) == 0
    return v.value


def run(L, fn_name, q, dev, N, w, Lq=None):
    out = torch.empty(q.shape, dtype=TORCH_DT[w.dtype_out], device="cuda")
    ptrs = [t.data_ptr() for t in (q, *dev, out)]
    n = _lib.int32_array(N)
    code = qda.dtype_code(q.dtype, out.dtype)
    s = torch.cuda.current_stream().cuda_stream
    if Lq is None:
        st = getattr(L, fn_name)(*ptrs, w.B, w.H, w.Hkv, n, w.D, w.GS, w.bits, code, s)
    else:
        st = L.qdecode_attn_multi(*ptrs, w.B, Lq, w.H, w.Hkv, n, w.D, w.GS, w.bits, code, s)
    assert st == 0
    torch.cuda.synchronize()
    return out.double().cpu().numpy()


CASES = [
    synth.small(B=4, H=8, Hkv=2, D=256, N=(1, 7, 9, 300), bits=8, GS=32, seed=61),
    synth.small(B=3, H=16, Hkv=4, D=256, N=(33, 1, 1000), bits=4, GS=64, dtype_out="fp32", seed=62),
    synth.small(B=2, H=8, Hkv=4, D=512, N=(5, 700), bits=4, GS=128, dtype_in="fp16", seed=63),
    synth.small(B=3, H=6, Hkv=3, D=128, N=(1, 17, 250), bits=8, GS=64, seed=64),
    synth.small(B=2, H=4, Hkv=1, D=64, N=(2, 129), bits=4, GS=32, seed=65),
    # the tensor-core kernel at D = 128 (two MMA tiles per pipeline step, 4 groups per row)
    synth.small(B=3, H=12, Hkv=3, D=128, N=(1, 300, 777), bits=4, GS=32, seed=66),
]


@pytest.mark.parametrize("splits", [0, 1, 3, 50, 199])
@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_checked_build_single_query(L, w, splits):
    q, cache, N = small_case(w)
    dev = upload_cache(*cache, w.dtype_in)
    status(L)
    L.qdecode_attn_debug_force_splits(splits)
    try:
        g = run(L, "qdecode_attn", q.cuda(), dev, N, w)
    finally:
        L.qdecode_attn_debug_force_splits(0)
    assert status(L) == 0
    ref = O.attention_packed(q.double().numpy(), *cache, N, w.H, w.Hkv, w.D, w.GS, w.bits)
    for (b, h), o in ref.items():
        assert np.abs(g[b, h] - o).max() <= TOL[w.dtype_out] * np.abs(o).max(), (b, h)


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_checked_build_multi_and_compat(L, w):
    _, cache, N = small_case(w)
    dev = upload_cache(*cache, w.dtype_in)
    Lq = min(3, min(N))
    q = synth.query_multi(w, Lq)
    status(L)
    g = run(L, "qdecode_attn_multi", q.cuda(), dev, N, w, Lq=Lq)
    assert status(L) == 0
    ref = O.attention_packed_multi(q.double().numpy(), *cache, N, Lq, w.H, w.Hkv, w.D, w.GS, w.bits)
    for (b, l, h), o in ref.items():
        assert np.abs(g[b, l, h] - o).max() <= TOL[w.dtype_out] * np.abs(o).max(), (b, l, h)
    q1 = synth.query(w)
    g = run(L, "qdecode_attn_compat", q1.cuda(), dev, N, w)
    assert status(L) == 0
    ref = O.attention_packed_compat(q1.double().numpy(), *cache, N, w.H, w.Hkv, w.D, w.GS, w.bits, w.dtype_in)
    for (b, h), o in ref.items():
        assert np.abs(g[b, h] - o).max() <= 1e-2 * np.abs(o).max(), (b, h)
