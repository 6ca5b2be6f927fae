"""The host-buffer entry point (qdecode_attn_host) through the C ABI: inputs and output in host memory, staged on
the device by the library. Its kernels are qdecode_attn's, so its output must equal qdecode_attn's on the same
inputs bit for bit; the oracle comparison of that path is in the parity tests, and one case here repeats it."""
import numpy as np
import pytest
import torch

import oracle as O
import attention_quantized_kv_split_gb300 as qda
from attention_quantized_kv_split_gb300 import build, synth

from harness import TORCH_DT, compare, small_case, upload_cache

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    qda.lib()
    yield


def host_copies(q, dev, pinned):
    """q and the cache exactly as the device holds them (the library's bytes), as contiguous host tensors."""
    ts = [q.contiguous()] + [t.cpu() for t in dev]
    return [t.pin_memory() for t in ts] if pinned else ts


def run_both(w, out_dtype=None, pinned=True):
    q, cache, N = small_case(w)
    dt = TORCH_DT[out_dtype or w.dtype_out]
    dev = upload_cache(*cache, w.dtype_in)
    ref = torch.empty(q.shape, dtype=dt, device="cuda")
    qda.qdecode_attn(q.cuda(), *dev, ref, N, w.Hkv, w.GS, w.bits)
    hin = host_copies(q, dev, pinned)
    hout = torch.empty(q.shape, dtype=dt)
    if pinned:
        hout = hout.pin_memory()
    qda.qdecode_attn_host(*hin, hout, N, w.Hkv, w.GS, w.bits)
    torch.cuda.synchronize()
    return q, cache, N, ref.cpu(), hout


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("D,bits,GS,out", [(256, 8, 32, None), (256, 4, 64, "fp32"), (512, 4, 128, None),
                                           (128, 8, 32, None), (64, 4, 32, "fp32")])
def test_host_equals_device(D, bits, GS, out, pinned):
    w = synth.small(B=3, H=8, Hkv=2, D=D, N=(700, 1, 257), bits=bits, GS=GS, seed=D + bits + GS)
    _, _, _, ref, got = run_both(w, out, pinned)
    assert torch.equal(ref.view(torch.uint8), got.view(torch.uint8))


def test_host_against_oracle():
    w = synth.small(B=2, H=16, Hkv=8, D=256, N=(3000, 45), bits=8, GS=32, seed=77)
    q, cache, N, _, got = run_both(w)
    ref = O.attention_packed(q.to(torch.float64).numpy(), *cache, N, w.H, w.Hkv, w.D, w.GS, w.bits)
    compare(got, ref, w.dtype_out)


def test_host_consecutive_calls_use_both_staging_sets():
    # five calls in a row without synchronising in between, each with its own inputs and output, growing and
    # shrinking: every result equals the device path's
    shapes = [(500,), (40, 9), (4000,), (7,), (1500, 2)]
    outs, refs = [], []
    keep = []
    for i, N in enumerate(shapes):
        w = synth.small(B=len(N), H=4, Hkv=2, D=256, N=N, bits=4, GS=32, seed=100 + i)
        q, cache, Nn = small_case(w)
        dev = upload_cache(*cache, w.dtype_in)
        ref = torch.empty(q.shape, dtype=TORCH_DT[w.dtype_out], device="cuda")
        qda.qdecode_attn(q.cuda(), *dev, ref, Nn, w.Hkv, w.GS, w.bits)
        hin = host_copies(q, dev, True)
        hout = torch.empty(q.shape, dtype=TORCH_DT[w.dtype_out]).pin_memory()
        keep.append(hin)
        qda.qdecode_attn_host(*hin, hout, Nn, w.Hkv, w.GS, w.bits)
        outs.append(hout)
        refs.append(ref)
    torch.cuda.synchronize()
    for ref, got in zip(refs, outs):
        assert torch.equal(ref.cpu().view(torch.uint8), got.view(torch.uint8))
    assert qda.qdecode_attn_device_status() == 0


def test_host_rejects_device_tensors():
    w = synth.small(B=1, H=4, Hkv=2, D=256, N=(64,), bits=4, GS=32, seed=3)
    q, cache, N = small_case(w)
    dev = upload_cache(*cache, w.dtype_in)
    with pytest.raises(ValueError):
        qda.qdecode_attn_host(q.cuda(), *dev, torch.empty(q.shape, dtype=q.dtype, device="cuda"), N, w.Hkv, w.GS,
                              w.bits)
