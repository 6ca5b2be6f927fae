"""The allocation-free entry point, qdecode_attn_noalloc, called through the C ABI.

It serves callers that may not allocate device memory themselves (a process whose allocator owns the device, a
latency-critical loop that cannot afford cudaMalloc's implicit synchronisation, a host that only hands out
pre-allocated buffers): its scratch is a fixed device array inside the library. It runs the same plan and kernels as
the regular entry point, so its output must equal that entry point's bit for bit, on consecutive calls that reuse
the array, and match the oracle within the parity tolerance; shapes that need more scratch than the array holds must
be refused before anything runs.

This file is collected last on purpose, and passes both alone in a fresh process and after the other tests.
"""
import ctypes

import pytest
import torch

import attention_quantized_kv_split_gb300 as qda
from attention_quantized_kv_split_gb300 import _lib, build, synth

from harness import TORCH_DT, compare, oracle_out, small_case, upload_cache

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    qda.lib()


def _abi_call(fn, q, dev, out, N, w):
    # straight through the C ABI: raw device pointers, a host array of lengths, the current stream
    B, H, D = q.shape
    ptrs = [t.data_ptr() for t in (q, *dev, out)]
    n = (ctypes.c_int32 * len(N))(*N)
    code = qda.dtype_code(q.dtype, out.dtype)
    return fn(*ptrs, B, H, w.Hkv, n, D, w.GS, w.bits, code, torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("w", [
    synth.workload(1),
    synth.small(B=3, H=16, Hkv=4, D=256, N=(700, 33, 2100), bits=4, GS=32, dtype_out="fp32", seed=31),
    synth.small(B=2, H=16, Hkv=8, D=256, N=(1500, 400), bits=8, GS=32, seed=32),
    synth.small(B=1, H=8, Hkv=4, D=512, N=(999,), bits=4, GS=128, dtype_in="fp16", seed=33),
    synth.small(B=2, H=4, Hkv=2, D=64, N=(130, 9), bits=4, GS=64, seed=34),
    synth.small(B=2, H=8, Hkv=2, D=128, N=(900, 300), bits=4, GS=64, seed=35),
], ids=lambda w: w.name)
def test_noalloc_matches_regular_entry_point_twice(w):
    q, cache, N = small_case(w)
    dev = upload_cache(*cache, w.dtype_in)
    qd = q.cuda()
    dt = TORCH_DT[w.dtype_out]
    ref = torch.empty(qd.shape, dtype=dt, device="cuda")
    assert _abi_call(_lib.lib().qdecode_attn, qd, dev, ref, N, w) == 0
    outs = []
    for _ in range(2):   # the second call runs on the scratch the first one left behind
        o = torch.full(qd.shape, float("nan"), dtype=dt, device="cuda")
        assert _abi_call(_lib.lib().qdecode_attn_noalloc, qd, dev, o, N, w) == 0
        outs.append(o)
    torch.cuda.synchronize()
    for o in outs:   # same plan, same kernels: the same bits as the regular entry point
        assert torch.equal(o.view(torch.uint8), ref.view(torch.uint8))
    compare(outs[1], oracle_out(q, cache, N, w), w.dtype_out)
    assert qda.qdecode_attn_device_status() == 0


def test_noalloc_refuses_shapes_beyond_its_scratch():
    # 512 one-row sequences of 8 KV heads with D = 512: the partials need far more than the fixed array
    B, H, Hkv, D, GS, bits = 512, 32, 8, 512, 128, 4
    N = [1] * B
    need = qda.qdecode_attn_workspace_bytes(B, H, Hkv, N, D, GS, bits)
    assert need > _lib.QDA_STATIC_SCRATCH_BYTES
    rows = Hkv * sum(N)
    w = synth.small(B=B, H=H, Hkv=Hkv, D=D, N=tuple(N), bits=bits, GS=GS)
    q = torch.zeros((B, H, D), dtype=torch.bfloat16, device="cuda")
    dev = (torch.zeros((rows, D * bits // 32), dtype=torch.int32, device="cuda"),
           *[torch.zeros((rows, D // GS), dtype=torch.bfloat16, device="cuda") for _ in range(2)],
           torch.zeros((rows, D * bits // 32), dtype=torch.int32, device="cuda"),
           *[torch.zeros((rows, D // GS), dtype=torch.bfloat16, device="cuda") for _ in range(2)])
    out = torch.empty_like(q)
    st = _abi_call(_lib.lib().qdecode_attn_noalloc, q, dev, out, N, w)
    assert st == _lib.QDA_ERR_SCRATCH
    assert b"scratch" in _lib.lib().qdecode_attn_strerror(st)
