"""Failure detection on the GPU without a fault: a pipeline wait that runs out reports through the device status
word, the call returns, and the context stays usable.

The first CTA's producer is told to stop before one of its chunks (a testing switch of the library), so that CTA's
consumers wait for data that never comes. Every wait in the split kernel is bounded (about one second): the
consumers give up, record bit 1 in the device error word, raise the CTA's abort flag and finish; the producer has
only its issued copies to drain. The host reads the status, switches the stall off, and the next call is correct."""
import time

import numpy as np
import pytest
import torch

import attention_quantized_kv_split_gb300 as qda
from attention_quantized_kv_split_gb300 import build, synth

from harness import TORCH_DT, compare, oracle_out, small_case, upload_cache

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    qda.lib()
    qda.qdecode_attn_debug_stall_chunk(-1)
    yield
    qda.qdecode_attn_debug_stall_chunk(-1)


def call(fn, q, dev, N, w):
    out = torch.empty(q.shape, dtype=TORCH_DT[w.dtype_out], device="cuda")
    fn(q.cuda(), *dev, out, N, w.Hkv, w.GS, w.bits)
    return out


@pytest.mark.parametrize("fn_name,D", [("qdecode_attn", 256), ("qdecode_attn", 128), ("qdecode_attn_compat", 512)])
def test_stalled_pipeline_is_reported_and_the_context_recovers(fn_name, D):
    fn = getattr(qda, fn_name)
    w = synth.small(B=1, H=8, Hkv=2, D=D, N=(6000,), bits=4, GS=64, seed=D)
    q, cache, N = small_case(w)
    dev = upload_cache(*cache, w.dtype_in)
    qda.qdecode_attn_device_status()            # start clean
    qda.qdecode_attn_debug_stall_chunk(0)        # the first chunk: every range has one
    try:
        t0 = time.time()
        call(fn, q, dev, N, w)
        torch.cuda.synchronize()
        elapsed = time.time() - t0
    finally:
        qda.qdecode_attn_debug_stall_chunk(-1)
    status = qda.qdecode_attn_device_status()
    assert status & 1, status                   # a consumer wait gave up
    assert elapsed < 10.0                       # bounded: about one second per stalled pass
    out = call(fn, q, dev, N, w)                # the context still works and the next call is clean
    torch.cuda.synchronize()
    assert qda.qdecode_attn_device_status() == 0
    if fn_name == "qdecode_attn":
        compare(out, oracle_out(q, cache, N, w), w.dtype_out)
    else:
        assert np.all(np.isfinite(out.double().cpu().numpy()))
