"""The decode calls inside a captured CUDA graph: after one warm-up call (which sizes the library's workspace and
sets the kernels' shared-memory limits), a call records its split and merge kernels into a graph without allocating,
and replays give the eager result bit for bit."""
import pytest
import torch

import attention_quantized_kv_split_gb300 as qda
from attention_quantized_kv_split_gb300 import build, synth

from harness import TORCH_DT, small_case, upload_cache

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    qda.lib()


@pytest.mark.parametrize("fn_name", ["qdecode_attn", "qdecode_attn_compat", "qdecode_attn_multi"])
def test_captured_call_replays_bitwise(fn_name):
    w = synth.small(B=3, H=16, Hkv=4, D=256, N=(900, 40, 2500), bits=4, GS=64, seed=71)
    q1, cache, N = small_case(w)
    dev = upload_cache(*cache, w.dtype_in)
    q = (synth.query_multi(w, 3) if fn_name == "qdecode_attn_multi" else q1).cuda()
    fn = getattr(qda, fn_name)
    eager = torch.empty(q.shape, dtype=TORCH_DT[w.dtype_out], device="cuda")
    fn(q, *dev, eager, N, w.Hkv, w.GS, w.bits)          # warm-up: workspace and kernel attributes
    torch.cuda.synchronize()
    out = torch.full_like(eager, float("nan"))
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            fn(q, *dev, out, N, w.Hkv, w.GS, w.bits, stream=s)
    for _ in range(3):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    assert qda.qdecode_attn_device_status() == 0
