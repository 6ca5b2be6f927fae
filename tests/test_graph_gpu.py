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


def test_replay_after_the_workspace_grew():
    # a call captured on the library's workspace keeps working after a later eager call of a larger shape made the
    # library grow its workspace: the outgrown buffer stays allocated, so the replay writes to valid memory
    w = synth.small(B=2, H=8, Hkv=2, D=256, N=(700, 90), bits=4, GS=64, seed=72)
    q, cache, N = small_case(w)
    dev = upload_cache(*cache, w.dtype_in)
    qd = q.cuda()
    eager = torch.empty(qd.shape, dtype=TORCH_DT[w.dtype_out], device="cuda")
    qda.qdecode_attn(qd, *dev, eager, N, w.Hkv, w.GS, w.bits)
    torch.cuda.synchronize()
    out = torch.full_like(eager, float("nan"))
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            qda.qdecode_attn(qd, *dev, out, N, w.Hkv, w.GS, w.bits, stream=s)
    # a much larger call: far more partial slots (8192 one-row units) than any other test's shape needs
    big = synth.small(B=512, H=64, Hkv=16, D=512, N=tuple([1] * 512), bits=4, GS=128, seed=73)
    need_small = qda.qdecode_attn_workspace_bytes(w.B, w.H, w.Hkv, N, w.D, w.GS, w.bits)
    need_big = qda.qdecode_attn_workspace_bytes(big.B, big.H, big.Hkv, list(big.N), big.D, big.GS, big.bits)
    assert need_big > 2 * max(need_small, 1 << 20)
    qb, cb, Nb = small_case(big)
    devb = upload_cache(*cb, big.dtype_in)
    ob = torch.empty(qb.shape, dtype=TORCH_DT[big.dtype_out], device="cuda")
    qda.qdecode_attn(qb.cuda(), *devb, ob, Nb, big.Hkv, big.GS, big.bits)
    torch.cuda.synchronize()
    for _ in range(2):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    assert qda.qdecode_attn_device_status() == 0
