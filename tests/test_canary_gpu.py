"""Out-of-bounds writes: guard bytes of a known pattern before and after the output and an installed workspace.

Every decode entry point writes only inside `out` and inside the workspace it was given (of exactly the size the
library reports), for the tensor-core and CUDA-core split kernels, multi-query decode and the two-pass compat form,
on ragged batches and forced split counts (up to one range per few rows). The guards must come back unchanged and
the outputs finite; a stray store of the merge or the split kernels past either buffer would change a guard."""
import numpy as np
import pytest
import torch

import attention_quantized_kv_split_gb300 as qda
from attention_quantized_kv_split_gb300 import build, synth

from harness import TORCH_DT, small_case, upload_cache

pytestmark = pytest.mark.gpu

GUARD = 8192          # guard bytes on each side (keeps every payload 16-byte aligned)
PATTERN = 0xA5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    qda.lib()
    qda.qdecode_attn_debug_force_splits(0)
    qda.qdecode_attn_set_workspace(None)
    yield
    qda.qdecode_attn_debug_force_splits(0)
    qda.qdecode_attn_set_workspace(None)


def guarded(nbytes: int):
    """A device buffer of GUARD + nbytes + GUARD bytes, all set to PATTERN; returns (buffer, payload byte view)."""
    buf = torch.full((GUARD + nbytes + GUARD,), PATTERN, dtype=torch.uint8, device="cuda")
    return buf, buf[GUARD:GUARD + nbytes]


def guards_intact(buf: torch.Tensor) -> bool:
    b = buf.cpu().numpy()
    return bool(np.all(b[:GUARD] == PATTERN) and np.all(b[-GUARD:] == PATTERN))


CASES = [
    # (workload, query positions, compat form)
    (synth.small(B=3, H=16, Hkv=4, D=256, N=(700, 33, 2100), bits=4, GS=32, dtype_out="fp32", seed=41), 1, False),
    (synth.small(B=2, H=8, Hkv=2, D=128, N=(1300, 257), bits=4, GS=64, seed=42), 1, False),
    (synth.small(B=4, H=16, Hkv=8, D=256, N=(1500, 9, 400, 77), bits=8, GS=32, seed=43), 1, False),
    (synth.small(B=2, H=8, Hkv=4, D=512, N=(999, 130), bits=4, GS=128, dtype_in="fp16", seed=44), 1, False),
    (synth.small(B=2, H=4, Hkv=2, D=64, N=(130, 9), bits=4, GS=64, seed=45), 1, False),
    (synth.small(B=2, H=8, Hkv=2, D=256, N=(600, 45), bits=4, GS=64, seed=46), 3, False),
    (synth.small(B=2, H=8, Hkv=2, D=256, N=(800, 70), bits=8, GS=64, seed=47), 1, True),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0].name}_L{c[1]}{'_compat' if c[2] else ''}")
@pytest.mark.parametrize("splits", [0, 7, 300])
def test_writes_stay_inside_out_and_workspace(case, splits):
    w, L, compat = case
    q, cache, N = small_case(w)
    dev = upload_cache(*cache, w.dtype_in)
    if L > 1:
        q = synth.query_multi(w, L)
    qd = q.cuda()
    dt = TORCH_DT[w.dtype_out]
    esize = torch.empty((), dtype=dt).element_size()
    out_buf, out_bytes = guarded(qd.numel() * esize)
    out = out_bytes.view(dt).view(qd.shape)
    qda.qdecode_attn_debug_force_splits(splits)
    try:
        if L > 1:
            need = qda.qdecode_attn_multi_plan(w.B, L, w.H, w.Hkv, N, w.D, w.GS, w.bits)["workspace_bytes"]
        else:
            need = qda.qdecode_attn_workspace_bytes(w.B, w.H, w.Hkv, N, w.D, w.GS, w.bits)
        ws_buf, ws = guarded((need + 15) // 16 * 16)
        qda.qdecode_attn_set_workspace(ws)
        try:
            if L > 1:
                qda.qdecode_attn_multi(qd, *dev, out, N, w.Hkv, w.GS, w.bits)
            elif compat:
                qda.qdecode_attn_compat(qd, *dev, out, N, w.Hkv, w.GS, w.bits)
            else:
                qda.qdecode_attn(qd, *dev, out, N, w.Hkv, w.GS, w.bits)
            torch.cuda.synchronize()
        finally:
            qda.qdecode_attn_set_workspace(None)
    finally:
        qda.qdecode_attn_debug_force_splits(0)
    assert guards_intact(out_buf), "a write landed outside out"
    assert guards_intact(ws_buf), "a write landed outside the workspace"
    assert np.all(np.isfinite(out.double().cpu().numpy()))
    assert qda.qdecode_attn_device_status() == 0
