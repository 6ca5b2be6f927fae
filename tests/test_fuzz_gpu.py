"""Seeded random shapes against the oracle: B, lengths (including 1-row sequences), H/Hkv, D, GS, bits, dtypes,
query positions and forced split counts drawn from one generator, for single-query, multi-query and compat calls.
Tolerances as in the other parity tests (the compat form at the 16-bit rule)."""
import numpy as np
import pytest
import torch

import oracle as O
import attention_quantized_kv_split_gb300 as qda
from attention_quantized_kv_split_gb300 import build, synth

from harness import TOL, TORCH_DT, small_case, upload_cache

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    qda.lib()
    qda.qdecode_attn_debug_force_splits(0)
    yield
    qda.qdecode_attn_debug_force_splits(0)


def draw(seed):
    r = np.random.default_rng(seed)
    D = int(r.choice([64, 128, 256, 512]))
    GS = int(r.choice([g for g in (32, 64, 128) if D % g == 0]))
    bits = int(r.choice([4, 8]))
    Hkv = int(r.choice([1, 2, 3, 4, 8]))
    nrep = int(r.choice([1, 2, 3, 4, 6, 8]))
    B = int(r.integers(1, 6))
    N = tuple(int(x) for x in r.choice([1, 2, 7, 16, 33, 100, 257, 900, 2500], size=B))
    dtin = str(r.choice(["bf16", "fp16"]))
    dtout = str(r.choice(["bf16", "fp16", "fp32"]))
    L = int(r.integers(1, 5))
    splits = int(r.choice([0, 0, 1, 5, 40]))
    w = synth.small(B=B, H=Hkv * nrep, Hkv=Hkv, D=D, N=N, bits=bits, GS=GS, dtype_in=dtin, dtype_out=dtout,
                    seed=1000 + seed)
    return w, L, splits


def check(g, ref, tol):
    g = g.double().cpu().numpy()
    for key, o in ref.items():
        assert np.all(np.isfinite(g[key])), key
        assert np.abs(g[key] - o).max() <= tol * np.abs(o).max(), key


@pytest.mark.parametrize("seed", range(40))
def test_random_shapes(seed):
    w, L, splits = draw(seed)
    q, cache, N = small_case(w)
    dev = upload_cache(*cache, w.dtype_in)
    dt = TORCH_DT[w.dtype_out]
    qda.qdecode_attn_debug_force_splits(splits)
    try:
        out = torch.empty((w.B, w.H, w.D), dtype=dt, device="cuda")
        qda.qdecode_attn(q.cuda(), *dev, out, N, w.Hkv, w.GS, w.bits)
        qv = q.double().numpy()
        check(out, O.attention_packed(qv, *cache, N, w.H, w.Hkv, w.D, w.GS, w.bits), TOL[w.dtype_out])
        Lq = min(L, min(N))
        qm = synth.query_multi(w, Lq)
        outm = torch.empty((w.B, Lq, w.H, w.D), dtype=dt, device="cuda")
        qda.qdecode_attn_multi(qm.cuda(), *dev, outm, N, w.Hkv, w.GS, w.bits)
        check(outm, O.attention_packed_multi(qm.double().numpy(), *cache, N, Lq, w.H, w.Hkv, w.D, w.GS, w.bits),
              TOL[w.dtype_out])
        outc = torch.empty((w.B, w.H, w.D), dtype=dt, device="cuda")
        qda.qdecode_attn_compat(q.cuda(), *dev, outc, N, w.Hkv, w.GS, w.bits)
        check(outc, O.attention_packed_compat(qv, *cache, N, w.H, w.Hkv, w.D, w.GS, w.bits, w.dtype_in), 1e-2)
    finally:
        qda.qdecode_attn_debug_force_splits(0)
    assert qda.qdecode_attn_device_status() == 0
