"""The seeded input generator draws what each workload asks for. CPU only."""
import math

import torch

from attention_quantized_kv_split_gb300 import synth


def test_lengths_fixed_and_ragged():
    assert synth.lengths(synth.workload(2)) == [8192]
    n = synth.lengths(synth.workload(4))
    assert len(n) == 8 and all(1024 <= v <= 65536 for v in n)
    assert n == synth.lengths(synth.workload(4))          # reproducible
    assert len(set(n)) > 1


def test_query_dtype_and_determinism():
    w = synth.workload(3)
    q = synth.query(w)
    assert q.dtype == torch.float16 and tuple(q.shape) == (1, 16, 512)
    assert torch.equal(q, synth.query(w))


def test_outlier_channels():
    w = synth.small(D=64, N=(400,), k_outliers=4, outlier_scale=20.0)
    K, V = synth.kv_unit(w, 0, 1, 400)
    sd = K.std(0)
    big = (sd > 5).nonzero().flatten()
    assert len(big) == 4
    assert torch.all(sd[big] > 15) and V.std(0).max() < 2


def test_planted_keys_cosine():
    w = synth.small(B=1, H=8, Hkv=2, D=256, N=(1000,), planted=32, v_uniform=True)
    q = synth.query(w)
    K, V = synth.kv_unit(w, 0, 1, 1000, q=q)
    rows = synth.planted_rows(w, 0, 1, 1000)
    assert len(set(rows)) == 32
    for i, r in enumerate(rows):
        h = 1 * w.nrep + i % w.nrep
        qh = q[0, h].float()
        cos = (K[r] @ qh / (K[r].norm() * qh.norm())).item()
        assert abs(cos - 0.9) < 1e-5
        assert abs(K[r].norm().item() - math.sqrt(256)) < 1e-3
    assert V.min() >= -1 and V.max() <= 1


def test_units_independent_streams():
    w = synth.workload(1)
    k0, _ = synth.kv_unit(w, 0, 0, 64)
    k1, _ = synth.kv_unit(w, 0, 1, 64)
    assert not torch.equal(k0, k1)
    k0b, _ = synth.kv_unit(w, 0, 0, 64)
    assert torch.equal(k0, k0b)
