"""GPU parity of small-L multi-query decode (qdecode_attn_multi) against the fp64 oracle, through the C ABI.

Each sequence has L query positions, its last L tokens; position l attends the first N[b] - L + 1 + l cache rows.
Tolerance per (sequence, position, head) as for single-query decode: max|delta| <= 1e-2 * max|o| for bf16/fp16
outputs, <= 1e-4 * max|o| for fp32 outputs."""
import numpy as np
import pytest
import torch

import oracle as O
import attention_quantized_kv_split_gb300 as qda
from attention_quantized_kv_split_gb300 import build, synth

from harness import TOL, TORCH_DT, gpu_quantized_workload, small_case, unit_oracle_cache, upload_cache

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    qda.lib()
    qda.qdecode_attn_debug_force_splits(0)
    yield
    qda.qdecode_attn_debug_force_splits(0)


def run_multi(q, dev, N, w, out_dtype=None, splits=0):
    out = torch.empty(q.shape, dtype=TORCH_DT[out_dtype or w.dtype_out], device="cuda")
    qda.qdecode_attn_debug_force_splits(splits)
    try:
        qda.qdecode_attn_multi(q.cuda(), *dev, out, N, w.Hkv, w.GS, w.bits)
    finally:
        qda.qdecode_attn_debug_force_splits(0)
    return out


def compare_multi(out, ref, out_dtype):
    g = out.to(torch.float64).cpu().numpy()
    for (b, l, h), o in ref.items():
        assert np.all(np.isfinite(g[b, l, h])), (b, l, h)
        err = np.abs(g[b, l, h] - o).max()
        bound = TOL[out_dtype] * np.abs(o).max()
        assert err <= bound, f"{(b, l, h)}: max|delta| {err:.3e} > {bound:.3e}"


def check(w, L, out_dtype=None, splits=0):
    _, cache, N = small_case(w)
    q = synth.query_multi(w, L)
    dev = upload_cache(*cache, w.dtype_in)
    out = run_multi(q, dev, N, w, out_dtype, splits)
    ref = O.attention_packed_multi(q.to(torch.float64).numpy(), *cache, N, L, w.H, w.Hkv, w.D, w.GS, w.bits)
    compare_multi(out, ref, out_dtype or w.dtype_out)
    return out, (q, dev, N)


SHAPES = [(D, bits, GS) for D in (64, 128, 256, 512) for bits in (4, 8) for GS in (32, 128) if D % GS == 0]


@pytest.mark.parametrize("L", [2, 3, 4])
@pytest.mark.parametrize("D,bits,GS", SHAPES)
def test_multi_shape_sweep(D, bits, GS, L):
    check(synth.small(B=2, H=4, Hkv=2, D=D, N=(131, L), bits=bits, GS=GS, seed=D * 3 + bits + GS + L), L)


@pytest.mark.parametrize("H,Hkv,L", [(8, 2, 4), (16, 8, 4), (16, 4, 2), (3, 1, 3), (32, 8, 2), (4, 4, 8), (8, 1, 8)])
def test_multi_gqa_and_positions(H, Hkv, L):
    check(synth.small(B=2, H=H, Hkv=Hkv, D=256, N=(300, 41), bits=4, GS=64, seed=H * 7 + Hkv + L), L)


@pytest.mark.parametrize("D", [128, 256, 512])
def test_multi_fp32_and_fp16(D):
    check(synth.small(B=1, H=8, Hkv=2, D=D, N=(777,), bits=4, GS=32, dtype_in="fp16", seed=D + 1), 3, "fp32")
    check(synth.small(B=1, H=8, Hkv=2, D=D, N=(777,), bits=8, GS=32, seed=D + 2), 2, "fp32")


@pytest.mark.parametrize("splits", [1, 2, 5, 17, 64, 200])
def test_multi_forced_splits(splits):
    # with many splits some row ranges lie entirely in the hidden tail of a position
    w = synth.small(B=3, H=8, Hkv=2, D=256, N=(90, 8, 400), bits=4, GS=64, seed=splits)
    check(w, 4, splits=splits)
    w = synth.small(B=2, H=4, Hkv=2, D=128, N=(64, 33), bits=8, GS=32, seed=splits + 1)
    check(w, 3, splits=splits)


def test_multi_every_position_sees_one_more_row():
    # N = L: position l sees exactly l + 1 rows (position 0 attends only the first row: its V row)
    w = synth.small(B=1, H=4, Hkv=1, D=256, N=(8,), bits=8, GS=32, seed=5)
    out, _ = check(w, 8, out_dtype="fp32")
    _, cache, N = small_case(w)
    kp, ks, kb, vp, vs, vb = cache
    v0 = O.dequantize(O.unpack(vp[0:1], 8, 256), vs[0:1], vb[0:1], 32)[0]
    g = out.to(torch.float64).cpu().numpy()
    for h in range(4):
        assert np.abs(g[0, 0, h] - v0).max() <= 1e-6 * np.abs(v0).max()


def test_multi_l1_is_single_query_bitwise():
    w = synth.small(B=2, H=16, Hkv=8, D=256, N=(1000, 77), bits=8, GS=32, seed=3)
    q, cache, N = small_case(w)
    dev = upload_cache(*cache, w.dtype_in)
    qd = q.cuda()
    one = torch.empty_like(qd)
    qda.qdecode_attn(qd, *dev, one, N, w.Hkv, w.GS, w.bits)
    multi = torch.empty_like(qd)[:, None]
    qda.qdecode_attn_multi(qd[:, None].contiguous(), *dev, multi, N, w.Hkv, w.GS, w.bits)
    torch.cuda.synchronize()
    assert torch.equal(one.view(torch.int16), multi[:, 0].view(torch.int16))


def test_multi_run_to_run_bitwise():
    w = synth.small(B=2, H=8, Hkv=2, D=512, N=(2000, 300), bits=4, GS=128, dtype_in="fp16", seed=9)
    out1, (q, dev, N) = check(w, 4)
    for _ in range(3):
        out2 = run_multi(q, dev, N, w)
        torch.cuda.synchronize()
        assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert qda.qdecode_attn_device_status() == 0


def test_multi_8k_workload_sampled():
    # the 8k configuration (B=1, H=16, Hkv=8, D=256, 8-bit, GS=32) with 4 query positions, as the bench runs it
    w = synth.workload(2)
    L = 4
    q1, cache, N = gpu_quantized_workload(w)
    q = synth.query_multi(w, L)
    out = torch.empty((w.B, L, w.H, w.D), dtype=TORCH_DT[w.dtype_out], device="cuda")
    qda.qdecode_attn_multi(q.cuda(), cache.kp, cache.ks, cache.kb, cache.vp, cache.vs, cache.vb, out, N, w.Hkv,
                           w.GS, w.bits)
    torch.cuda.synchronize()
    nrep = w.H // w.Hkv
    for kvh in (0, 5):
        unit = unit_oracle_cache(w, 0, kvh, N, q1)
        qs = q[:, :, kvh * nrep:(kvh + 1) * nrep].to(torch.float64).numpy()
        ref = O.attention_packed_multi(qs, *unit, [N[0]], L, nrep, 1, w.D, w.GS, w.bits)
        sub = out[:, :, kvh * nrep:(kvh + 1) * nrep]
        compare_multi(sub, ref, w.dtype_out)
    assert qda.qdecode_attn_device_status() == 0
