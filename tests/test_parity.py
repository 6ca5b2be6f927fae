"""GPU parity: the library's decode attention against the fp64 oracle, per head, through the C ABI.

Tolerance (per head): max|delta| <= 1e-2 * max|o| for bf16/fp16 outputs and <= 1e-4 * max|o| for fp32 outputs.
Small cases and the full-size workloads compare every head (for the full-size workloads the oracle quantizes each
(sequence, KV head) unit itself from the same generated rows, and the library's quantized bytes must match its
bytes exactly)."""
import numpy as np
import pytest
import torch

import oracle as O
import attention_quantized_kv_split_gb300 as qda
from attention_quantized_kv_split_gb300 import _lib as qlib, build, synth

from harness import (TORCH_DT, compare, gpu_quantized_workload, oracle_out, run_gpu, small_case,
                     unit_oracle_cache, upload_cache)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    qda.lib()
    qda.qdecode_attn_debug_force_splits(0)
    yield
    qda.qdecode_attn_debug_force_splits(0)


def check_small(w, out_dtype=None, splits=0):
    q, cache, N = small_case(w)
    dev = upload_cache(*cache, w.dtype_in)
    qda.qdecode_attn_debug_force_splits(splits)
    try:
        out = run_gpu(q, dev, N, w, out_dtype)
    finally:
        qda.qdecode_attn_debug_force_splits(0)
    ref = oracle_out(q, cache, N, w)
    compare(out, ref, out_dtype or w.dtype_out)
    return out, (q, dev, N)


def test_workload1_all_heads():
    check_small(synth.workload(1))
    assert qda.qdecode_attn_device_status() == 0


SWEEP = [(D, bits, GS) for D in (64, 128, 256, 512) for bits in (4, 8) for GS in (32, 64, 128) if D % GS == 0]


@pytest.mark.parametrize("N", [1, 33, 257])
@pytest.mark.parametrize("D,bits,GS", SWEEP)
def test_shape_sweep(D, bits, GS, N):
    check_small(synth.small(B=1, H=4, Hkv=2, D=D, N=(N,), bits=bits, GS=GS, seed=D * 31 + bits * 7 + GS + N))


@pytest.mark.parametrize("H,Hkv", [(1, 1), (2, 1), (4, 1), (8, 1), (16, 2), (3, 1), (6, 2), (24, 2), (32, 1)])
def test_gqa_ratios(H, Hkv):
    check_small(synth.small(B=2, H=H, Hkv=Hkv, D=128, N=(300, 41), bits=4, GS=32, seed=H * 5 + Hkv))


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("dt_in,dt_out", [("bf16", "bf16"), ("bf16", "fp16"), ("bf16", "fp32"), ("fp16", "fp16"),
                                          ("fp16", "bf16"), ("fp16", "fp32")])
def test_dtypes(dt_in, dt_out, D):
    # four query heads per KV head: the tensor-core kernel, whose D = 128 instances take the input dtype as a
    # template argument
    check_small(synth.small(B=1, H=8, Hkv=2, D=D, N=(777,), bits=4, GS=64, dtype_in=dt_in, dtype_out=dt_out))


def test_ragged_batch():
    check_small(synth.small(B=5, H=8, Hkv=4, D=256, N=(1, 17, 300, 8, 1025), bits=4, GS=64, seed=3))


def test_maximum_batch_of_tiny_sequences():
    # QDA_MAX_B sequences of 1-6 rows: 1024 (sequence, KV head) units, so every CTA range crosses dozens of unit
    # boundaries (one partial slot per segment) and the merge covers 4096 heads
    N = tuple(1 + (b * 5) % 6 for b in range(qlib.QDA_MAX_B))
    check_small(synth.small(B=len(N), H=8, Hkv=2, D=256, N=N, bits=4, GS=64, seed=11))


@pytest.mark.parametrize("D", [128, 256])
def test_maximum_query_heads_per_kv_head(D):
    # QDA_MAX_NREP query heads share one KV head (the lean kernel takes them 4 at a time in 16 head chunks)
    check_small(synth.small(B=1, H=qlib.QDA_MAX_NREP, Hkv=1, D=D, N=(300,), bits=8, GS=32, seed=D + 64))


def test_ragged_tail_scale_bytes():
    # D = GS = 64: one 2-byte scale per row, 3 * 13 = 39 rows -> the arrays end off a 16-byte boundary
    check_small(synth.small(B=1, H=6, Hkv=3, D=64, N=(13,), bits=4, GS=64, seed=4))
    check_small(synth.small(B=3, H=2, Hkv=1, D=128, N=(5, 3, 11), bits=8, GS=128, seed=5), splits=3)


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 50, 400])
def test_forced_splits_within_tolerance(splits):
    w = synth.small(B=3, H=8, Hkv=2, D=256, N=(700, 5, 1300), bits=4, GS=32, dtype_out="fp32", seed=9)
    out1, (q, dev, N) = check_small(w, splits=splits)
    qda.qdecode_attn_debug_force_splits(splits)
    try:
        out2 = run_gpu(q, dev, N, w)
    finally:
        qda.qdecode_attn_debug_force_splits(0)
    assert torch.equal(out1, out2)


@pytest.mark.parametrize("D,GS,out", [(128, 32, "fp32"), (512, 64, None), (512, 128, "fp32")])
def test_merge_over_head_dimension_slices(D, GS, out):
    # enough forced splits that every head's partials span many slots: the merge then runs one CTA per 64 values of
    # the head dimension (D / 64 CTAs per head); the result must still match the oracle and repeat bit for bit
    w = synth.small(B=2, H=8, Hkv=2, D=D, N=(1500, 37), bits=4, GS=GS, dtype_out=out or "bf16", seed=D + GS)
    out1, (q, dev, N) = check_small(w, splits=600)
    qda.qdecode_attn_debug_force_splits(600)
    try:
        out2 = run_gpu(q, dev, N, w)
    finally:
        qda.qdecode_attn_debug_force_splits(0)
    assert torch.equal(out1, out2)


def test_run_to_run_bitwise_identical():
    w = synth.small(B=4, H=16, Hkv=4, D=256, N=(3000, 20, 1, 9000), bits=4, GS=64, seed=21)
    q, cache, N = small_case(w)
    dev = upload_cache(*cache, w.dtype_in)
    outs = [run_gpu(q, dev, N, w) for _ in range(5)]
    for o in outs[1:]:
        assert torch.equal(outs[0].view(torch.int16), o.view(torch.int16))


def test_non_default_stream():
    w = synth.workload(1)
    q, cache, N = small_case(w)
    dev = upload_cache(*cache, w.dtype_in)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out = run_gpu(q, dev, N, w, stream=s)
    s.synchronize()
    compare(out, oracle_out(q, cache, N, w), w.dtype_out)


def test_caller_workspace():
    w = synth.small(B=2, H=8, Hkv=2, D=128, N=(900, 77), bits=8, GS=64, seed=8)
    q, cache, N = small_case(w)
    dev = upload_cache(*cache, w.dtype_in)
    need = qda.qdecode_attn_workspace_bytes(w.B, w.H, w.Hkv, N, w.D, w.GS, w.bits)
    small = torch.empty(max(16, need // 2), dtype=torch.uint8, device="cuda")
    ws = torch.empty(need + 256, dtype=torch.uint8, device="cuda")
    try:
        qda.qdecode_attn_set_workspace(small)
        with pytest.raises(qda.QdaError):
            run_gpu(q, dev, N, w)
        qda.qdecode_attn_set_workspace(ws)
        out = run_gpu(q, dev, N, w)
    finally:
        qda.qdecode_attn_set_workspace(None)
    compare(out, oracle_out(q, cache, N, w), w.dtype_out)


# --------------------------------------------------------------------------- full-size workloads (every unit)

SAMPLE_UNITS = {2: None, 3: None, 4: None, 5: None}   # every (sequence, KV head) of every workload


@pytest.mark.parametrize("idx", [2, 3, 4, 5])
def test_full_workload_sampled(idx):
    w = synth.workload(idx)
    q, cache, N = gpu_quantized_workload(w)
    out = torch.empty((w.B, w.H, w.D), dtype=TORCH_DT[w.dtype_out], device="cuda")
    qda.decode_attention(q.to("cuda"), cache, out=out)      # the launch configuration the bench times
    out2 = torch.empty_like(out)
    qda.decode_attention(q.to("cuda"), cache, out=out2)
    assert torch.equal(out.view(torch.uint8), out2.view(torch.uint8))
    units = SAMPLE_UNITS[idx] or [(b, k) for b in range(w.B) for k in range(w.Hkv)]
    qv = q.to(torch.float64).numpy()
    g = out.to(torch.float64).cpu().numpy()
    for b, kvh in units:
        kp, ks, kb, vp, vs, vb = unit_oracle_cache(w, b, kvh, N, q)
        r0, r1 = cache.unit_rows(b, kvh)
        # the library's quantizer produced exactly the oracle's bytes for this unit
        assert np.array_equal(cache.kp[r0:r1].cpu().numpy().view(np.uint32), kp)
        assert np.array_equal(cache.vp[r0:r1].cpu().numpy().view(np.uint32), vp)
        for dev_t, ref in ((cache.ks, ks), (cache.kb, kb), (cache.vs, vs), (cache.vb, vb)):
            assert np.array_equal(dev_t[r0:r1].float().cpu().numpy(), ref)
        Kd = O.dequantize(O.unpack(kp, w.bits, w.D), ks, kb, w.GS)
        Vd = O.dequantize(O.unpack(vp, w.bits, w.D), vs, vb, w.GS)
        for j in range(w.nrep):
            h = kvh * w.nrep + j
            o = O.attention_head(qv[b, h], Kd, Vd)
            err = np.abs(g[b, h] - o).max()
            tol = {"bf16": 1e-2, "fp16": 1e-2, "fp32": 1e-4}[w.dtype_out] * np.abs(o).max()
            assert err <= tol, f"{w.name} head {(b, h)}: {err:.3e} > {tol:.3e}"
    assert qda.qdecode_attn_device_status() == 0


def test_dispatch_counter_advances():
    before = qda.qdecode_attn_calls()
    check_small(synth.workload(1))
    assert qda.qdecode_attn_calls() == before + 1
