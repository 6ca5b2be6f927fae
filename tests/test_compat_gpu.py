"""GPU parity of the two-pass compat form (qdecode_attn_compat) against the oracle's compat form, through the C ABI.

The compat form rounds every score and every normalised probability to the input dtype T. The GPU forms a score
as an fp32 dot in its own order and a probability with fp32 exponentials, so a value that lies within fp32 rounding
of a T rounding boundary can round to the neighbouring T value on one side only; each such flip moves the output by
about one ulp of T times that row's weight. The result is therefore defined to T's precision, and the tolerance is
the 16-bit rule for every output dtype: max|delta| <= 1e-2 * max|o| per head. Inputs are not peaky (no planted
keys): with scores near 20 one bf16 ulp of a dominant score is a 13 % change of its weight."""
import numpy as np
import pytest
import torch

import oracle as O
import attention_quantized_kv_split_gb300 as qda
from attention_quantized_kv_split_gb300 import build, synth

from harness import TORCH_DT, gpu_quantized_workload, small_case, unit_oracle_cache, upload_cache

pytestmark = pytest.mark.gpu

TOL_COMPAT = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _lib_built():
    build.build()
    qda.lib()
    qda.qdecode_attn_debug_force_splits(0)
    yield
    qda.qdecode_attn_debug_force_splits(0)


def run_compat(q, dev, N, w, out_dtype=None, splits=0):
    out = torch.empty(q.shape, dtype=TORCH_DT[out_dtype or w.dtype_out], device="cuda")
    qda.qdecode_attn_debug_force_splits(splits)
    try:
        qda.qdecode_attn_compat(q.cuda(), *dev, out, N, w.Hkv, w.GS, w.bits)
    finally:
        qda.qdecode_attn_debug_force_splits(0)
    return out


def compare_compat(out, ref):
    g = out.to(torch.float64).cpu().numpy()
    for (b, h), o in ref.items():
        assert np.all(np.isfinite(g[b, h])), (b, h)
        err = np.abs(g[b, h] - o).max()
        bound = TOL_COMPAT * np.abs(o).max()
        assert err <= bound, f"{(b, h)}: max|delta| {err:.3e} > {bound:.3e}"


def check(w, out_dtype=None, splits=0):
    q, cache, N = small_case(w)
    dev = upload_cache(*cache, w.dtype_in)
    out = run_compat(q, dev, N, w, out_dtype, splits)
    ref = O.attention_packed_compat(q.to(torch.float64).numpy(), *cache, N, w.H, w.Hkv, w.D, w.GS, w.bits,
                                    w.dtype_in)
    compare_compat(out, ref)
    return out, (q, dev, N)


SHAPES = [(D, bits, GS) for D in (64, 128, 256, 512) for bits in (4, 8) for GS in (32, 64, 128) if D % GS == 0]


@pytest.mark.parametrize("N", [1, 33, 257, 3000])
@pytest.mark.parametrize("D,bits,GS", SHAPES)
def test_compat_shape_sweep(D, bits, GS, N):
    check(synth.small(B=1, H=4, Hkv=2, D=D, N=(N,), bits=bits, GS=GS, seed=D + bits * 5 + GS + N))


@pytest.mark.parametrize("H,Hkv", [(16, 8), (8, 2), (32, 8), (6, 2), (16, 1)])
def test_compat_gqa(H, Hkv):
    check(synth.small(B=2, H=H, Hkv=Hkv, D=256, N=(700, 90), bits=4, GS=64, seed=H + Hkv))


@pytest.mark.parametrize("dtype_in,dtype_out", [("bf16", "bf16"), ("fp16", "fp16"), ("bf16", "fp32"),
                                                ("fp16", "fp32"), ("fp16", "bf16")])
def test_compat_dtypes(dtype_in, dtype_out):
    check(synth.small(B=2, H=8, Hkv=2, D=512, N=(1200, 64), bits=8, GS=128, dtype_in=dtype_in, seed=17), dtype_out)


@pytest.mark.parametrize("splits", [1, 2, 7, 64, 300])
def test_compat_forced_splits(splits):
    # pass B combines pass A's statistics over every range of a unit, including empty ones at large counts
    check(synth.small(B=3, H=8, Hkv=2, D=256, N=(500, 9, 1500), bits=4, GS=32, seed=splits), splits=splits)


def test_compat_maximum_batch():
    # QDA_MAX_B sequences of 1-6 rows: pass B folds pass A's statistics for 1024 units, most of them inside one range
    N = tuple(1 + (b * 5) % 6 for b in range(512))
    check(synth.small(B=len(N), H=4, Hkv=2, D=256, N=N, bits=8, GS=64, seed=13))


def test_compat_run_to_run_bitwise():
    w = synth.small(B=2, H=16, Hkv=8, D=256, N=(4000, 333), bits=8, GS=32, seed=41)
    out1, (q, dev, N) = check(w)
    for _ in range(3):
        out2 = run_compat(q, dev, N, w)
        torch.cuda.synchronize()
        assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert qda.qdecode_attn_device_status() == 0


def _tied_rows():
    """Two quantized K rows whose scores against q = 16 e_0 (score = dequantised k_0) differ but round to the same
    bf16 value, both well inside that value's rounding interval: found among seeded candidates with the oracle's
    quantizer."""
    rng = np.random.default_rng(7)
    cand = np.zeros((4000, 256), np.float32)
    cand[:, 0] = rng.uniform(0.9, 1.0, 4000).astype(np.float32)
    cand[:, 1:32] = 0.95
    cand[:, 1], cand[:, 2] = 0.9, 1.0          # the first group's range: a code step of ~0.1/255, below a bf16 ulp
    c, sc, bi = O.quantize(cand, 32, 8, "bf16")
    k0 = O.dequantize(c, sc, bi, 32)[:, 0].astype(np.float32).astype(np.float64)
    r = O.round_to(k0.astype(np.float32), "bf16").astype(np.float64)
    ulp = 2.0 ** -8
    inner = np.abs(k0 - r) < 0.25 * ulp        # far from the rounding boundaries (half an ulp away)
    for v in np.unique(r[inner]):
        idx = np.flatnonzero(inner & (r == v))
        vals = k0[idx]
        if vals.max() > vals.min():
            return cand[idx[np.argmin(vals)]], cand[idx[np.argmax(vals)]]
    raise AssertionError("no tied pair among the candidates")


def test_compat_differs_from_exact_softmax_where_rounding_matters():
    # two rows whose scores meet in bf16 but not exactly: compat weighs them equally, the single-pass path does not
    ka, kb = _tied_rows()
    K = np.stack([ka, kb])
    V = np.zeros((2, 256), np.float32)
    V[0, 5], V[1, 5] = 1.0, -1.0
    cache = O.quantize_cache(K, V, 32, 8, "bf16")
    dev = upload_cache(*cache, "bf16")
    q = torch.zeros((1, 1, 256), dtype=torch.bfloat16)
    q[0, 0, 0] = 16.0                       # sqrt(D): the score is the dequantised k_0
    out_c = torch.empty((1, 1, 256), dtype=torch.float32, device="cuda")
    qda.qdecode_attn_compat(q.cuda(), *dev, out_c, [2], 1, 32, 8)
    out_e = torch.empty_like(out_c)
    qda.qdecode_attn(q.cuda(), *dev, out_e, [2], 1, 32, 8)
    torch.cuda.synchronize()
    ref_c = O.attention_packed_compat(q.double().numpy(), *cache, [2], 1, 1, 256, 32, 8, "bf16")[(0, 0)]
    ref_e = O.attention_packed(q.double().numpy(), *cache, [2], 1, 1, 256, 32, 8)[(0, 0)]
    kp, ks, kb, vp, vs, vb = cache
    Vd = O.dequantize(O.unpack(vp, 8, 256), vs, vb, 32)
    even = 0.5 * (Vd[0, 5] + Vd[1, 5])          # both probabilities are T(1/2) = 1/2 exactly
    assert ref_c[5] == even and abs(ref_e[5] - even) > 1e-4
    assert abs(out_c[0, 0, 5].item() - even) <= 1e-6
    assert abs(out_e[0, 0, 5].item() - ref_e[5]) <= 1e-4 * np.abs(ref_e).max()


@pytest.mark.parametrize("D", [64, 128])
def test_compat_small_head_dims_gqa_and_splits(D):
    # D = 64 and 128: 8 or 4 K lanes per row, V rows shared by 8 or 16 lanes
    check(synth.small(B=2, H=24, Hkv=3, D=D, N=(900, 50), bits=8, GS=32, seed=D))
    check(synth.small(B=2, H=8, Hkv=2, D=D, N=(300, 77), bits=4, GS=32, dtype_in="fp16", seed=D + 1), "fp32",
          splits=37)


def test_compat_8k_workload_sampled():
    w = synth.workload(2)
    q, cache, N = gpu_quantized_workload(w)
    out = torch.empty((w.B, w.H, w.D), dtype=TORCH_DT[w.dtype_out], device="cuda")
    qda.qdecode_attn_compat(q.cuda(), cache.kp, cache.ks, cache.kb, cache.vp, cache.vs, cache.vb, out, N, w.Hkv,
                            w.GS, w.bits)
    torch.cuda.synchronize()
    nrep = w.H // w.Hkv
    for kvh in (0, 3, 7):
        unit = unit_oracle_cache(w, 0, kvh, N, q)
        qs = q[:, kvh * nrep:(kvh + 1) * nrep].to(torch.float64).numpy()
        ref = O.attention_packed_compat(qs, *unit, [N[0]], nrep, 1, w.D, w.GS, w.bits, w.dtype_in)
        compare_compat(out[:, kvh * nrep:(kvh + 1) * nrep], ref)
    assert qda.qdecode_attn_device_status() == 0


def _clear_of_midpoints(p, dtype, margin):
    """True when every probability p (fp64, > 0) lies farther than margin * p from the midpoint between the two
    `dtype` values around it: any value within that relative distance of p rounds to the same `dtype` value (the
    fp32 step the oracle takes first moves p by 2^-24 of itself, far less)."""
    r = O.round_to(p.astype(np.float32), dtype)
    pat = O.bits16(r, dtype).astype(np.int64)                       # positive values: patterns increase with value
    r = r.astype(np.float64)
    other = O.from_bits16(np.where(r > p, pat - 1, pat + 1).astype(np.uint16), dtype).astype(np.float64)
    mid = 0.5 * (r + other)
    return bool(np.all(np.abs(p - mid) > margin * p))


def _exact_score_case(D, bits, GS, N, dtype, seed, margin):
    """Two query heads whose scores are exact in `dtype`: the first group of every K row is quantized with scale
    step (a power of two) and bias 0 (its minimum 0 and maximum (2^bits - 1) * step are planted at d = 1, 2), and
    head j's q is sqrt(D) at d = 4 j, so its score is the row's dequantised k_{4j} = code * step -- a value with at
    most 8 significant bits, the same on every side. Seeds are tried in turn until no probability of either head
    lies within `margin` of a rounding midpoint of `dtype` (oracle values): then every rounding decision of the
    compat form is the same on the GPU as in the oracle."""
    top = 2 ** bits - 1
    step = 2.0 ** -6 if bits == 8 else 2.0 ** -4
    for s in range(seed, seed + 200):
        rng = np.random.default_rng(s)
        K = rng.uniform(0.0, top * step, (N, D)).astype(np.float32)
        K[:, 1], K[:, 2] = 0.0, top * step
        K[:, 0] = rng.integers(0, top + 1, N) * step
        K[:, 4] = rng.integers(0, top + 1, N) * step
        V = rng.standard_normal((N, D)).astype(np.float32)
        cache = O.quantize_cache(K, V, GS, bits, dtype)
        kp, ks, kb = cache[:3]
        Kd = O.dequantize(O.unpack(kp, bits, D), ks, kb, GS)
        clear = True
        for j in range(2):
            sc = Kd[:, 4 * j].astype(np.float64)
            assert np.array_equal(sc, O.round_to(sc.astype(np.float32), dtype)), "scores exact in the input dtype"
            e = np.exp(sc - sc.max())
            clear = clear and _clear_of_midpoints(e / e.sum(), dtype, margin)
        if clear:
            q = torch.zeros((1, 2, D), dtype=TORCH_DT[dtype])
            q[0, 0, 0] = q[0, 1, 4] = float(np.sqrt(D))
            return q, cache
    raise AssertionError("no seed without a probability near a rounding midpoint")


@pytest.mark.parametrize("dtype_in,D,bits,GS,N,splits", [("bf16", 256, 8, 32, 64, 0), ("bf16", 256, 4, 64, 96, 3),
                                                         ("fp16", 64, 8, 32, 24, 0), ("fp16", 256, 4, 32, 40, 2)])
def test_compat_fp32_output_exact_where_no_rounding_is_ambiguous(dtype_in, D, bits, GS, N, splits):
    # Where no score and no probability sits near a rounding boundary of the input dtype, the compat form has no
    # rounding flips, so its fp32 output is held to the fp32 tolerance of the single-pass path, not the 16-bit rule.
    # The margin 2^-15 (3.1e-5) is four times a worst-case bound on the GPU's relative error in a probability here,
    # about 7e-6: the fp32 products of exact scores (|s| <= 4) with log2 e, the fp32 exp2, and fp32 sums of at most
    # 96 terms for the denominator.
    q, cache = _exact_score_case(D, bits, GS, N, dtype_in, seed=100 * D + 10 * bits + N, margin=2.0 ** -15)
    dev = upload_cache(*cache, dtype_in)
    out = torch.empty((1, 2, D), dtype=torch.float32, device="cuda")
    qda.qdecode_attn_debug_force_splits(splits)
    try:
        qda.qdecode_attn_compat(q.cuda(), *dev, out, [N], 1, GS, bits)
    finally:
        qda.qdecode_attn_debug_force_splits(0)
    torch.cuda.synchronize()
    ref = O.attention_packed_compat(q.to(torch.float64).numpy(), *cache, [N], 2, 1, D, GS, bits, dtype_in)
    g = out.to(torch.float64).cpu().numpy()
    for (b, h), o in ref.items():
        err = np.abs(g[b, h] - o).max()
        assert err <= 1e-4 * np.abs(o).max(), f"head {h}: max|delta| {err:.3e} > {1e-4 * np.abs(o).max():.3e}"
    assert qda.qdecode_attn_device_status() == 0
