"""Pins for the CPU oracle: it is checked against closed forms, hand-written examples, library routines, brute force
and invariants of the mathematics, never against itself. CPU only."""
import math
import os

import numpy as np
import pytest
import torch

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------------------------------ dtype rounding


def test_round_to_bf16_ties_to_even():
    # 1 + 2^-8 is halfway between bf16 neighbours 1 and 1 + 2^-7: ties go to the even mantissa (1.0);
    # 1 + 3*2^-8 is halfway between 1 + 2^-7 and 1 + 2^-6: goes to 1 + 2^-6.
    x = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -8 + 2 ** -20, -(1 + 2 ** -8)], np.float32)
    assert O.round_to(x, "bf16").tolist() == [1.0, 1 + 2 ** -6, 1 + 2 ** -7, -1.0]


def test_round_to_fp16_ties_to_even():
    # fp16 has 10 fraction bits: 1 + 2^-11 is a tie -> 1.0; 1 + 3*2^-11 -> 1 + 2^-9
    x = np.array([1 + 2 ** -11, 1 + 3 * 2 ** -11, 2049.0, 2051.0], np.float32)
    assert O.round_to(x, "fp16").tolist() == [1.0, 1 + 2 ** -9, 2048.0, 2052.0]


def test_bits16_roundtrip_and_known_patterns():
    assert O.bits16(np.array([1.0, -2.0], np.float32), "bf16").tolist() == [0x3F80, 0xC000]
    assert O.bits16(np.array([1.0, -2.0], np.float32), "fp16").tolist() == [0x3C00, 0xC000]
    v = O.round_to(np.random.default_rng(0).standard_normal(1000).astype(np.float32), "bf16")
    assert np.array_equal(O.from_bits16(O.bits16(v, "bf16"), "bf16"), v)


# ------------------------------------------------------------------------------------------ pack / unpack


def _golden_pack():
    rows = []
    with open(os.path.join(GOLDEN, "pack_examples.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            bits, codes, word = (p.strip() for p in line.split("|"))
            rows.append((int(bits), [int(c) for c in codes.split()], int(word, 16)))
    return rows


@pytest.mark.parametrize("bits,codes,word", _golden_pack())
def test_pack_golden(bits, codes, word):
    w = O.pack(np.array(codes, np.uint32), bits)
    assert w.tolist() == [word]
    assert O.unpack(np.array([word], np.uint32), bits, len(codes)).tolist() == codes


@pytest.mark.parametrize("bits", [4, 8])
def test_pack_roundtrip_random_words(bits):
    # random words -> codes -> words must be the identity (bit-exact) over 1e6 words
    rng = np.random.default_rng(bits)
    per = 32 // bits
    words = rng.integers(0, 2 ** 32, size=(1000, 1000), dtype=np.uint64).astype(np.uint32)
    codes = O.unpack(words, bits, 1000 * per)
    assert codes.max() < 2 ** bits
    assert np.array_equal(O.pack(codes, bits), words)


def test_pack_bit_positions_one_hot():
    # every single code position lands on its own bit field
    for bits in (4, 8):
        per = 32 // bits
        for i in range(per):
            c = np.zeros(per, np.uint32)
            c[i] = 1
            assert O.pack(c, bits)[0] == 1 << (bits * i)


# ------------------------------------------------------------------------------------------ quantizer


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("GS", [32, 64, 128])
def test_quantize_closed_form_4bit(dtype, GS):
    # a group holding integers with min -1 and max 14: scale (14 - -1)/15 = 1 and bias -1 exactly,
    # every code is x + 1, the min maps to 0 and the max to 15
    rng = np.random.default_rng(GS)
    x = rng.integers(-1, 15, size=(3, GS)).astype(np.float32)
    x[:, 0], x[:, 1] = -1, 14
    c, s, b = O.quantize(x, GS, 4, dtype)
    assert s.tolist() == [[1.0]] * 3 and b.tolist() == [[-1.0]] * 3
    assert np.array_equal(c, (x + 1).astype(np.uint32))
    assert np.array_equal(O.dequantize(c, s, b, GS), x.astype(np.float64))


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_quantize_closed_form_8bit(dtype):
    # integers 0..255 with scale 255/255 = 1 and bias 0: codes are the values themselves
    x = np.arange(256, dtype=np.float32).reshape(8, 32)[::-1].copy()
    x[:, 0], x[:, 1] = 0, 255
    c, s, b = O.quantize(x, 32, 8, dtype)
    assert np.all(s == 1.0) and np.all(b == 0.0)
    assert np.array_equal(c, x.astype(np.uint32))


def test_quantize_scale_is_range_over_levels():
    # a two-value group {0, 3}: 4-bit scale 3/15 = 0.2 (rounded to bf16), 8-bit 3/255
    x = np.zeros((1, 32), np.float32)
    x[0, 5] = 3.0
    _, s4, b4 = O.quantize(x, 32, 4, "bf16")
    _, s8, _ = O.quantize(x, 32, 8, "fp16")
    assert s4[0, 0] == torch.tensor(0.2).to(torch.bfloat16).float().item()
    assert s8[0, 0] == torch.tensor(3.0 / 255.0).to(torch.float16).float().item()
    assert b4[0, 0] == 0.0


def test_quantize_zero_range_group():
    x = np.full((2, 64), 0.3, np.float32)
    c, s, b = O.quantize(x, 64, 4, "bf16")
    assert np.all(c == 0) and np.all(s == 0)
    assert np.all(b == np.float32(torch.tensor(0.3).to(torch.bfloat16).float().item()))


def test_quantize_rounds_half_to_even():
    # scale 1, bias 0; values 0.5, 1.5, 2.5 sit on ties -> codes 0, 2, 2
    x = np.zeros((1, 32), np.float32)
    x[0, :4] = [0.0, 0.5, 1.5, 2.5]
    x[0, 4] = 15.0
    c, s, b = O.quantize(x, 32, 4, "bf16")
    assert s[0, 0] == 1.0 and b[0, 0] == 0.0
    assert c[0, :4].tolist() == [0, 0, 2, 2]


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_quantize_error_bound(bits, dtype):
    # |x - x_hat| <= s_hat/2 plus what rounding the scale and bias to 16 bits can add at the clamped ends,
    # and the bound is nearly reached (a floor instead of a round would break the first, a coarser grid the second)
    rng = np.random.default_rng(3)
    GS = 64
    x = rng.standard_normal((512, 4 * GS)).astype(np.float32)
    c, s, b = O.quantize(x, GS, bits, dtype)
    xh = O.dequantize(c, s, b, GS).reshape(512, 4, GS)
    g = x.reshape(512, 4, GS).astype(np.float64)
    lo, hi = g.min(-1), g.max(-1)
    qmax = 2 ** bits - 1
    exact_scale = (hi - lo) / qmax
    slack = qmax * np.abs(s - exact_scale) + np.abs(b - lo) + 1e-6 * np.abs(g).max(-1)
    err = np.abs(xh - g).max(-1)
    assert np.all(err <= s / 2 + slack)
    assert np.median(err / s) > 0.4


# ------------------------------------------------------------------------------------------ attention


def _softmax_loop(q, K, V):
    # brute force with Python floats and math.exp: an independent restatement of softmax(q.K^T/sqrt(D)).V
    D = len(q)
    s = [sum(q[d] * K[n][d] for d in range(D)) / math.sqrt(D) for n in range(len(K))]
    m = max(s)
    e = [math.exp(v - m) for v in s]
    z = sum(e)
    return [sum(e[n] * V[n][d] for n in range(len(K))) / z for d in range(D)]


@pytest.mark.parametrize("D", [32, 64])
@pytest.mark.parametrize("N", [1, 2, 5, 8])
def test_attention_brute_force_tiny(D, N):
    rng = np.random.default_rng(N * 100 + D)
    H, Hkv, GS, bits = 4, 2, 32, 4
    q = O.round_to(rng.standard_normal((H, D)).astype(np.float32), "bf16").astype(np.float64)
    Kx = rng.standard_normal((Hkv, N, D)).astype(np.float32)
    Vx = rng.standard_normal((Hkv, N, D)).astype(np.float32)
    kc, ks, kb = O.quantize(Kx, GS, bits, "bf16")
    vc, vs, vb = O.quantize(Vx, GS, bits, "bf16")
    K = O.dequantize(kc, ks, kb, GS)
    V = O.dequantize(vc, vs, vb, GS)
    out = O.attention(q, K, V)
    # library routine: scaled_dot_product_attention in fp64 on the dequantized arrays (its default scale is
    # 1/sqrt(D)); GQA by repeating each KV head over its group of query heads
    nrep = H // Hkv
    Kr = torch.from_numpy(np.repeat(K, nrep, axis=0))[:, None]
    Vr = torch.from_numpy(np.repeat(V, nrep, axis=0))[:, None]
    ref = torch.nn.functional.scaled_dot_product_attention(torch.from_numpy(q)[:, None, None], Kr, Vr)
    np.testing.assert_allclose(out, ref[:, 0, 0].numpy(), rtol=1e-12, atol=1e-12)
    for h in range(H):
        loop = _softmax_loop(q[h].tolist(), K[h // nrep].tolist(), V[h // nrep].tolist())
        np.testing.assert_allclose(out[h], loop, rtol=1e-11, atol=1e-12)


def test_attention_scale_closed_form():
    # two keys, k0 = 0 and k1 = c*e_0; with q = e_0 the weights are 1 : e^(c/sqrt(D))
    D, c = 64, 3.0
    q = np.zeros(D)
    q[0] = 1.0
    K = np.zeros((2, D))
    K[1, 0] = c
    V = np.zeros((2, D))
    V[0, 1], V[1, 1] = 1.0, 0.0
    w = math.exp(c / math.sqrt(D))
    out = O.attention_head(q, K, V)
    assert abs(out[1] - 1.0 / (1.0 + w)) < 1e-15


def test_attention_all_equal_scores_is_mean_of_v():
    rng = np.random.default_rng(11)
    N, D = 97, 64
    row = rng.standard_normal(D)
    K = np.tile(row, (N, 1))
    V = rng.standard_normal((N, D))
    q = rng.standard_normal(D)
    np.testing.assert_allclose(O.attention_head(q, K, V), V.mean(0), rtol=1e-12, atol=1e-13)


def test_attention_one_hot_dominant_key():
    rng = np.random.default_rng(12)
    N, D = 64, 64
    q = np.zeros(D)
    q[3] = 1.0
    K = rng.standard_normal((N, D)) * 0.01
    j = 17
    K[j, 3] = 60.0 * math.sqrt(D) + 1.0          # score margin >= 60 over every other key
    V = rng.uniform(-1, 1, (N, D))
    out = O.attention_head(q, K, V)
    assert np.abs(out - V[j]).max() < N * math.exp(-60) * 2


@pytest.mark.parametrize("S", [1, 2, 3, 7, 40])
def test_blocked_equals_unblocked(S):
    rng = np.random.default_rng(S)
    N, D = 40, 64
    q = rng.standard_normal(D) * 3
    K = rng.standard_normal((N, D))
    V = rng.standard_normal((N, D))
    ref = O.attention_head(q, K, V)
    blk = O.attention_blocked(q, K, V, S)
    assert np.abs(blk - ref).max() <= 1e-12 * np.abs(ref).max()


def test_factored_dot_identity():
    # sum_d (s*c_d + b) q_d == s * sum_d c_d q_d + b * sum_d q_d per group (the dequant factored out of the dot)
    rng = np.random.default_rng(5)
    D, GS = 256, 64
    x = rng.standard_normal((16, D)).astype(np.float32)
    c, s, b = O.quantize(x, GS, 4, "bf16")
    q = rng.standard_normal(D)
    direct = O.dequantize(c, s, b, GS) @ q
    cg = c.reshape(16, D // GS, GS).astype(np.float64)
    qg = q.reshape(D // GS, GS)
    factored = (s * (cg * qg).sum(-1) + b * qg.sum(-1)).sum(-1)
    np.testing.assert_allclose(direct, factored, rtol=1e-12, atol=1e-12)


def test_gqa_head_map_is_contiguous():
    # kv head j serves query heads j*nrep .. j*nrep + nrep - 1 (not h % Hkv)
    H, Hkv, N, D = 8, 2, 5, 32
    q = np.random.default_rng(0).standard_normal((H, D))
    K = np.zeros((Hkv, N, D))
    V = np.stack([np.full((N, D), 1.0), np.full((N, D), 2.0)])
    out = O.attention(q, K, V)
    assert np.all(out[:4] == 1.0) and np.all(out[4:] == 2.0)


def test_packed_interface_ragged_layout():
    # sequences back to back, [Hkv, N[b], .] each: the packed path must agree with per-sequence dequantized math
    rng = np.random.default_rng(9)
    N = [3, 7, 1]
    B, H, Hkv, D, GS, bits = 3, 4, 2, 64, 32, 8
    rows = Hkv * sum(N)
    Kx = rng.standard_normal((rows, D)).astype(np.float32)
    Vx = rng.standard_normal((rows, D)).astype(np.float32)
    kp, ks, kb, vp, vs, vb = O.quantize_cache(Kx, Vx, GS, bits, "fp16")
    q = rng.standard_normal((B, H, D))
    got = O.attention_packed(q, kp, ks, kb, vp, vs, vb, N, H, Hkv, D, GS, bits)
    r = 0
    for b, n in enumerate(N):
        Kb = np.stack([O.dequantize(*O.quantize(Kx[r + j * n: r + (j + 1) * n], GS, bits, "fp16"), GS)
                       for j in range(Hkv)])
        Vb = np.stack([O.dequantize(*O.quantize(Vx[r + j * n: r + (j + 1) * n], GS, bits, "fp16"), GS)
                       for j in range(Hkv)])
        ref = O.attention(q[b], Kb, Vb)
        for h in range(H):
            np.testing.assert_array_equal(got[(b, h)], ref[h])
        r += Hkv * n
    assert r == rows


# ----------------------------------------------------------------------- small-L multi-query decode (L queries)


def test_visible_rows_closed_form():
    # the L new tokens are the last L cache rows; position l sees rows 0 .. n - L + l
    assert [O.visible_rows(10, 3, l) for l in range(3)] == [8, 9, 10]
    assert O.visible_rows(5, 1, 0) == 5
    assert [O.visible_rows(4, 4, l) for l in range(4)] == [1, 2, 3, 4]
    for bad in ((3, 4, 0), (5, 2, 2), (5, 0, 0), (5, 2, -1)):
        with pytest.raises(ValueError):
            O.visible_rows(*bad)


def _multi_case(seed, N, L, H, Hkv, D, GS, bits, dtype="bf16"):
    rng = np.random.default_rng(seed)
    rows = Hkv * sum(N)
    Kx = rng.standard_normal((rows, D)).astype(np.float32)
    Vx = rng.standard_normal((rows, D)).astype(np.float32)
    cache = O.quantize_cache(Kx, Vx, GS, bits, dtype)
    q = O.round_to(rng.standard_normal((len(N), L, H, D)).astype(np.float32), dtype).astype(np.float64)
    return q, cache, Kx, Vx


def test_multi_query_matches_masked_sdpa():
    # library routine with an explicit causal mask over the whole window, instead of truncating the rows
    N, L, H, Hkv, D, GS, bits = [6, 9], 3, 4, 2, 32, 32, 4
    q, cache, _, _ = _multi_case(21, N, L, H, Hkv, D, GS, bits)
    got = O.attention_packed_multi(q, *cache, N, L, H, Hkv, D, GS, bits)
    kp, ks, kb, vp, vs, vb = cache
    nrep = H // Hkv
    for b, n in enumerate(N):
        mask = torch.tensor([[k <= n - L + l for k in range(n)] for l in range(L)])
        for h in range(H):
            r0, r1 = O.unit_rows(N, Hkv, b, h // nrep)
            K = torch.from_numpy(O.dequantize(O.unpack(kp[r0:r1], bits, D), ks[r0:r1], kb[r0:r1], GS))
            V = torch.from_numpy(O.dequantize(O.unpack(vp[r0:r1], bits, D), vs[r0:r1], vb[r0:r1], GS))
            ref = torch.nn.functional.scaled_dot_product_attention(torch.from_numpy(q[b, :, h]), K, V, attn_mask=mask)
            for l in range(L):
                np.testing.assert_allclose(got[(b, l, h)], ref[l].numpy(), rtol=1e-12, atol=1e-12)


def test_multi_query_last_position_is_single_query():
    # the last position sees the whole window: single-query decode over the same cache
    N, L, H, Hkv, D, GS, bits = [5, 12], 4, 8, 2, 64, 32, 8
    q, cache, _, _ = _multi_case(22, N, L, H, Hkv, D, GS, bits, "fp16")
    got = O.attention_packed_multi(q, *cache, N, L, H, Hkv, D, GS, bits)
    ref = O.attention_packed(q[:, L - 1], *cache, N, H, Hkv, D, GS, bits)
    for b in range(len(N)):
        for h in range(H):
            np.testing.assert_array_equal(got[(b, L - 1, h)], ref[(b, h)])


def test_multi_query_ignores_rows_after_own_position():
    # changing row n - L + l + 1 of a unit changes what position l + 1 sees but not position l
    N, L, H, Hkv, D, GS, bits = [10], 3, 2, 1, 32, 32, 4
    q, cache, Kx, Vx = _multi_case(23, N, L, H, Hkv, D, GS, bits)
    base = O.attention_packed_multi(q, *cache, N, L, H, Hkv, D, GS, bits)
    for l in range(L - 1):
        row = N[0] - L + l + 1
        K2, V2 = Kx.copy(), Vx.copy()
        K2[row] *= -3.0
        V2[row] += 5.0
        alt = O.attention_packed_multi(q, *O.quantize_cache(K2, V2, GS, bits, "bf16"), N, L, H, Hkv, D, GS, bits)
        for h in range(H):
            np.testing.assert_array_equal(alt[(0, l, h)], base[(0, l, h)])
            assert np.abs(alt[(0, l + 1, h)] - base[(0, l + 1, h)]).max() > 1e-3


# ------------------------------------------------------------------ two-pass variant with compat rounding points


@pytest.mark.parametrize("dtype,third", [("bf16", 0.333984375), ("fp16", 0.333251953125)])
def test_compat_equal_scores_weights_are_rounded_thirds(dtype, third):
    # three equal scores: each probability is T(1/3) (not renormalised), so o = T(1/3) * (v0 + v1 + v2)
    rng = np.random.default_rng(31)
    D = 64
    K = np.tile(rng.standard_normal(D), (3, 1))
    V = rng.standard_normal((3, D))
    q = rng.standard_normal(D)
    out = O.attention_head_compat(q, K, V, dtype)
    np.testing.assert_allclose(out, third * V.sum(0), rtol=1e-15, atol=1e-15)


def test_compat_scores_round_before_the_softmax():
    # scores 1 and 1 + 2^-10 are one value in bf16 (ulp 2^-7 at 1): equal weights 1/2, unlike the exact softmax;
    # in fp16 (ulp 2^-10 at 1) they stay apart
    D = 64
    q = np.zeros(D)
    q[0] = 8.0                                  # sqrt(D): score = K[:, 0]
    K = np.zeros((2, D))
    K[0, 0], K[1, 0] = 1.0, 1.0 + 2.0 ** -10
    V = np.zeros((2, D))
    V[0, 1], V[1, 1] = 1.0, -1.0
    assert O.attention_head_compat(q, K, V, "bf16")[1] == 0.0
    w = math.exp(2.0 ** -10)
    p0, p1 = O.round_to(np.array([1 / (1 + w), w / (1 + w)], np.float32), "fp16").astype(np.float64)
    assert O.attention_head_compat(q, K, V, "fp16")[1] == p0 - p1 != 0.0
    assert abs(O.attention_head(q, K, V)[1] - (1 - w) / (1 + w)) < 1e-15


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_compat_matches_library_softmax_with_casts(dtype):
    # the same rounding points through torch: fp64 scores cast to fp32 then T, torch.softmax, cast, matmul
    rng = np.random.default_rng(32)
    N, D = 50, 128
    q = rng.standard_normal(D)
    K = rng.standard_normal((N, D))
    V = rng.standard_normal((N, D))
    T = {"bf16": torch.bfloat16, "fp16": torch.float16}[dtype]
    s = (torch.from_numpy(K) @ torch.from_numpy(q) / math.sqrt(D)).float().to(T).double()
    p = torch.softmax(s, 0).float().to(T).double()
    ref = (p @ torch.from_numpy(V)).numpy()
    np.testing.assert_allclose(O.attention_head_compat(q, K, V, dtype), ref, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("S", [1, 2, 3, 7, 40])
def test_two_pass_blocked_equals_direct(S):
    rng = np.random.default_rng(33 + S)
    N, D = 40, 64
    q = rng.standard_normal(D) * 2
    K = rng.standard_normal((N, D))
    V = rng.standard_normal((N, D))
    for dtype in ("bf16", "fp16"):
        ref = O.attention_head_compat(q, K, V, dtype)
        blk = O.attention_two_pass_blocked(q, K, V, S, dtype)
        assert np.abs(blk - ref).max() <= 1e-12 * np.abs(ref).max()


def test_compat_packed_interface():
    rng = np.random.default_rng(34)
    N = [4, 9]
    B, H, Hkv, D, GS, bits = 2, 4, 2, 64, 32, 4
    rows = Hkv * sum(N)
    Kx = rng.standard_normal((rows, D)).astype(np.float32)
    Vx = rng.standard_normal((rows, D)).astype(np.float32)
    cache = O.quantize_cache(Kx, Vx, GS, bits, "bf16")
    q = rng.standard_normal((B, H, D))
    got = O.attention_packed_compat(q, *cache, N, H, Hkv, D, GS, bits, "bf16")
    kp, ks, kb, vp, vs, vb = cache
    for b in range(B):
        for h in range(H):
            r0, r1 = O.unit_rows(N, Hkv, b, h // 2)
            K = O.dequantize(O.unpack(kp[r0:r1], bits, D), ks[r0:r1], kb[r0:r1], GS)
            V = O.dequantize(O.unpack(vp[r0:r1], bits, D), vs[r0:r1], vb[r0:r1], GS)
            np.testing.assert_array_equal(got[(b, h)], O.attention_head_compat(q[b, h], K, V, "bf16"))


# --------------------------------------------------------------- affine-quantized weight GEMV (comparison workload)


def test_qgemv_closed_form_integer_codes():
    # a group [0, 1, ..., GS-1] repeated: scale 1, bias 0, codes = the integers; x = 1 gives the row sums
    K, GS, N = 256, 64, 3
    row = np.tile(np.arange(GS, dtype=np.float32) * (255 / (GS - 1)), K // GS)
    row = np.round(row)                                 # integers 0..255 with min 0 and max 255
    w = np.stack([row] * N).astype(np.float32)
    c, s, b = O.quantize(w, GS, 8, "bf16")
    assert np.all(s == 1.0) and np.all(b == 0.0)
    y = O.qgemv(np.ones((2, K)), O.pack(c, 8), s, b, K, GS, 8)
    np.testing.assert_array_equal(y, np.full((2, N), row.sum()))


def test_qgemv_bias_only_rows():
    # all codes 0: y[t, n] = sum_g b[n, g] * sum_{k in g} x[t, k]
    rng = np.random.default_rng(41)
    T, N, K, GS = 3, 5, 128, 32
    wp = np.zeros((N, K * 4 // 32), np.uint32)
    ws = rng.uniform(0.1, 1, (N, K // GS))
    wb = rng.standard_normal((N, K // GS))
    x = rng.standard_normal((T, K))
    y = O.qgemv(x, wp, ws, wb, K, GS, 4)
    ref = np.einsum("ng,tg->tn", wb, x.reshape(T, K // GS, GS).sum(-1))
    np.testing.assert_allclose(y, ref, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("bits", [4, 8])
def test_qgemv_brute_force_loops(bits):
    rng = np.random.default_rng(42 + bits)
    T, N, K, GS = 2, 3, 64, 32
    w = rng.standard_normal((N, K)).astype(np.float32)
    c, s, b = O.quantize(w, GS, bits, "fp16")
    x = rng.standard_normal((T, K))
    y = O.qgemv(x, O.pack(c, bits), s, b, K, GS, bits)
    for t in range(T):
        for n in range(N):
            ref = sum(float(x[t, k]) * (float(c[n, k]) * float(s[n, k // GS]) + float(b[n, k // GS])) for k in range(K))
            assert abs(y[t, n] - ref) <= 1e-12 * max(1.0, abs(ref))


# ------------------------------------------------------------------------------------ appending to the cache


@pytest.mark.parametrize("bits,GS,dtype", [(4, 32, "bf16"), (8, 64, "fp16"), (4, 128, "fp16")])
def test_cache_append_equals_quantizing_the_longer_cache(bits, GS, dtype):
    # the quantizer works row by row, so appending quantized rows equals quantizing the concatenated rows
    rng = np.random.default_rng(51 + bits)
    N, Hkv, T, D = [5, 0, 12], 2, 3, 128
    B = len(N)
    old_k = [rng.standard_normal((Hkv, n, D)).astype(np.float32) for n in N]
    old_v = [rng.standard_normal((Hkv, n, D)).astype(np.float32) for n in N]
    Kn = rng.standard_normal((B, Hkv, T, D)).astype(np.float32)
    Vn = rng.standard_normal((B, Hkv, T, D)).astype(np.float32)
    flat = lambda xs: np.concatenate([x.reshape(-1, D) for x in xs])
    old = O.quantize_cache(flat(old_k), flat(old_v), GS, bits, dtype)
    got = O.cache_append(old, N, Kn, Vn, Hkv, D, GS, bits, dtype)
    long_k = [np.concatenate([old_k[b], Kn[b]], axis=1) for b in range(B)]
    long_v = [np.concatenate([old_v[b], Vn[b]], axis=1) for b in range(B)]
    ref = O.quantize_cache(flat(long_k), flat(long_v), GS, bits, dtype)
    for g, r in zip(got, ref):
        np.testing.assert_array_equal(g, r)


def test_cache_append_attention_sees_the_new_rows():
    # decode over the appended cache with L = T query positions equals decode over the longer fp32 rows
    rng = np.random.default_rng(52)
    N, Hkv, T, D, GS, bits, H = [7, 3], 1, 2, 64, 32, 8, 2
    B = len(N)
    old_k = rng.standard_normal((sum(N) * Hkv, D)).astype(np.float32)
    old_v = rng.standard_normal((sum(N) * Hkv, D)).astype(np.float32)
    Kn = rng.standard_normal((B, Hkv, T, D)).astype(np.float32)
    Vn = rng.standard_normal((B, Hkv, T, D)).astype(np.float32)
    new = O.cache_append(O.quantize_cache(old_k, old_v, GS, bits, "bf16"), N, Kn, Vn, Hkv, D, GS, bits, "bf16")
    N2 = [n + T for n in N]
    q = rng.standard_normal((B, T, H, D))
    out = O.attention_packed_multi(q, *new, N2, T, H, Hkv, D, GS, bits)
    kp, ks, kb, vp, vs, vb = new
    for b in range(B):
        r0, r1 = O.unit_rows(N2, Hkv, b, 0)
        Kd = O.dequantize(O.unpack(kp[r0:r1], bits, D), ks[r0:r1], kb[r0:r1], GS)
        Vd = O.dequantize(O.unpack(vp[r0:r1], bits, D), vs[r0:r1], vb[r0:r1], GS)
        for t in range(T):
            for h in range(H):
                np.testing.assert_array_equal(out[(b, t, h)], O.attention_head(q[b, t, h], Kd[:N[b] + 1 + t], Vd[:N[b] + 1 + t]))
