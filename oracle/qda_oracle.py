"""Plain, slow CPU oracle for single-query decode attention over an affine-quantized KV cache.

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import or call anything in this package. The GPU library never does, and this file imports nothing from it.

What it computes, step by step, in the order of the method's description:

1. ``quantize``: per group of GS consecutive elements along D, an MLX-style min/max affine quantizer
   (maya-mac ``mlx_kernels.py``, ``_linear_kernel`` 8-bit weight load: ``w = q * scale + bias``; the
   configuration text fixes ``scale = (max - min) / (2^bits - 1)``, ``bias = min``).
2. ``pack`` / ``unpack``: codes packed LSB-first into uint32 words, ``32 / bits`` codes per word
   (maya-mac ``_linear_kernel``: byte j of a word is ``(a >> 8j) & 0xff``; mlx-bun
   ``fused-decode-kernel.ts`` SCORE_ROW: nibble k of a 16-bit read sits at bits 4k..4k+3).
3. ``dequantize``: ``x_hat = scale * code + bias`` in fp64.
4. ``attention``: per (sequence b, query head h), with KV head ``h // (H / Hkv)``
   (``fused-decode-kernel.ts`` SCORE_PREAMBLE, ``kv = h / NREP``), scores ``q . k_hat / sqrt(D)``
   (maya-mac ``_ATTEND``/``attend``: ``head_dim ** -0.5``), a max-subtracted softmax over all N rows (decode
   attends the whole window: ``fusedDecodeSdpa``), and the probability-weighted sum of the V rows.
5. ``attention_blocked``: the same result through per-block (max, sum-exp, unnormalised o) statistics and the
   merge ``out = sum_g o_g e^(m_g - M) / sum_g l_g e^(m_g - M)`` (``fused-decode-kernel.ts`` BLOCK_SOURCE and
   MERGE_SOURCE), used only to check that splitting the rows does not change the result.
6. ``attention_packed_multi``: L query positions per sequence (the last L tokens, already in the cache), each
   attending the rows up to its own (``visible_rows``); L = 1 is step 4.
7. ``attention_head_compat`` / ``attention_two_pass_blocked`` / ``attention_packed_compat``: the two-pass variant
   with the pages' compat rounding points (scores and normalised probabilities rounded to the input dtype T).
8. ``qgemv``: the same affine codec under a plain matrix-vector product (a comparison workload).
9. ``cache_append``: the step before decode: every KV head's old rows, then the new tokens' rows quantized.

Readings taken where the pages are silent (each pinned by a test in ``tests/test_oracle.py``):

* the scale and bias are computed in fp32 from fp32 data and stored rounded (RNE) to the q dtype (bf16 or fp16);
* a code is ``clamp(rint((x - b_hat) / s_hat), 0, 2^bits - 1)`` with every operation in IEEE fp32 and
  round-half-to-even; a group whose stored scale is 0 gets code 0;
* the attention itself is exact fp64 on the dequantized values; no intermediate is rounded to bf16/fp16
  (except in the compat form of step 7, which rounds where the pages' two-pass kernels do);
* with L query positions per sequence, position l attends the first N - L + 1 + l rows (causal among the L
  new tokens, which are the last L rows of the cache).

Layouts match the GPU library's: q ``[B, H, D]``; per sequence b (back to back, no padding) the packed cache is
``[Hkv, N[b], D*bits/32]`` uint32 and the scales and biases ``[Hkv, N[b], D/GS]``.
"""
from __future__ import annotations

import math

import numpy as np
import torch

DTYPES = ("bf16", "fp16", "fp32")
_TORCH = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}


def round_to(x, dtype: str) -> np.ndarray:
    """Round fp32 values to the nearest ``dtype`` value (ties to even); returned as fp32 holding those values."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(_TORCH[dtype]).to(torch.float32).numpy()


def bits16(x, dtype: str) -> np.ndarray:
    """Raw 16-bit patterns (uint16) of values already representable in ``dtype`` (bf16 or fp16)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(_TORCH[dtype])
    return t.view(torch.int16).numpy().view(np.uint16)


def from_bits16(b, dtype: str) -> np.ndarray:
    """fp32 values of raw bf16/fp16 bit patterns."""
    t = torch.from_numpy(np.ascontiguousarray(b, dtype=np.uint16).view(np.int16)).view(_TORCH[dtype])
    return t.to(torch.float32).numpy()


# ----------------------------------------------------------------------------------------------- quantizer


def quantize(x, GS: int, bits: int, dtype: str):
    """Affine min/max quantization of the last axis in groups of GS.

    Returns ``(codes uint32 [..., D], s_hat fp32 [..., D/GS], b_hat fp32 [..., D/GS])``; ``s_hat`` and ``b_hat``
    hold values exactly representable in ``dtype``. Every float step is IEEE fp32.
    """
    x = np.asarray(x, dtype=np.float32)
    D = x.shape[-1]
    if D % GS:
        raise ValueError("D must be a multiple of GS")
    g = x.reshape(*x.shape[:-1], D // GS, GS)
    qmax = np.float32(2 ** bits - 1)
    lo = g.min(axis=-1)
    hi = g.max(axis=-1)
    scale = (hi - lo) / qmax                       # fp32 subtraction and division
    s_hat = round_to(scale, dtype)
    b_hat = round_to(lo, dtype)
    with np.errstate(divide="ignore", invalid="ignore"):
        t = (g - b_hat[..., None]) / s_hat[..., None]
    code = np.rint(t)                              # round half to even
    code = np.where(s_hat[..., None] == 0, np.float32(0), code)
    code = np.clip(code, 0, qmax).astype(np.uint32)
    return code.reshape(x.shape), s_hat.astype(np.float32), b_hat.astype(np.float32)


def pack(codes, bits: int) -> np.ndarray:
    """Pack codes (last axis D) LSB-first: code i goes to word i // (32/bits) at bit bits * (i % (32/bits))."""
    codes = np.asarray(codes, dtype=np.uint64)
    per = 32 // bits
    D = codes.shape[-1]
    if D % per:
        raise ValueError("D must fill whole words")
    if codes.size and codes.max() >= (1 << bits):
        raise ValueError("code out of range")
    c = codes.reshape(*codes.shape[:-1], D // per, per)
    shifted = c << (np.arange(per, dtype=np.uint64) * np.uint64(bits))
    return np.bitwise_or.reduce(shifted, axis=-1).astype(np.uint32)


def unpack(words, bits: int, D: int) -> np.ndarray:
    """Inverse of ``pack``: uint32 words ``[..., D*bits/32]`` to codes ``[..., D]`` (uint32)."""
    words = np.asarray(words, dtype=np.uint32)
    per = 32 // bits
    shifts = (np.arange(per, dtype=np.uint32) * np.uint32(bits))
    c = (words[..., None] >> shifts) & np.uint32((1 << bits) - 1)
    return c.reshape(*words.shape[:-1], D)


def dequantize(codes, s_hat, b_hat, GS: int) -> np.ndarray:
    """``x_hat = s_hat * code + b_hat`` per group, in fp64."""
    codes = np.asarray(codes, dtype=np.float64)
    D = codes.shape[-1]
    c = codes.reshape(*codes.shape[:-1], D // GS, GS)
    x = np.asarray(s_hat, np.float64)[..., None] * c + np.asarray(b_hat, np.float64)[..., None]
    return x.reshape(codes.shape)


# ----------------------------------------------------------------------------------------------- attention


def attention_head(q, K, V) -> np.ndarray:
    """One query head over one KV head, fp64: ``softmax(K q / sqrt(D)) V`` with the max subtracted."""
    q = np.asarray(q, np.float64)
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    D = q.shape[-1]
    s = (K @ q) / math.sqrt(D)
    m = s.max()
    p = np.exp(s - m)
    return (p @ V) / p.sum()


def attention(q, K, V) -> np.ndarray:
    """Single-sequence GQA decode attention. q ``[H, D]``; K, V ``[Hkv, N, D]`` (dequantized); out ``[H, D]``."""
    q = np.asarray(q, np.float64)
    H = q.shape[0]
    Hkv = K.shape[0]
    if H % Hkv:
        raise ValueError("H must be a multiple of Hkv")
    nrep = H // Hkv
    out = np.empty_like(q)
    for h in range(H):
        kv = h // nrep
        out[h] = attention_head(q[h], K[kv], V[kv])
    return out


def attention_blocked(q, K, V, S: int) -> np.ndarray:
    """One head, rows cut into S contiguous blocks: per-block (m, l, o) then the fixed-order merge."""
    q = np.asarray(q, np.float64)
    N = K.shape[0]
    D = q.shape[-1]
    edges = [(N * i) // S for i in range(S + 1)]
    ms, ls, os_ = [], [], []
    for a, b in zip(edges[:-1], edges[1:]):
        if b <= a:
            continue
        s = (np.asarray(K[a:b], np.float64) @ q) / math.sqrt(D)
        m = s.max()
        p = np.exp(s - m)
        ms.append(m)
        ls.append(p.sum())
        os_.append(p @ np.asarray(V[a:b], np.float64))
    M = max(ms)
    den = sum(l * math.exp(m - M) for m, l in zip(ms, ls))
    num = sum(o * math.exp(m - M) for m, o in zip(ms, os_))
    return num / den


def attention_head_compat(q, K, V, dtype: str) -> np.ndarray:
    """One head in the pages' two-pass form with its rounding points (mlx-bun ``fused-decode-kernel.ts`` header:
    kernel A takes per-block (max, sum-exp) over scores rounded to T, kernel C sums ``T(exp(s - M) / denom) *
    dequant(V)`` with the full-row (M, denom), the merge sums the blocks and casts to T).

    T is ``dtype`` (bf16 or fp16). A score is ``q . k / sqrt(D)``, rounded to fp32 and then to T (the two steps a
    fp32 kernel takes); a probability is ``exp(s - M) / denom`` in fp64, rounded to fp32 and then to T; the
    weighted V sum is fp64 and is not renormalised. The caller rounds the output to its dtype.
    """
    q = np.asarray(q, np.float64)
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    D = q.shape[-1]
    s = round_to(((K @ q) / math.sqrt(D)).astype(np.float32), dtype).astype(np.float64)
    M = s.max()
    e = np.exp(s - M)
    p = round_to((e / e.sum()).astype(np.float32), dtype).astype(np.float64)
    return p @ V


def attention_two_pass_blocked(q, K, V, S: int, dtype: str) -> np.ndarray:
    """``attention_head_compat`` computed as the pages' two passes over S contiguous blocks: per-block (m, l) of the
    rounded scores, the full-row (M, denom) from them, per-block sums of rounded probabilities times V, and the
    blocks added in order."""
    q = np.asarray(q, np.float64)
    N = K.shape[0]
    D = q.shape[-1]
    edges = [(N * i) // S for i in range(S + 1)]
    blocks = [(a, b) for a, b in zip(edges[:-1], edges[1:]) if b > a]
    score = [round_to(((np.asarray(K[a:b], np.float64) @ q) / math.sqrt(D)).astype(np.float32), dtype)
             .astype(np.float64) for a, b in blocks]
    stats = [(s.max(), np.exp(s - s.max()).sum()) for s in score]            # pass A
    M = max(m for m, _ in stats)
    denom = sum(l * math.exp(m - M) for m, l in stats)
    out = np.zeros(V.shape[-1])
    for (a, b), s in zip(blocks, score):                                        # pass B, then the sum
        p = round_to((np.exp(s - M) / denom).astype(np.float32), dtype).astype(np.float64)
        out = out + p @ np.asarray(V[a:b], np.float64)
    return out


# ------------------------------------------------------------------------------- the packed-cache interface


def seq_row_offsets(N, Hkv: int):
    """Row (of D elements) where each sequence's ``[Hkv, N[b], .]`` block starts in the back-to-back layout."""
    offs = [0]
    for n in N:
        offs.append(offs[-1] + Hkv * int(n))
    return offs


def unit_rows(N, Hkv: int, b: int, kvh: int):
    """Row range ``[r0, r1)`` of KV head ``kvh`` of sequence ``b``."""
    offs = seq_row_offsets(N, Hkv)
    r0 = offs[b] + kvh * int(N[b])
    return r0, r0 + int(N[b])


def attention_packed(q, kp, ks, kb, vp, vs, vb, N, H: int, Hkv: int, D: int, GS: int, bits: int, heads=None):
    """Decode attention straight from the packed cache layout the GPU library reads.

    q ``[B, H, D]`` (values); kp/vp ``[rows, D*bits/32]`` uint32; ks/kb/vs/vb ``[rows, D/GS]`` scale/bias values
    (fp32 holding bf16/fp16 values); ``rows = Hkv * sum(N)``. ``heads``: iterable of (b, h) to compute (default
    all). Returns a dict {(b, h): out[D] fp64}.
    """
    q = np.asarray(q, np.float64)
    B = len(N)
    nrep = H // Hkv
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(H)]
    res = {}
    cache = {}
    for b, h in heads:
        kvh = h // nrep
        key = (b, kvh)
        if key not in cache:
            r0, r1 = unit_rows(N, Hkv, b, kvh)
            Kd = dequantize(unpack(kp[r0:r1], bits, D), ks[r0:r1], kb[r0:r1], GS)
            Vd = dequantize(unpack(vp[r0:r1], bits, D), vs[r0:r1], vb[r0:r1], GS)
            cache = {key: (Kd, Vd)}          # keep one unit resident: bounded memory at large N
        Kd, Vd = cache[key]
        res[(b, h)] = attention_head(q[b, h], Kd, Vd)
    return res


def visible_rows(n: int, L: int, l: int) -> int:
    """Rows of a sequence of ``n`` cache rows that query position ``l`` of ``L`` attends.

    The L query positions are the sequence's last L tokens, whose K and V rows are already in the cache (rows
    n - L .. n - 1); position l sees every row up to and including its own, ``n - L + 1 + l`` rows in all. With
    L = 1 this is the whole window of single-query decode (mlx-bun ``fused-decode-kernel.ts``, header comment:
    L > 1 goes to a separate N-tiled path; @mlx-bun/inference ``trellis/reduce.ts``: matrix-vector kernels take
    up to ``TRELLIS_MATVEC_MAX_M = 4`` rows at once).
    """
    if not 1 <= L <= n or not 0 <= l < L:
        raise ValueError("need 1 <= L <= n and 0 <= l < L")
    return n - L + 1 + l


def attention_packed_multi(q, kp, ks, kb, vp, vs, vb, N, L: int, H: int, Hkv: int, D: int, GS: int, bits: int,
                           heads=None):
    """Decode attention for L query positions per sequence from the packed cache (small-L multi-query decode).

    q ``[B, L, H, D]`` (values); cache arrays as in ``attention_packed``. Query (b, l, h) attends the first
    ``visible_rows(N[b], L, l)`` rows of its KV head ``h // (H / Hkv)``. ``heads``: iterable of (b, l, h)
    (default all). Returns {(b, l, h): out[D] fp64}.
    """
    q = np.asarray(q, np.float64)
    B = len(N)
    nrep = H // Hkv
    if heads is None:
        heads = [(b, l, h) for b in range(B) for l in range(L) for h in range(H)]
    res = {}
    cache = {}
    for b, l, h in heads:
        kvh = h // nrep
        key = (b, kvh)
        if key not in cache:
            r0, r1 = unit_rows(N, Hkv, b, kvh)
            Kd = dequantize(unpack(kp[r0:r1], bits, D), ks[r0:r1], kb[r0:r1], GS)
            Vd = dequantize(unpack(vp[r0:r1], bits, D), vs[r0:r1], vb[r0:r1], GS)
            cache = {key: (Kd, Vd)}
        Kd, Vd = cache[key]
        n = visible_rows(int(N[b]), L, l)
        res[(b, l, h)] = attention_head(q[b, l, h], Kd[:n], Vd[:n])
    return res


def attention_packed_compat(q, kp, ks, kb, vp, vs, vb, N, H: int, Hkv: int, D: int, GS: int, bits: int,
                            dtype: str, heads=None):
    """``attention_packed`` with the two-pass rounding points of ``attention_head_compat`` (T = ``dtype``)."""
    q = np.asarray(q, np.float64)
    B = len(N)
    nrep = H // Hkv
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(H)]
    res = {}
    cache = {}
    for b, h in heads:
        kvh = h // nrep
        key = (b, kvh)
        if key not in cache:
            r0, r1 = unit_rows(N, Hkv, b, kvh)
            Kd = dequantize(unpack(kp[r0:r1], bits, D), ks[r0:r1], kb[r0:r1], GS)
            Vd = dequantize(unpack(vp[r0:r1], bits, D), vs[r0:r1], vb[r0:r1], GS)
            cache = {key: (Kd, Vd)}
        Kd, Vd = cache[key]
        res[(b, h)] = attention_head_compat(q[b, h], Kd, Vd, dtype)
    return res


def cache_append(old, N, K_new, V_new, Hkv: int, D: int, GS: int, bits: int, dtype: str):
    """Append T new tokens per sequence to a packed cache (maya-mac ``mlx_kernels.py``, ``_ATTEND``: each pass writes
    the cache anew, every KV head's old rows followed by this pass's new rows).

    old: (kp, ks, kb, vp, vs, vb) in the back-to-back layout for lengths N; K_new, V_new ``[B, Hkv, T, D]`` fp32.
    Returns the six arrays for lengths N[b] + T: per (b, kvh) the old rows unchanged, then the new rows quantized.
    """
    K_new = np.asarray(K_new, np.float32)
    V_new = np.asarray(V_new, np.float32)
    B, _, T, _ = K_new.shape
    kn = quantize_cache(K_new.reshape(-1, D), V_new.reshape(-1, D), GS, bits, dtype)
    parts = [[] for _ in range(6)]
    r_old = 0
    for b in range(B):
        n = int(N[b])
        for kvh in range(Hkv):
            i_new = (b * Hkv + kvh) * T
            for a in range(6):
                parts[a].append(np.asarray(old[a])[r_old:r_old + n])
                parts[a].append(kn[a][i_new:i_new + T])
            r_old += n
    return tuple(np.concatenate(p) for p in parts)


def qgemv(x, wp, ws, wb, K: int, GS: int, bits: int) -> np.ndarray:
    """Matrix-vector product with an affine-quantized weight matrix, fp64 (maya-mac ``mlx_kernels.py``,
    ``_linear_kernel``: each weight is ``code * scale + bias`` with one scale and bias per group of GS consecutive
    elements of a row, codes packed LSB-first; ``y[t, n] = sum_k x[t, k] * w[n, k]``, here without the kernel's
    optional LayerNorm, activation and residual epilogues).

    x ``[T, K]`` (values); wp ``[N, K*bits/32]`` uint32; ws, wb ``[N, K/GS]`` (values). Returns y ``[T, N]``.
    """
    W = dequantize(unpack(wp, bits, K), ws, wb, GS)
    return np.asarray(x, np.float64) @ W.T


def quantize_cache(K, V, GS: int, bits: int, dtype: str):
    """Quantize fp32 K and V rows ``[rows, D]`` and pack them: returns kp, ks, kb, vp, vs, vb."""
    kc, ks, kb = quantize(K, GS, bits, dtype)
    vc, vs, vb = quantize(V, GS, bits, dtype)
    return pack(kc, bits), ks, kb, pack(vc, bits), vs, vb
