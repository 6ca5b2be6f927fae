"""Seeded synthetic inputs for quantized-KV decode attention: the five benchmark workloads and small test cases.

This module only draws numbers: fp32 K and V rows, the query, the sequence lengths and the structure a workload
asks for (outlier channels, keys planted along the query). It holds none of the attention or quantization
arithmetic, so the GPU library and the CPU oracle can both be fed from it. Draws come from ``torch.Generator``
objects seeded per (workload seed, tensor, sequence, KV head), so any KV head can be regenerated on its own.
A CPU and a CUDA generator give different numbers for the same seed; callers hand the same drawn tensors to both
sides of a comparison.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import torch

DT = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}
BASE_SEED = 20261202


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Hkv: int
    D: int
    bits: int
    GS: int
    dtype_in: str
    dtype_out: str
    N: Optional[tuple] = None          # fixed lengths; None = drawn (ragged)
    n_range: Optional[tuple] = None    # inclusive [lo, hi] for drawn lengths
    k_outliers: int = 0                # channels per KV head multiplied by outlier_scale (K only)
    outlier_scale: float = 20.0
    planted: int = 0                   # keys per KV head planted along a query direction
    planted_cos: float = 0.9
    v_uniform: bool = False            # V ~ U(-1, 1) instead of N(0, 1)
    seed: int = BASE_SEED

    @property
    def nrep(self) -> int:
        return self.H // self.Hkv


def _wl(idx, **kw):
    return Workload(seed=BASE_SEED + idx, **kw)


# The five workloads: small parity case, the 8k latency case, long-context fp16 with outlier channels, a ragged
# batch of eight sequences, and a 128k peaky-softmax case with fp32 output.
WORKLOADS = [
    _wl(1, name="c1_B1_H8_Hkv2_D256_N512_4b_GS64_bf16", B=1, H=8, Hkv=2, D=256, bits=4, GS=64,
        dtype_in="bf16", dtype_out="bf16", N=(512,)),
    _wl(2, name="c2_B1_H16_Hkv8_D256_N8192_8b_GS32_bf16", B=1, H=16, Hkv=8, D=256, bits=8, GS=32,
        dtype_in="bf16", dtype_out="bf16", N=(8192,)),
    _wl(3, name="c3_B1_H16_Hkv8_D512_N32768_4b_GS128_fp16", B=1, H=16, Hkv=8, D=512, bits=4, GS=128,
        dtype_in="fp16", dtype_out="fp16", N=(32768,), k_outliers=4),
    _wl(4, name="c4_B8_H32_Hkv8_D256_N1k-64k_4b_GS64_bf16", B=8, H=32, Hkv=8, D=256, bits=4, GS=64,
        dtype_in="bf16", dtype_out="bf16", n_range=(1024, 65536)),
    _wl(5, name="c5_B1_H16_Hkv4_D256_N131072_4b_GS32_bf16_fp32out", B=1, H=16, Hkv=4, D=256, bits=4, GS=32,
        dtype_in="bf16", dtype_out="fp32", N=(131072,), planted=32, v_uniform=True),
]


def workload(i: int) -> Workload:
    """Workload by 1-based index (1..5)."""
    return WORKLOADS[i - 1]


def _gen(seed: int, *key: int, device="cpu") -> torch.Generator:
    # splitmix64-style mixing of the key into one 63-bit seed, so every (tensor, b, kvh) stream is independent
    z = seed & 0xFFFFFFFFFFFFFFFF
    for k in key:
        z = (z + 0x9E3779B97F4A7C15 + (k & 0xFFFFFFFF)) & 0xFFFFFFFFFFFFFFFF
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & 0xFFFFFFFFFFFFFFFF
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & 0xFFFFFFFFFFFFFFFF
        z ^= z >> 31
    g = torch.Generator(device=device)
    g.manual_seed(z & 0x7FFFFFFFFFFFFFFF)
    return g


T_Q, T_K, T_V, T_LEN, T_OUTL, T_PLANT_ROWS, T_PLANT_DIR, T_QMULTI = range(1, 9)


def lengths(w: Workload) -> List[int]:
    """Per-sequence cache lengths: fixed, or uniform integers in the inclusive range, drawn from the seed."""
    if w.N is not None:
        return list(w.N)
    lo, hi = w.n_range
    g = _gen(w.seed, T_LEN)
    return [int(v) for v in torch.randint(lo, hi + 1, (w.B,), generator=g)]


def query(w: Workload, device="cpu") -> torch.Tensor:
    """q ``[B, H, D]`` ~ N(0, 1), rounded to the input dtype."""
    g = _gen(w.seed, T_Q, device=device)
    q = torch.randn(w.B, w.H, w.D, generator=g, device=device, dtype=torch.float32)
    return q.to(DT[w.dtype_in])


def query_multi(w: Workload, L: int, device="cpu") -> torch.Tensor:
    """q ``[B, L, H, D]`` ~ N(0, 1) for L query positions per sequence, rounded to the input dtype."""
    g = _gen(w.seed, T_QMULTI, L, device=device)
    q = torch.randn(w.B, L, w.H, w.D, generator=g, device=device, dtype=torch.float32)
    return q.to(DT[w.dtype_in])


def kv_unit(w: Workload, b: int, kvh: int, n: int, q: Optional[torch.Tensor] = None, device="cpu"):
    """fp32 K and V rows ``[n, D]`` of KV head ``kvh`` of sequence ``b``.

    Structure by workload: outlier channels (``k_outliers`` distinct channels of K per KV head, times
    ``outlier_scale``), planted keys (``planted`` distinct rows per KV head; planted key i lies at cosine
    ``planted_cos`` to query head ``kvh * nrep + i % nrep``, with norm sqrt(D)), V uniform in (-1, 1).
    """
    D = w.D
    gk = _gen(w.seed, T_K, b, kvh, device=device)
    K = torch.randn(n, D, generator=gk, device=device, dtype=torch.float32)
    gv = _gen(w.seed, T_V, b, kvh, device=device)
    if w.v_uniform:
        V = torch.rand(n, D, generator=gv, device=device, dtype=torch.float32) * 2.0 - 1.0
    else:
        V = torch.randn(n, D, generator=gv, device=device, dtype=torch.float32)
    if w.k_outliers:
        go = _gen(w.seed, T_OUTL, b, kvh)
        ch = torch.randperm(D, generator=go)[: w.k_outliers].to(device)
        K[:, ch] *= w.outlier_scale
    if w.planted:
        if q is None:
            q = query(w, device="cpu")
        gr = _gen(w.seed, T_PLANT_ROWS, b, kvh)
        rows = torch.randperm(n, generator=gr)[: min(w.planted, n)]
        gd = _gen(w.seed, T_PLANT_DIR, b, kvh)
        c = w.planted_cos
        for i, r in enumerate(rows.tolist()):
            h = kvh * w.nrep + (i % w.nrep)
            qh = q[b, h].to(torch.float64).cpu()
            qh = qh / qh.norm()
            u = torch.randn(D, generator=gd, dtype=torch.float64)
            u = u - (u @ qh) * qh
            u = u / u.norm()
            k = math.sqrt(D) * (c * qh + math.sqrt(1.0 - c * c) * u)
            K[r] = k.to(torch.float32).to(device)
    return K, V


def planted_rows(w: Workload, b: int, kvh: int, n: int) -> List[int]:
    """Row indices (within the KV head) that ``kv_unit`` plants, in planting order."""
    if not w.planted:
        return []
    gr = _gen(w.seed, T_PLANT_ROWS, b, kvh)
    return torch.randperm(n, generator=gr)[: min(w.planted, n)].tolist()


def small(B=1, H=4, Hkv=2, D=64, N=(37,), bits=4, GS=32, dtype_in="bf16", dtype_out=None, seed=7, **kw) -> Workload:
    """A small ad-hoc workload for sweeps (same generator, any shape)."""
    return Workload(name=f"small_B{B}_H{H}_Hkv{Hkv}_D{D}_{bits}b_GS{GS}", B=B, H=H, Hkv=Hkv, D=D, bits=bits, GS=GS,
                    dtype_in=dtype_in, dtype_out=dtype_out or dtype_in, N=tuple(N), seed=seed, **kw)
