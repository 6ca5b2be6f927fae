"""Shared helpers for the GPU tests: build a case from the seeded generator, quantize it with the oracle (small
cases) or with the library's quantizer (full-size workloads), run the library, and compare per head."""
from __future__ import annotations

import numpy as np
import torch

import oracle as O
import attention_quantized_kv_split_gb300 as qda
from attention_quantized_kv_split_gb300 import synth

TORCH_DT = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}
TOL = {"bf16": 1e-2, "fp16": 1e-2, "fp32": 1e-4}   # max|delta| <= TOL * max|o| per head


def upload_cache(kp, ks, kb, vp, vs, vb, dtype: str, device="cuda"):
    """Oracle-quantized numpy buffers -> the library's device tensors (bit patterns copied exactly)."""
    dt = TORCH_DT[dtype]

    def sc(a):
        return torch.from_numpy(O.bits16(a, dtype).view(np.int16)).view(dt).to(device)

    def pk(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int32)).to(device)

    return pk(kp), sc(ks), sc(kb), pk(vp), sc(vs), sc(vb)


def small_case(w: synth.Workload):
    """Generate on the CPU, quantize with the oracle. Returns (q tensor, numpy cache tuple, N)."""
    N = synth.lengths(w)
    q = synth.query(w)
    Ks, Vs = [], []
    for b in range(w.B):
        for kvh in range(w.Hkv):
            K, V = synth.kv_unit(w, b, kvh, N[b], q=q)
            Ks.append(K.numpy())
            Vs.append(V.numpy())
    K = np.concatenate(Ks)
    V = np.concatenate(Vs)
    cache = O.quantize_cache(K, V, w.GS, w.bits, w.dtype_in)
    return q, cache, N


def run_gpu(q, dev_cache, N, w: synth.Workload, out_dtype: str = None, stream=None):
    out_dtype = out_dtype or w.dtype_out
    qd = q.to("cuda")
    out = torch.empty(qd.shape, dtype=TORCH_DT[out_dtype], device="cuda")
    qda.qdecode_attn(qd, *dev_cache, out, N, w.Hkv, w.GS, w.bits, stream=stream)
    return out


def oracle_out(q, cache, N, w: synth.Workload, heads=None):
    qv = q.to(torch.float64).numpy()
    return O.attention_packed(qv, *cache, N, w.H, w.Hkv, w.D, w.GS, w.bits, heads=heads)


def compare(gpu_out: torch.Tensor, ref: dict, out_dtype: str):
    """Per-head check against the oracle; returns the worst ratio max|delta| / (TOL * max|o|)."""
    g = gpu_out.to(torch.float64).cpu().numpy()
    worst = 0.0
    for (b, h), o in ref.items():
        err = np.abs(g[b, h] - o).max()
        bound = TOL[out_dtype] * np.abs(o).max()
        assert np.all(np.isfinite(g[b, h])), (b, h)
        worst = max(worst, err / bound)
        assert err <= bound, f"head {(b, h)}: max|delta| {err:.3e} > {bound:.3e}"
    return worst


def gpu_quantized_workload(w: synth.Workload, q=None):
    """Full-size workload generated on the GPU and quantized by the library's quantizer."""
    N = synth.lengths(w)
    if q is None:
        q = synth.query(w)
    cache = qda.QuantizedKV.empty(N, w.Hkv, w.D, w.GS, w.bits, TORCH_DT[w.dtype_in])
    for b in range(w.B):
        for kvh in range(w.Hkv):
            K, V = synth.kv_unit(w, b, kvh, N[b], q=q, device="cuda")
            cache.quantize_into(b, kvh, K, V)
            del K, V
    return q, cache, N


def unit_oracle_cache(w: synth.Workload, b: int, kvh: int, N, q):
    """The oracle's quantization of one unit, regenerated with the same (CUDA) generator stream."""
    K, V = synth.kv_unit(w, b, kvh, N[b], q=q, device="cuda")
    return O.quantize_cache(K.cpu().numpy(), V.cpu().numpy(), w.GS, w.bits, w.dtype_in)
