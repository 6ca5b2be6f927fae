"""Quantized-KV single-query decode attention for GB300 (sm_103a).

The work happens in libqdecode_attn.so (hand-written CUDA behind a C ABI, include/qdecode_attn.h). This module
only marshals torch tensors (device memory and streams) into that ABI, under the same names.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Sequence

import torch

from . import _lib
from ._lib import (QDA_BF16, QDA_FP16, QDA_FP32, QdaError, QdaPlan, lib)  # noqa: F401

_DT_CODE = {torch.bfloat16: QDA_BF16, torch.float16: QDA_FP16, torch.float32: QDA_FP32}
_CODE_DT = {v: k for k, v in _DT_CODE.items()}


def dtype_code(in_dtype: torch.dtype, out_dtype: Optional[torch.dtype] = None) -> int:
    """The ABI's dtype argument: input dtype in the low byte, output dtype in the next."""
    return _DT_CODE[in_dtype] | ((_DT_CODE[out_dtype] if out_dtype is not None else 0) << 8)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def qdecode_attn(q: torch.Tensor, k_packed: torch.Tensor, k_scales: torch.Tensor, k_biases: torch.Tensor,
                 v_packed: torch.Tensor, v_scales: torch.Tensor, v_biases: torch.Tensor, out: torch.Tensor,
                 N: Sequence[int], Hkv: int, GS: int, bits: int, stream=None) -> torch.Tensor:
    """out[b, h] = softmax(q[b, h] . K_hat[b, h // (H/Hkv)]^T / sqrt(D)) V_hat[...] from the packed cache.

    q ``[B, H, D]`` bf16/fp16; packed ``[Hkv * sum(N), D*bits/32]`` int32/uint32 (sequences back to back, each
    ``[Hkv, N[b], .]``); scales/biases ``[Hkv * sum(N), D/GS]`` in q's dtype; out ``[B, H, D]`` (bf16, fp16 or
    fp32). Asynchronous on ``stream`` (default: torch's current stream).
    """
    B, H, D = q.shape
    n = _lib.int32_array(N)
    st = lib().qdecode_attn(_ptr(q), _ptr(k_packed), _ptr(k_scales), _ptr(k_biases), _ptr(v_packed),
                            _ptr(v_scales), _ptr(v_biases), _ptr(out), B, H, Hkv, n, D, GS, bits,
                            dtype_code(q.dtype, out.dtype), _stream(stream))
    _lib.check(st, "qdecode_attn")
    return out


def qdecode_attn_noalloc(q: torch.Tensor, k_packed: torch.Tensor, k_scales: torch.Tensor, k_biases: torch.Tensor,
                         v_packed: torch.Tensor, v_scales: torch.Tensor, v_biases: torch.Tensor, out: torch.Tensor,
                         N: Sequence[int], Hkv: int, GS: int, bits: int, stream=None) -> torch.Tensor:
    """qdecode_attn for callers that must not allocate device memory: the library's fixed scratch array is used
    instead of a workspace (shapes needing more than QDA_STATIC_SCRATCH_BYTES are rejected). Calls that overlap
    on the GPU share that array and must be serialised by the caller."""
    B, H, D = q.shape
    st = lib().qdecode_attn_noalloc(_ptr(q), _ptr(k_packed), _ptr(k_scales), _ptr(k_biases), _ptr(v_packed),
                                    _ptr(v_scales), _ptr(v_biases), _ptr(out), B, H, Hkv, _lib.int32_array(N), D,
                                    GS, bits, dtype_code(q.dtype, out.dtype), _stream(stream))
    _lib.check(st, "qdecode_attn_noalloc")
    return out


def qdecode_attn_host(q: torch.Tensor, k_packed: torch.Tensor, k_scales: torch.Tensor, k_biases: torch.Tensor,
                      v_packed: torch.Tensor, v_scales: torch.Tensor, v_biases: torch.Tensor, out: torch.Tensor,
                      N: Sequence[int], Hkv: int, GS: int, bits: int, stream=None) -> torch.Tensor:
    """qdecode_attn with every tensor in HOST memory (contiguous CPU tensors; pinned ones copy at full speed): the
    library stages the inputs on the current device, decodes and copies out back, asynchronously on `stream`.
    Synchronise the stream before reading out or changing the inputs."""
    ts = (q, k_packed, k_scales, k_biases, v_packed, v_scales, v_biases, out)
    if any(t.is_cuda or not t.is_contiguous() for t in ts):
        raise ValueError("qdecode_attn_host takes contiguous host tensors")
    B, H, D = q.shape
    st = lib().qdecode_attn_host(*(_ptr(t) for t in ts), B, H, Hkv, _lib.int32_array(N), D, GS, bits,
                                 dtype_code(q.dtype, out.dtype), _stream(stream))
    _lib.check(st, "qdecode_attn_host")
    return out


def qdecode_attn_compat(q: torch.Tensor, k_packed: torch.Tensor, k_scales: torch.Tensor, k_biases: torch.Tensor,
                        v_packed: torch.Tensor, v_scales: torch.Tensor, v_biases: torch.Tensor, out: torch.Tensor,
                        N: Sequence[int], Hkv: int, GS: int, bits: int, stream=None) -> torch.Tensor:
    """qdecode_attn in the two-pass form with compat rounding: scores and normalised probabilities rounded to the
    input dtype, the probability-weighted V rows summed without renormalising."""
    B, H, D = q.shape
    st = lib().qdecode_attn_compat(_ptr(q), _ptr(k_packed), _ptr(k_scales), _ptr(k_biases), _ptr(v_packed),
                                   _ptr(v_scales), _ptr(v_biases), _ptr(out), B, H, Hkv, _lib.int32_array(N), D,
                                   GS, bits, dtype_code(q.dtype, out.dtype), _stream(stream))
    _lib.check(st, "qdecode_attn_compat")
    return out


def qdecode_attn_multi(q: torch.Tensor, k_packed: torch.Tensor, k_scales: torch.Tensor, k_biases: torch.Tensor,
                       v_packed: torch.Tensor, v_scales: torch.Tensor, v_biases: torch.Tensor, out: torch.Tensor,
                       N: Sequence[int], Hkv: int, GS: int, bits: int, stream=None) -> torch.Tensor:
    """Small-L multi-query decode: q and out ``[B, L, H, D]``; the L positions are each sequence's last L tokens
    (already the last L rows of its cache, counted in N), and position l attends the first N[b] - L + 1 + l
    rows. Cache arguments as for qdecode_attn."""
    B, L, H, D = q.shape
    st = lib().qdecode_attn_multi(_ptr(q), _ptr(k_packed), _ptr(k_scales), _ptr(k_biases), _ptr(v_packed),
                                  _ptr(v_scales), _ptr(v_biases), _ptr(out), B, L, H, Hkv, _lib.int32_array(N), D,
                                  GS, bits, dtype_code(q.dtype, out.dtype), _stream(stream))
    _lib.check(st, "qdecode_attn_multi")
    return out


def bind_qdecode_attn(q: torch.Tensor, k_packed: torch.Tensor, k_scales: torch.Tensor, k_biases: torch.Tensor,
                      v_packed: torch.Tensor, v_scales: torch.Tensor, v_biases: torch.Tensor, out: torch.Tensor,
                      N: Sequence[int], Hkv: int, GS: int, bits: int, stream=None):
    """qdecode_attn with every argument marshalled once: returns a no-argument callable for repeated calls on
    the same buffers (decode loops, timing)."""
    B, H, D = q.shape
    args = (_ptr(q), _ptr(k_packed), _ptr(k_scales), _ptr(k_biases), _ptr(v_packed), _ptr(v_scales),
            _ptr(v_biases), _ptr(out), B, H, Hkv, _lib.int32_array(N), D, GS, bits, dtype_code(q.dtype, out.dtype),
            _stream(stream))
    fn = lib().qdecode_attn

    def call():
        st = fn(*args)
        if st:
            raise _lib.QdaError(st, "qdecode_attn")
    call.keepalive = (q, k_packed, k_scales, k_biases, v_packed, v_scales, v_biases, out)
    return call


def qdecode_attn_plan(B: int, H: int, Hkv: int, N: Sequence[int], D: int, GS: int, bits: int, num_sms: int = 0,
                      ctas_per_sm: int = 0) -> dict:
    plan = QdaPlan()
    st = lib().qdecode_attn_plan(B, H, Hkv, _lib.int32_array(N), D, GS, bits, num_sms, ctas_per_sm,
                                 ctypes.byref(plan))
    _lib.check(st, "qdecode_attn_plan")
    return plan.as_dict()


def qdecode_attn_multi_plan(B: int, L: int, H: int, Hkv: int, N: Sequence[int], D: int, GS: int, bits: int,
                            num_sms: int = 0, ctas_per_sm: int = 0) -> dict:
    plan = QdaPlan()
    st = lib().qdecode_attn_multi_plan(B, L, H, Hkv, _lib.int32_array(N), D, GS, bits, num_sms, ctas_per_sm,
                                       ctypes.byref(plan))
    _lib.check(st, "qdecode_attn_multi_plan")
    return plan.as_dict()


def qdecode_attn_workspace_bytes(B: int, H: int, Hkv: int, N: Sequence[int], D: int, GS: int, bits: int) -> int:
    out = ctypes.c_size_t()
    st = lib().qdecode_attn_workspace_bytes(B, H, Hkv, _lib.int32_array(N), D, GS, bits, ctypes.byref(out))
    _lib.check(st, "qdecode_attn_workspace_bytes")
    return out.value


def qdecode_attn_set_workspace(buf: Optional[torch.Tensor]) -> None:
    st = lib().qdecode_attn_set_workspace(_ptr(buf), 0 if buf is None else buf.numel() * buf.element_size())
    _lib.check(st, "qdecode_attn_set_workspace")


def qdecode_attn_debug_force_splits(num_ctas: int) -> None:
    _lib.check(lib().qdecode_attn_debug_force_splits(num_ctas), "qdecode_attn_debug_force_splits")


def qdecode_attn_debug_stall_chunk(chunk: int) -> None:
    """Testing aid: the first CTA's producer stops before its chunk ``chunk`` (-1: off); see the C header."""
    _lib.check(lib().qdecode_attn_debug_stall_chunk(chunk), "qdecode_attn_debug_stall_chunk")


def qdecode_attn_set_split_event(event: Optional[torch.cuda.Event]) -> None:
    handle = None if event is None else event.cuda_event
    _lib.check(lib().qdecode_attn_set_split_event(handle), "qdecode_attn_set_split_event")


def qdecode_quantize(x: torch.Tensor, GS: int, bits: int, dtype: torch.dtype, packed: torch.Tensor,
                     scales: torch.Tensor, biases: torch.Tensor, stream=None) -> None:
    """Quantize fp32 rows ``x [rows, D]`` into ``packed [rows, D*bits/32]``, ``scales``/``biases [rows, D/GS]``
    (dtype bf16 or fp16). Writing into views offset to a cache's next rows appends to that cache."""
    rows, D = x.shape
    st = lib().qdecode_quantize(_ptr(x), rows, D, GS, bits, dtype_code(dtype), _ptr(packed), _ptr(scales),
                                _ptr(biases), _stream(stream))
    _lib.check(st, "qdecode_quantize")


def qdecode_qgemv(x: torch.Tensor, w_packed: torch.Tensor, w_scales: torch.Tensor, w_biases: torch.Tensor,
                  y: torch.Tensor, GS: int, bits: int, stream=None) -> torch.Tensor:
    """y[t, n] = sum_k x[t, k] * (scale * code + bias)[n, k]: x ``[T, K]`` bf16/fp16, packed ``[N, K*bits/32]``,
    scales/biases ``[N, K/GS]`` in x's dtype, y ``[T, N]`` (bf16, fp16 or fp32)."""
    T, K = x.shape
    N = w_packed.shape[0]
    st = lib().qdecode_qgemv(_ptr(x), _ptr(w_packed), _ptr(w_scales), _ptr(w_biases), _ptr(y), T, N, K, GS, bits,
                             dtype_code(x.dtype, y.dtype), _stream(stream))
    _lib.check(st, "qdecode_qgemv")
    return y


def qdecode_attn_device_status() -> int:
    flags = ctypes.c_uint()
    _lib.check(lib().qdecode_attn_device_status(ctypes.byref(flags)), "qdecode_attn_device_status")
    return flags.value


def qdecode_attn_calls() -> int:
    return lib().qdecode_attn_calls()


# ------------------------------------------------------------------------------------------- conveniences


class QuantizedKV:
    """A packed cache in the library's layout: sequences back to back, each ``[Hkv, N[b], .]``."""

    def __init__(self, packed_k, scales_k, biases_k, packed_v, scales_v, biases_v, N, Hkv, D, GS, bits):
        self.kp, self.ks, self.kb = packed_k, scales_k, biases_k
        self.vp, self.vs, self.vb = packed_v, scales_v, biases_v
        self.N, self.Hkv, self.D, self.GS, self.bits = list(N), Hkv, D, GS, bits

    @classmethod
    def empty(cls, N, Hkv, D, GS, bits, dtype, device="cuda"):
        rows = Hkv * sum(N)
        W, NG = D * bits // 32, D // GS
        mk = lambda shape, dt: torch.empty(shape, dtype=dt, device=device)  # noqa: E731
        return cls(mk((rows, W), torch.int32), mk((rows, NG), dtype), mk((rows, NG), dtype),
                   mk((rows, W), torch.int32), mk((rows, NG), dtype), mk((rows, NG), dtype), N, Hkv, D, GS, bits)

    @property
    def dtype(self):
        return self.ks.dtype

    def unit_rows(self, b: int, kvh: int):
        r0 = self.Hkv * sum(self.N[:b]) + kvh * self.N[b]
        return r0, r0 + self.N[b]

    def quantize_into(self, b: int, kvh: int, K: torch.Tensor, V: torch.Tensor, row0: int = 0, stream=None):
        """Quantize fp32 K, V rows ``[n, D]`` into rows ``row0 .. row0 + n`` of KV head ``kvh`` of sequence b."""
        r0, r1 = self.unit_rows(b, kvh)
        a = r0 + row0
        e = a + K.shape[0]
        if e > r1:
            raise ValueError("rows past the end of this KV head")
        qdecode_quantize(K, self.GS, self.bits, self.dtype, self.kp[a:e], self.ks[a:e], self.kb[a:e], stream)
        qdecode_quantize(V, self.GS, self.bits, self.dtype, self.vp[a:e], self.vs[a:e], self.vb[a:e], stream)

    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in (self.kp, self.ks, self.kb, self.vp, self.vs, self.vb))

    def append(self, K_new: torch.Tensor, V_new: torch.Tensor, out: "QuantizedKV" = None, stream=None) -> "QuantizedKV":
        """The cache with T new tokens per sequence (``K_new``, ``V_new`` fp32 ``[B, Hkv, T, D]``): every KV head's
        old rows, then the new rows quantized (qdecode_cache_append). Writes ``out`` (allocated when None)."""
        B, Hkv, T, D = K_new.shape
        kn, vn = K_new.contiguous(), V_new.contiguous()
        if out is None:
            out = QuantizedKV.empty([n + T for n in self.N], self.Hkv, self.D, self.GS, self.bits, self.dtype,
                                    device=K_new.device)
        st = lib().qdecode_cache_append(
            _ptr(self.kp), _ptr(self.ks), _ptr(self.kb), _ptr(self.vp), _ptr(self.vs), _ptr(self.vb),
            _ptr(kn), _ptr(vn), _ptr(out.kp), _ptr(out.ks), _ptr(out.kb),
            _ptr(out.vp), _ptr(out.vs), _ptr(out.vb), B, Hkv, _lib.int32_array(self.N), T, D, self.GS, self.bits,
            dtype_code(self.dtype), _stream(stream))
        _lib.check(st, "qdecode_cache_append")
        return out


def bind_decode_attention(q: torch.Tensor, cache: QuantizedKV, out: torch.Tensor, stream=None):
    """Pre-marshalled decode_attention over a QuantizedKV (see bind_qdecode_attn)."""
    return bind_qdecode_attn(q, cache.kp, cache.ks, cache.kb, cache.vp, cache.vs, cache.vb, out, cache.N, cache.Hkv,
                             cache.GS, cache.bits, stream)


def decode_attention(q: torch.Tensor, cache: QuantizedKV, out_dtype: Optional[torch.dtype] = None,
                     out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Allocating wrapper of qdecode_attn over a QuantizedKV."""
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype or q.dtype, device=q.device)
    return qdecode_attn(q, cache.kp, cache.ks, cache.kb, cache.vp, cache.vs, cache.vb, out, cache.N, cache.Hkv,
                        cache.GS, cache.bits, stream)
