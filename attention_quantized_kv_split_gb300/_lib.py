"""ctypes view of libqdecode_attn.so (the C ABI declared in include/qdecode_attn.h). Loading fails loudly when the
library has not been built: there is no other implementation to fall back to."""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libqdecode_attn.so")

QDA_OK = 0
QDA_ERR_INVALID = -1
QDA_ERR_UNSUPPORTED = -2
QDA_ERR_ALIGN = -3
QDA_ERR_CUDA = -4
QDA_ERR_WORKSPACE = -5
QDA_ERR_SCRATCH = -6
QDA_STATIC_SCRATCH_BYTES = 8 << 20
QDA_BF16, QDA_FP16, QDA_FP32 = 1, 2, 3
QDA_MAX_B = 512
QDA_MAX_NREP = 64
QDA_MAX_L = 8
QDA_QGEMV_MAX_T = 4


class QdaPlan(ctypes.Structure):
    _fields_ = [
        ("num_ctas", ctypes.c_int),
        ("head_chunks", ctypes.c_int),
        ("heads_per_cta", ctypes.c_int),
        ("tile_rows", ctypes.c_int),
        ("stages", ctypes.c_int),
        ("threads", ctypes.c_int),
        ("units", ctypes.c_int),
        ("smem_bytes", ctypes.c_int),
        ("total_rows", ctypes.c_longlong),
        ("slots", ctypes.c_longlong),
        ("workspace_bytes", ctypes.c_size_t),
    ]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


_I, _P, _LL, _SZ = ctypes.c_int, ctypes.c_void_p, ctypes.c_longlong, ctypes.c_size_t
_PI32 = ctypes.POINTER(ctypes.c_int32)

SIGNATURES = {
    "qdecode_attn": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _PI32, _I, _I, _I, _I, _P]),
    "qdecode_attn_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _PI32, _I, _I, _I, _I, _P]),
    "qdecode_attn_host": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _PI32, _I, _I, _I, _I, _P]),
    "qdecode_attn_compat": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _PI32, _I, _I, _I, _I, _P]),
    "qdecode_attn_multi": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _PI32, _I, _I, _I, _I, _P]),
    "qdecode_attn_multi_plan": (_I, [_I, _I, _I, _I, _PI32, _I, _I, _I, _I, _I, ctypes.POINTER(QdaPlan)]),
    "qdecode_attn_plan": (_I, [_I, _I, _I, _PI32, _I, _I, _I, _I, _I, ctypes.POINTER(QdaPlan)]),
    "qdecode_attn_workspace_bytes": (_I, [_I, _I, _I, _PI32, _I, _I, _I, ctypes.POINTER(_SZ)]),
    "qdecode_attn_set_workspace": (_I, [_P, _SZ]),
    "qdecode_attn_debug_force_splits": (_I, [_I]),
    "qdecode_attn_debug_stall_chunk": (_I, [_I]),
    "qdecode_attn_set_split_event": (_I, [_P]),
    "qdecode_qgemv": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "qdecode_cache_append": (_I, [_P] * 14 + [_I, _I, _PI32, _I, _I, _I, _I, _I, _P]),
    "qdecode_quantize": (_I, [_P, _LL, _I, _I, _I, _I, _P, _P, _P, _P]),
    "qdecode_attn_strerror": (ctypes.c_char_p, [_I]),
    "qdecode_attn_last_cuda_error": (_I, []),
    "qdecode_attn_device_status": (_I, [ctypes.POINTER(ctypes.c_uint)]),
    "qdecode_attn_calls": (_LL, []),
}

_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library (built in-tree by attention_quantized_kv_split_gb300.build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -m attention_quantized_kv_split_gb300.build` "
                "(nvcc for sm_103a). The decode attention path has no other implementation.")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


class QdaError(RuntimeError):
    def __init__(self, status: int, where: str):
        text = lib().qdecode_attn_strerror(status).decode()
        cuda = lib().qdecode_attn_last_cuda_error() if status == QDA_ERR_CUDA else 0
        super().__init__(f"{where}: status {status} ({text})" + (f", cudaError {cuda}" if cuda else ""))
        self.status = status
        self.cuda_error = cuda


def check(status: int, where: str) -> None:
    if status != QDA_OK:
        raise QdaError(status, where)


def int32_array(values):
    arr = (ctypes.c_int32 * len(values))(*[int(v) for v in values])
    return arr
