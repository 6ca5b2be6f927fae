"""The C ABI without a GPU: the library loads, exports what the header declares, rejects bad arguments before any
launch, and plans deterministically. No call here reaches a kernel."""
import ctypes
import os
import re

import pytest

from attention_quantized_kv_split_gb300 import _lib, build as qbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    qbuild.build()
    return _lib.lib()


def header_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w \*]*?\b(qdecode_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = header_functions()
    assert "qdecode_attn" in names and "qdecode_quantize" in names and len(names) >= 10


def test_library_exports_every_declared_symbol(L):
    for name in header_functions():
        assert hasattr(L, name), name
        assert name in _lib.SIGNATURES, f"{name} has no ctypes signature"


FAKE = 0x7F0000000000  # never dereferenced: every call below fails its host-side checks first


def call(L, B=1, H=8, Hkv=2, N=(512,), D=256, GS=64, bits=4, dtype=1, ptrs=None, nptr=None):
    p = [FAKE + 256 * i for i in range(8)] if ptrs is None else ptrs
    n = _lib.int32_array(N) if nptr is None else nptr
    return L.qdecode_attn(*p, B, H, Hkv, n, D, GS, bits, dtype, None)


@pytest.mark.parametrize("i", range(8))
def test_null_pointer_is_invalid(L, i):
    p = [FAKE + 256 * k for k in range(8)]
    p[i] = None
    assert call(L, ptrs=p) == _lib.QDA_ERR_INVALID


@pytest.mark.parametrize("i", range(8))
def test_misaligned_pointer(L, i):
    p = [FAKE + 256 * k for k in range(8)]
    p[i] += 8
    assert call(L, ptrs=p) == _lib.QDA_ERR_ALIGN


@pytest.mark.parametrize("kw,status", [
    (dict(bits=3), _lib.QDA_ERR_UNSUPPORTED),
    (dict(bits=2), _lib.QDA_ERR_UNSUPPORTED),
    (dict(GS=48), _lib.QDA_ERR_UNSUPPORTED),
    (dict(GS=16), _lib.QDA_ERR_UNSUPPORTED),
    (dict(D=96, GS=32), _lib.QDA_ERR_UNSUPPORTED),
    (dict(D=1024, GS=64), _lib.QDA_ERR_UNSUPPORTED),
    (dict(D=64, GS=128), _lib.QDA_ERR_UNSUPPORTED),
    (dict(H=6, Hkv=4), _lib.QDA_ERR_INVALID),
    (dict(N=(0,)), _lib.QDA_ERR_INVALID),
    (dict(B=2, N=(5, -1)), _lib.QDA_ERR_INVALID),
    (dict(B=0, N=(1,)), _lib.QDA_ERR_INVALID),
    (dict(H=0), _lib.QDA_ERR_INVALID),
    (dict(Hkv=0), _lib.QDA_ERR_INVALID),
    (dict(B=_lib.QDA_MAX_B + 1, N=(4,) * (_lib.QDA_MAX_B + 1)), _lib.QDA_ERR_UNSUPPORTED),
    (dict(H=130, Hkv=2), _lib.QDA_ERR_UNSUPPORTED),
    (dict(dtype=0), _lib.QDA_ERR_INVALID),
    (dict(dtype=3), _lib.QDA_ERR_INVALID),            # fp32 input is not a cache dtype
    (dict(dtype=1 | (4 << 8)), _lib.QDA_ERR_INVALID),
    (dict(dtype=1 | (1 << 16)), _lib.QDA_ERR_INVALID),
])
def test_argument_errors(L, kw, status):
    assert call(L, **kw) == status


def test_null_lengths_invalid(L):
    assert L.qdecode_attn(*[FAKE] * 8, 1, 8, 2, None, 256, 64, 4, 1, None) == _lib.QDA_ERR_INVALID


def test_quantize_argument_errors(L):
    q = L.qdecode_quantize
    assert q(None, 4, 256, 64, 4, 1, FAKE, FAKE, FAKE, None) == _lib.QDA_ERR_INVALID
    assert q(FAKE, 0, 256, 64, 4, 1, FAKE, FAKE, FAKE, None) == _lib.QDA_ERR_INVALID
    assert q(FAKE, 4, 256, 64, 3, 1, FAKE, FAKE, FAKE, None) == _lib.QDA_ERR_UNSUPPORTED
    assert q(FAKE, 4, 256, 48, 4, 1, FAKE, FAKE, FAKE, None) == _lib.QDA_ERR_UNSUPPORTED
    assert q(FAKE + 4, 4, 256, 64, 4, 1, FAKE, FAKE, FAKE, None) == _lib.QDA_ERR_ALIGN
    assert q(FAKE, 4, 256, 64, 4, 7, FAKE, FAKE, FAKE, None) == _lib.QDA_ERR_INVALID


def test_strerror_covers_codes(L):
    for s in (0, -1, -2, -3, -4, -5):
        assert len(L.qdecode_attn_strerror(s)) > 5
    assert L.qdecode_attn_strerror(-99) == b"unknown status"


def plan(L, B, H, Hkv, N, D, GS, bits, sms=152, occ=2):
    p = _lib.QdaPlan()
    st = L.qdecode_attn_plan(B, H, Hkv, _lib.int32_array(N), D, GS, bits, sms, occ, ctypes.byref(p))
    assert st == 0
    return p.as_dict()


def cta_row(T, C, c):
    if c >= C:
        return T
    if c <= 0:
        return 0
    return ((T * c) // C) & ~7


@pytest.mark.parametrize("shape", [
    (1, 8, 2, [512], 256, 64, 4),
    (1, 16, 8, [8192], 256, 32, 8),
    (1, 16, 8, [32768], 512, 128, 4),
    (8, 32, 8, [1024, 65536, 3001, 40000, 17, 9999, 1, 65000], 256, 64, 4),
    (1, 16, 4, [131072], 256, 32, 4),
    (3, 24, 3, [5, 7, 9], 128, 32, 8),
])
def test_plan_properties(L, shape):
    B, H, Hkv, N, D, GS, bits = shape
    p = plan(L, *shape)
    T = Hkv * sum(N)
    assert p["total_rows"] == T
    assert p["units"] == B * Hkv
    assert p["slots"] == p["num_ctas"] + B * Hkv
    nrep = H // Hkv
    assert p["heads_per_cta"] * p["head_chunks"] >= nrep
    assert p["heads_per_cta"] & (p["heads_per_cta"] - 1) == 0
    C = p["num_ctas"]
    assert 1 <= C <= 152 * 2
    assert C == 1 or T // C >= 120          # no range much below the per-CTA row floor
    bounds = [cta_row(T, C, c) for c in range(C + 1)]
    assert bounds[0] == 0 and bounds[-1] == T
    assert all(a <= b for a, b in zip(bounds, bounds[1:]))
    assert all(b % 8 == 0 for b in bounds[1:-1])
    assert p["tile_rows"] % 16 == 0 and p["stages"] >= 2
    assert p["smem_bytes"] <= 227 * 1024
    hp = p["heads_per_cta"] * p["head_chunks"]
    assert p["workspace_bytes"] >= p["slots"] * hp * (D + 2) * 4
    assert plan(L, *shape) == p                    # deterministic


def test_force_splits(L):
    try:
        assert L.qdecode_attn_debug_force_splits(7) == 0
        assert plan(L, 1, 8, 2, [512], 256, 64, 4)["num_ctas"] == 7
        assert L.qdecode_attn_debug_force_splits(-1) == _lib.QDA_ERR_INVALID
    finally:
        L.qdecode_attn_debug_force_splits(0)
    assert plan(L, 1, 8, 2, [512], 256, 64, 4)["num_ctas"] == 8


def test_plan_argument_errors(L):
    p = _lib.QdaPlan()
    assert L.qdecode_attn_plan(1, 8, 2, _lib.int32_array([4]), 256, 64, 4, 152, 2, None) == _lib.QDA_ERR_INVALID
    assert L.qdecode_attn_plan(1, 8, 3, _lib.int32_array([4]), 256, 64, 4, 152, 2, ctypes.byref(p)) == -1
    assert L.qdecode_attn_plan(1, 8, 2, _lib.int32_array([4]), 256, 64, 5, 152, 2, ctypes.byref(p)) == -2


def call_multi(L, B=1, Lq=2, H=8, Hkv=2, N=(512,), D=256, GS=64, bits=4, dtype=1):
    p = [FAKE + 256 * i for i in range(8)]
    return L.qdecode_attn_multi(*p, B, Lq, H, Hkv, _lib.int32_array(N), D, GS, bits, dtype, None)


@pytest.mark.parametrize("kw,status", [
    (dict(Lq=0), _lib.QDA_ERR_INVALID),
    (dict(Lq=-1), _lib.QDA_ERR_INVALID),
    (dict(Lq=_lib.QDA_MAX_L + 1, N=(64,)), _lib.QDA_ERR_UNSUPPORTED),
    (dict(Lq=4, N=(3,)), _lib.QDA_ERR_INVALID),              # fewer cache rows than query positions
    (dict(B=2, Lq=3, N=(9, 2)), _lib.QDA_ERR_INVALID),
    (dict(Lq=8, H=64, Hkv=4, N=(64,)), _lib.QDA_ERR_UNSUPPORTED),   # 8 positions x 16 heads > QDA_MAX_NREP
    (dict(bits=3), _lib.QDA_ERR_UNSUPPORTED),
    (dict(H=6, Hkv=4), _lib.QDA_ERR_INVALID),
])
def test_multi_argument_errors(L, kw, status):
    assert call_multi(L, **kw) == status


def test_multi_pointer_checks(L):
    p = [FAKE + 256 * i for i in range(8)]
    p[3] = None
    assert L.qdecode_attn_multi(*p, 1, 2, 8, 2, _lib.int32_array([64]), 256, 64, 4, 1, None) == _lib.QDA_ERR_INVALID
    p = [FAKE + 256 * i for i in range(8)]
    p[7] += 2
    assert L.qdecode_attn_multi(*p, 1, 2, 8, 2, _lib.int32_array([64]), 256, 64, 4, 1, None) == _lib.QDA_ERR_ALIGN


def multi_plan(L, B, Lq, H, Hkv, N, D, GS, bits, sms=152, occ=2):
    p = _lib.QdaPlan()
    st = L.qdecode_attn_multi_plan(B, Lq, H, Hkv, _lib.int32_array(N), D, GS, bits, sms, occ, ctypes.byref(p))
    assert st == 0
    return p.as_dict()


@pytest.mark.parametrize("shape", [
    (1, 8, 2, [512], 256, 64, 4),
    (1, 16, 8, [8192], 256, 32, 8),
    (1, 16, 8, [32768], 512, 128, 4),
    (3, 24, 3, [5, 7, 9], 128, 32, 8),
])
@pytest.mark.parametrize("Lq", [1, 2, 3, 4, 8])
def test_multi_plan_serves_every_position(L, shape, Lq):
    B, H, Hkv, N, D, GS, bits = shape
    if Lq > min(N):   # a sequence shorter than its query positions
        st = L.qdecode_attn_multi_plan(B, Lq, H, Hkv, _lib.int32_array(N), D, GS, bits, 152, 2,
                                       ctypes.byref(_lib.QdaPlan()))
        assert st == _lib.QDA_ERR_INVALID
        return
    p = multi_plan(L, B, Lq, H, Hkv, N, D, GS, bits)
    assert p["heads_per_cta"] * p["head_chunks"] >= (H // Hkv) * Lq
    assert p["total_rows"] == Hkv * sum(N) and p["slots"] == p["num_ctas"] + B * Hkv
    assert p["smem_bytes"] <= 227 * 1024 and p["stages"] >= 2
    hp = p["heads_per_cta"] * p["head_chunks"]
    assert p["workspace_bytes"] >= p["slots"] * hp * (D + 2) * 4
    if Lq == 1:
        assert p == plan(L, *shape)


def test_compat_argument_errors(L):
    p = [FAKE + 256 * i for i in range(8)]
    n = _lib.int32_array([64])
    assert L.qdecode_attn_compat(*p, 1, 8, 2, n, 96, 32, 4, 1, None) == _lib.QDA_ERR_UNSUPPORTED
    assert L.qdecode_attn_compat(*p, 1, 8, 2, n, 64, 32, 3, 1, None) == _lib.QDA_ERR_UNSUPPORTED
    assert L.qdecode_attn_compat(*p, 1, 8, 3, n, 256, 32, 4, 1, None) == _lib.QDA_ERR_INVALID
    assert L.qdecode_attn_compat(*p, 1, 8, 2, n, 256, 48, 4, 1, None) == _lib.QDA_ERR_UNSUPPORTED
    q = list(p)
    q[2] = None
    assert L.qdecode_attn_compat(*q, 1, 8, 2, n, 256, 32, 4, 1, None) == _lib.QDA_ERR_INVALID


def test_qgemv_argument_errors(L):
    g = L.qdecode_qgemv
    p = [FAKE + 256 * i for i in range(5)]
    assert g(None, *p[1:], 1, 64, 1024, 64, 8, 1, None) == _lib.QDA_ERR_INVALID
    assert g(*p, 0, 64, 1024, 64, 8, 1, None) == _lib.QDA_ERR_INVALID
    assert g(*p, 1, 0, 1024, 64, 8, 1, None) == _lib.QDA_ERR_INVALID
    assert g(*p, 5, 64, 1024, 64, 8, 1, None) == _lib.QDA_ERR_UNSUPPORTED      # T > QDA_QGEMV_MAX_T
    assert g(*p, 1, 64, 1000, 8, 8, 1, None) == _lib.QDA_ERR_UNSUPPORTED       # GS
    assert g(*p, 1, 64, 1280, 64, 8, 1, None) == _lib.QDA_ERR_UNSUPPORTED      # K not a multiple of 512
    assert g(*p, 1, 64, 1024, 64, 2, 1, None) == _lib.QDA_ERR_UNSUPPORTED
    assert g(*p, 1, 64, 1024, 64, 8, 3, None) == _lib.QDA_ERR_INVALID          # fp32 input
    q = list(p)
    q[4] += 4
    assert g(*q, 1, 64, 1024, 64, 8, 1, None) == _lib.QDA_ERR_ALIGN


def test_cache_append_argument_errors(L):
    a = L.qdecode_cache_append
    old = [FAKE + 256 * i for i in range(6)]
    new = [FAKE + 4096, FAKE + 8192]
    out = [FAKE + 16384 + 256 * i for i in range(6)]
    n = _lib.int32_array([5, 0])
    def call(B=2, Hkv=2, nn=n, T=1, D=256, GS=64, bits=4, dtype=1, o=old, w=new, x=out):
        return a(*o, *w, *x, B, Hkv, nn, T, D, GS, bits, dtype, None)
    assert call(T=0) == _lib.QDA_ERR_INVALID
    assert call(Hkv=0) == _lib.QDA_ERR_INVALID
    assert call(nn=_lib.int32_array([5, -1])) == _lib.QDA_ERR_INVALID
    assert call(nn=None) == _lib.QDA_ERR_INVALID
    assert call(D=96, GS=32) == _lib.QDA_ERR_UNSUPPORTED
    assert call(bits=3) == _lib.QDA_ERR_UNSUPPORTED
    assert call(dtype=3) == _lib.QDA_ERR_INVALID
    assert call(o=[None] * 6) == _lib.QDA_ERR_INVALID             # old rows exist but no old cache
    assert call(x=[None] + out[1:]) == _lib.QDA_ERR_INVALID
    assert call(w=[new[0] + 4, new[1]]) == _lib.QDA_ERR_ALIGN


def test_host_entry_argument_errors(L):
    # the host-buffer entry point checks its arguments like qdecode_attn before touching a device
    p = [FAKE + 256 * i for i in range(8)]
    n = _lib.int32_array([64])
    h = L.qdecode_attn_host
    assert h(*p, 1, 8, 2, n, 96, 32, 4, 1, None) == _lib.QDA_ERR_UNSUPPORTED
    assert h(*p, 1, 8, 3, n, 256, 32, 4, 1, None) == _lib.QDA_ERR_INVALID
    assert h(*p, 1, 8, 2, n, 256, 32, 5, 1, None) == _lib.QDA_ERR_UNSUPPORTED
    assert h(*p, 1, 8, 2, n, 256, 32, 4, 7, None) == _lib.QDA_ERR_INVALID
    assert h(*p, 1, 8, 2, _lib.int32_array([0]), 256, 32, 4, 1, None) == _lib.QDA_ERR_INVALID
    q = list(p)
    q[7] = None
    assert h(*q, 1, 8, 2, n, 256, 32, 4, 1, None) == _lib.QDA_ERR_INVALID


def test_cta_row_magic_division():
    # the kernels split rows among C CTAs with floor(T * c / C) computed as the high half of (T * c) * ceil(2^64 / C);
    # that must equal the exact quotient for every CTA count the plan can choose (1..4096) and every row total the
    # argument checks admit (T < 2^37: int32 sequence offsets times at most 64 KV heads)
    import random
    rng = random.Random(5)
    Ts = [1, 7, 8, 4095, 4096, 65536, (1 << 31) - 1, (1 << 37) - 1, (1 << 37) - 4096] + \
         [rng.randrange(1, 1 << 37) for _ in range(40)]
    for C in list(range(1, 4097)):
        m = ((1 << 64) - 1) // C + 1
        for T in (Ts if C % 97 == 0 or C < 64 or C > 4000 else Ts[:4] + Ts[-3:]):
            for c in {1, C - 1, C // 2, rng.randrange(1, C + 1)}:
                if c <= 0 or c >= C:
                    continue
                x = T * c
                assert (x * m) >> 64 == x // C, (T, C, c)
