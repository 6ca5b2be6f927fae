"""GPU cache append (qdecode_cache_append): the appended cache must equal the oracle's bit for bit, and decoding
over a cache grown step by step must match the oracle."""
import numpy as np
import pytest
import torch

import oracle as O
import attention_quantized_kv_split_gb300 as qda
from attention_quantized_kv_split_gb300 import build, synth

from harness import TOL, TORCH_DT, upload_cache

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    qda.lib()


def to_cache(arrays, N, Hkv, D, GS, bits, dtype):
    dev = upload_cache(*arrays, dtype)
    return qda.QuantizedKV(*dev, N, Hkv, D, GS, bits)


def host_arrays(cache, dtype):
    def sc(t):
        return O.from_bits16(t.view(torch.int16).cpu().numpy().view(np.uint16), dtype)
    return (cache.kp.cpu().numpy().view(np.uint32), sc(cache.ks), sc(cache.kb),
            cache.vp.cpu().numpy().view(np.uint32), sc(cache.vs), sc(cache.vb))


@pytest.mark.parametrize("D,GS,bits,dtype", [(64, 32, 4, "bf16"), (128, 64, 8, "fp16"), (256, 32, 8, "bf16"),
                                             (256, 64, 4, "fp16"), (512, 128, 4, "bf16"), (512, 32, 8, "bf16")])
@pytest.mark.parametrize("T", [1, 3])
def test_append_bit_exact(D, GS, bits, dtype, T):
    rng = np.random.default_rng(D + GS + bits + T)
    N, Hkv = [17, 0, 300, 1], 3
    B = len(N)
    rows = Hkv * sum(N)
    old = O.quantize_cache(rng.standard_normal((rows, D)).astype(np.float32),
                           rng.standard_normal((rows, D)).astype(np.float32), GS, bits, dtype)
    Kn = rng.standard_normal((B, Hkv, T, D)).astype(np.float32) * 3
    Vn = rng.standard_normal((B, Hkv, T, D)).astype(np.float32)
    cache = to_cache(old, N, Hkv, D, GS, bits, dtype)
    new = cache.append(torch.from_numpy(Kn).cuda(), torch.from_numpy(Vn).cuda())
    torch.cuda.synchronize()
    assert new.N == [n + T for n in N]
    got = host_arrays(new, dtype)
    ref = O.cache_append(old, N, Kn, Vn, Hkv, D, GS, bits, dtype)
    for g, r in zip(got, ref):
        np.testing.assert_array_equal(g, r)


def test_append_from_empty():
    rng = np.random.default_rng(3)
    B, Hkv, T, D, GS, bits = 2, 2, 4, 128, 32, 4
    empty = qda.QuantizedKV.empty([0, 0], Hkv, D, GS, bits, torch.bfloat16)
    Kn = rng.standard_normal((B, Hkv, T, D)).astype(np.float32)
    Vn = rng.standard_normal((B, Hkv, T, D)).astype(np.float32)
    new = empty.append(torch.from_numpy(Kn).cuda(), torch.from_numpy(Vn).cuda())
    torch.cuda.synchronize()
    ref = O.quantize_cache(Kn.reshape(-1, D), Vn.reshape(-1, D), GS, bits, "bf16")
    for g, r in zip(host_arrays(new, "bf16"), ref):
        np.testing.assert_array_equal(g, r)


def test_decode_loop_grows_the_cache():
    # a few decode steps: append one token per sequence, then attend over the longer cache
    w = synth.small(B=2, H=8, Hkv=2, D=256, N=(64, 9), bits=8, GS=32, seed=12)
    rng = np.random.default_rng(12)
    N = list(w.N)
    rows = w.Hkv * sum(N)
    arrays = O.quantize_cache(rng.standard_normal((rows, w.D)).astype(np.float32),
                              rng.standard_normal((rows, w.D)).astype(np.float32), w.GS, w.bits, "bf16")
    cache = to_cache(arrays, N, w.Hkv, w.D, w.GS, w.bits, "bf16")
    for step in range(4):
        Kn = rng.standard_normal((w.B, w.Hkv, 1, w.D)).astype(np.float32)
        Vn = rng.standard_normal((w.B, w.Hkv, 1, w.D)).astype(np.float32)
        cache = cache.append(torch.from_numpy(Kn).cuda(), torch.from_numpy(Vn).cuda())
        arrays = O.cache_append(arrays, N, Kn, Vn, w.Hkv, w.D, w.GS, w.bits, "bf16")
        N = [n + 1 for n in N]
        q = torch.from_numpy(rng.standard_normal((w.B, w.H, w.D)).astype(np.float32)).to(torch.bfloat16)
        out = qda.decode_attention(q.cuda(), cache)
        torch.cuda.synchronize()
        ref = O.attention_packed(q.double().numpy(), *arrays, N, w.H, w.Hkv, w.D, w.GS, w.bits)
        g = out.double().cpu().numpy()
        for (b, h), o in ref.items():
            assert np.abs(g[b, h] - o).max() <= TOL["bf16"] * np.abs(o).max(), (step, b, h)
