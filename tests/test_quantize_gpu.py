"""GPU quantize-and-append: the library's quantizer must write exactly the oracle quantizer's bytes."""
import numpy as np
import pytest
import torch

import oracle as O
import attention_quantized_kv_split_gb300 as qda
from attention_quantized_kv_split_gb300 import build

from harness import TORCH_DT

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    qda.lib()


def gpu_quantize(x: np.ndarray, GS, bits, dtype):
    rows, D = x.shape
    xd = torch.from_numpy(x).cuda()
    packed = torch.empty((rows, D * bits // 32), dtype=torch.int32, device="cuda")
    sc = torch.empty((rows, D // GS), dtype=TORCH_DT[dtype], device="cuda")
    bi = torch.empty_like(sc)
    qda.qdecode_quantize(xd, GS, bits, TORCH_DT[dtype], packed, sc, bi)
    return packed.cpu().numpy().view(np.uint32), sc.float().cpu().numpy(), bi.float().cpu().numpy()


def inputs(rows, D, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, D)).astype(np.float32)
    x[0] = 0.25                                                # zero-range groups
    x[1] = np.arange(D) % 16 - 1                               # closed-form integer groups
    x[2] *= 1e4                                                # large range
    x[3] *= 1e-30                                              # tiny range (scale may round to 0 in fp16)
    x[4, ::3] *= 20                                            # outliers
    return x


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("D,GS", [(64, 32), (64, 64), (128, 32), (128, 128), (256, 32), (256, 64), (512, 128),
                                  (512, 32)])
def test_quantizer_bit_exact(D, GS, bits, dtype):
    x = inputs(1031, D, D + GS + bits)
    kp, ks, kb = O.quantize_cache(x, x, GS, bits, dtype)[:3]
    gp, gs, gb = gpu_quantize(x, GS, bits, dtype)
    assert np.array_equal(gp, kp)
    assert np.array_equal(gs, ks)
    assert np.array_equal(gb, kb)


def test_append_into_cache_rows():
    # quantizing into a slice of a cache writes only those rows
    D, GS, bits, dtype = 256, 64, 4, "bf16"
    cache = qda.QuantizedKV.empty([10], 1, D, GS, bits, torch.bfloat16)
    for t in (cache.kp, cache.vp):
        t.fill_(-1)
    x = inputs(8, D, 1)[5:8].copy()
    cache.quantize_into(0, 0, torch.from_numpy(x).cuda(), torch.from_numpy(x).cuda(), row0=4)
    kp = O.quantize_cache(x, x, GS, bits, dtype)[0]
    got = cache.kp.cpu().numpy().view(np.uint32)
    assert np.array_equal(got[4:7], kp)
    assert np.all(got[:4] == 0xFFFFFFFF) and np.all(got[7:] == 0xFFFFFFFF)
