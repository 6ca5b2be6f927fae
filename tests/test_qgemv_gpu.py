"""GPU parity of the affine-quantized weight GEMV (qdecode_qgemv) against the fp64 oracle, through the C ABI.

The kernel forms exact codes and accumulates in fp32; each output is a sum of K products, so its error is a few
fp32 ulps of the sum of |x * w|. Tolerance per output row t: max|delta| <= 1e-4 * max|y[t]| for fp32 outputs and
1e-2 * max|y[t]| for bf16/fp16 outputs (the output rounding)."""
import numpy as np
import pytest
import torch

import oracle as O
import attention_quantized_kv_split_gb300 as qda
from attention_quantized_kv_split_gb300 import build

from harness import TOL, TORCH_DT

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    qda.lib()


def make(T, N, K, GS, bits, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    w = torch.randn(N, K, generator=g).numpy()
    x = torch.randn(T, K, generator=g).to(TORCH_DT[dtype])
    c, s, b = O.quantize(w, GS, bits, dtype)
    wp = O.pack(c, bits)
    dev = (torch.from_numpy(wp.view(np.int32)).cuda(),
           torch.from_numpy(O.bits16(s, dtype).view(np.int16)).view(TORCH_DT[dtype]).cuda(),
           torch.from_numpy(O.bits16(b, dtype).view(np.int16)).view(TORCH_DT[dtype]).cuda())
    ref = O.qgemv(x.to(torch.float64).numpy(), wp, s, b, K, GS, bits)
    return x, dev, ref


def check(T, N, K, GS, bits, dtype="bf16", out="fp32", seed=0):
    x, dev, ref = make(T, N, K, GS, bits, dtype, seed)
    y = torch.full((T, N), float("nan"), dtype=TORCH_DT[out], device="cuda")
    qda.qdecode_qgemv(x.cuda(), *dev, y, GS, bits)
    torch.cuda.synchronize()
    g = y.to(torch.float64).cpu().numpy()
    assert np.all(np.isfinite(g))
    for t in range(T):
        err = np.abs(g[t] - ref[t]).max()
        assert err <= TOL[out] * np.abs(ref[t]).max(), (t, err)
    return y


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("GS", [32, 64, 128])
@pytest.mark.parametrize("T", [1, 2, 3, 4])
def test_qgemv_sweep(bits, GS, T):
    check(T, 97, 1024, GS, bits, seed=bits * 100 + GS + T)


@pytest.mark.parametrize("N", [1, 3, 31, 32, 33, 1000])
def test_qgemv_row_counts(N):
    check(2, N, 512, 64, 8, seed=N)
    check(1, N, 1024, 32, 4, seed=N + 1)


@pytest.mark.parametrize("K,N", [(14336, 4096), (8192, 512), (3072, 7)])
def test_qgemv_k_split(K, N):
    # few row groups: K is split across warps (2 or 4 parts) to fill the GPU
    check(1, N, K, 64, 8, seed=K + N)
    check(3, N, K, 128, 4, out="bf16", seed=K + N + 1)


@pytest.mark.parametrize("dtype,out", [("bf16", "bf16"), ("fp16", "fp16"), ("fp16", "fp32"), ("bf16", "fp16")])
def test_qgemv_dtypes(dtype, out):
    check(1, 300, 2048, 64, 8, dtype, out, seed=7)
    check(4, 300, 2048, 32, 4, dtype, out, seed=8)


def test_qgemv_large_and_repeatable():
    # an MLP-sized matrix (K = 4096, N = 14336), as the bench times it
    y1 = check(1, 14336, 4096, 64, 8, seed=11)
    x, dev, _ = make(1, 14336, 4096, 64, 8, "bf16", 11)
    y2 = torch.empty_like(y1)
    qda.qdecode_qgemv(x.cuda(), *dev, y2, 64, 8)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)


@pytest.mark.parametrize("T,bits", [(3, 8), (4, 4)])
def test_qgemv_several_inputs_large_and_repeatable(T, bits):
    # three or four input rows at an MLP size (the kernel's largest register use, one CTA per SM); the lanes' sums
    # meet in a fixed order, so two calls agree bit for bit
    y1 = check(T, 14336, 4096, 64, bits, seed=12 + T)
    x, dev, _ = make(T, 14336, 4096, 64, bits, "bf16", 12 + T)
    y2 = torch.empty_like(y1)
    qda.qdecode_qgemv(x.cuda(), *dev, y2, 64, bits)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
