"""The projection steps on their own (tensor-core GEMM, bf16): tile edges,
ragged tails, both accumulator buffers and the head-split epilogue, against
the oracle's projections on the same bf16 values."""

import numpy as np
import pytest
import torch

import oracle
from head_scaled_dot_gb300 import mha
from helpers import f64, rel_err

pytestmark = pytest.mark.gpu


def bf16(shape, g, scale=1.0):
    return (torch.randn(shape, generator=g) * scale).bfloat16()


@pytest.mark.parametrize("M,K,N", [
    (128, 64, 256),     # one tile
    (256, 128, 512),    # several tiles, two k-blocks
    (300, 200, 136),    # ragged M, K and N (N tail inside a 32-column chunk)
    (4096, 1024, 1024),  # many tiles per CTA: both TMEM buffers reused
    (8, 64, 64),
])
def test_output_projection_gemm(M, K, N):
    g = torch.Generator().manual_seed(M + K + N)
    Z = bf16((1, M, K), g)
    W = bf16((K, N), g, K ** -0.5)
    Y = mha.output_projection(Z.cuda(), W.cuda(), 1, K)
    torch.cuda.synchronize()
    ref = f64(Z)[0] @ f64(W)
    got = f64(Y)[0]
    assert np.isfinite(got).all()
    assert rel_err(got, ref) <= 4e-3


def test_output_projection_gemm_exact_on_integers():
    """Small integers are exact in bf16 and in the fp32 accumulator, so the
    result must match bit for bit: catches any swizzle or descriptor slip."""
    g = torch.Generator().manual_seed(3)
    M, K, N = 256, 192, 256
    Z = torch.randint(-3, 4, (1, M, K), generator=g).bfloat16()
    W = torch.randint(-3, 4, (K, N), generator=g).bfloat16()
    Y = mha.output_projection(Z.cuda(), W.cuda(), 1, K)
    torch.cuda.synchronize()
    ref = f64(Z)[0] @ f64(W)
    assert np.array_equal(f64(Y)[0], ref)


@pytest.mark.parametrize("B,T,n_k,d_model,h,d_h,d_vh,cross", [
    (2, 256, 256, 128, 2, 64, 64, False),
    (1, 200, 200, 256, 3, 128, 64, False),
    (2, 100, 333, 64, 2, 64, 128, True),
])
def test_qkv_projection_head_split(B, T, n_k, d_model, h, d_h, d_vh, cross):
    g = torch.Generator().manual_seed(B * T + h)
    X = bf16((B, T, d_model), g)
    Xkv = bf16((B, n_k, d_model), g) if cross else None
    WQ = bf16((d_model, h * d_h), g, d_model ** -0.5)
    WK = bf16((d_model, h * d_h), g, d_model ** -0.5)
    WV = bf16((d_model, h * d_vh), g, d_model ** -0.5)
    WO = bf16((h * d_vh, 8), g)
    Q, K, V = mha.qkv_projection(X.cuda(), None if Xkv is None else Xkv.cuda(), WQ.cuda(),
                                 WK.cuda(), WV.cuda(), h, d_h, d_vh)
    torch.cuda.synchronize()
    _, inter = oracle.mha_forward(f64(X), f64(Xkv), f64(WQ), f64(WK), f64(WV), f64(WO), h, d_h,
                                  d_vh, 0.1, return_intermediates=True)
    for name, got in (("Q", Q), ("K", K), ("V", V)):
        assert rel_err(f64(got), inter[name]) <= 4e-3, name
