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


@pytest.mark.parametrize("B,T,n_k,lens,cross", [
    (3, 300, 300, [300, 131, 1], False),   # panels span batch items (T % 128 != 0)
    (2, 1024, 1024, [129, 1000], False),
    (4, 64, 200, [1, 200, 129, 128], True),  # cross: keys only
])
def test_qkv_projection_computes_only_the_rows_attention_reads(B, T, n_k, lens, cross):
    """With a padding mask the projection writes the rows below valid_len[b]
    rounded up to 128 (K and V; Q too for self-attention) and leaves every
    other row as it was (NaN here)."""
    d_model, h, d_h, d_vh = 128, 2, 64, 128
    g = torch.Generator().manual_seed(B * T + n_k)
    X = bf16((B, T, d_model), g)
    Xkv = bf16((B, n_k, d_model), g) if cross else None
    WQ = bf16((d_model, h * d_h), g, d_model ** -0.5)
    WK = bf16((d_model, h * d_h), g, d_model ** -0.5)
    WV = bf16((d_model, h * d_vh), g, d_model ** -0.5)
    nk = n_k if cross else T
    nan = lambda *s: torch.full(s, float("nan"), dtype=torch.bfloat16, device="cuda")
    out = (nan(B, h, T, d_h), nan(B, h, nk, d_h), nan(B, h, nk, d_vh))
    Q, K, V = mha.qkv_projection(X.cuda(), None if Xkv is None else Xkv.cuda(), WQ.cuda(),
                                 WK.cuda(), WV.cuda(), h, d_h, d_vh, mask="padding",
                                 valid_len=lens, out=out)
    torch.cuda.synchronize()
    _, inter = oracle.mha_forward(f64(X), f64(Xkv), f64(WQ), f64(WK), f64(WV),
                                  f64(bf16((h * d_vh, 8), g)), h, d_h, d_vh, 0.1,
                                  return_intermediates=True)
    for name, got, rows_sel in (("Q", Q, not cross), ("K", K, True), ("V", V, True)):
        got = f64(got)
        n = got.shape[2]
        for b in range(B):
            need = min(n, (lens[b] + 127) // 128 * 128) if rows_sel else n
            assert rel_err(got[b, :, :need], inter[name][b, :, :need]) <= 4e-3, name
            # rows past `need` may be written only where a 128-row panel of
            # the flattened B * n rows also holds needed rows of a neighbour
            panel_lo = ((b * n + need) + 127) // 128 * 128 - b * n
            nxt = (b + 1) * n  # the next batch item's rows start there
            untouched_to = min(n, ((nxt // 128) * 128 - b * n) if b + 1 < B else n)
            if panel_lo < untouched_to:
                assert np.isnan(got[b, :, panel_lo:untouched_to]).all(), name


@pytest.mark.parametrize("B,T,lens", [(3, 300, [300, 1, 131]), (2, 1024, [100, 1024]),
                                      (5, 128, [1, 128, 64, 127, 2])])
def test_output_projection_zero_rows_past_the_valid_length(B, T, lens):
    """Rows i >= valid_len[b] of Y are exact zeros (their Z rows are zeros,
    as the attention step writes them); panels made only of such rows are
    written without a product, the rest are multiplied as usual."""
    K, N = 192, 256
    g = torch.Generator().manual_seed(B * T)
    Z = bf16((B, T, K), g)
    for b, L in enumerate(lens):
        Z[b, L:] = 0
    W = bf16((K, N), g, K ** -0.5)
    Y = torch.full((B, T, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    mha.output_projection(Z.cuda(), W.cuda(), 1, K, valid_len=lens, out=Y)
    torch.cuda.synchronize()
    got = f64(Y)
    ref = f64(Z) @ f64(W)
    assert np.isfinite(got).all()
    for b, L in enumerate(lens):
        assert np.all(got[b, L:] == 0.0)
    assert rel_err(got, ref) <= 4e-3


def test_general_form_three_inputs_three_groups():
    """Separate X_q, X_k, X_v buffers (three A operands, three groups of the
    grouped launch) against the oracle, padding on keys."""
    B, n_q, n_k, d_q, d_k, d_v, h, d = 2, 140, 300, 64, 96, 128, 2, 64
    g = torch.Generator().manual_seed(77)
    X_q, X_k, X_v = bf16((B, n_q, d_q), g), bf16((B, n_k, d_k), g), bf16((B, n_k, d_v), g)
    W_Q, W_K = bf16((d_q, h * d), g, d_q ** -0.5), bf16((d_k, h * d), g, d_k ** -0.5)
    W_V, W_O = bf16((d_v, h * d), g, d_v ** -0.5), bf16((h * d, 72), g, (h * d) ** -0.5)
    lens = [5, 300]
    Y = mha.forward_general(X_q.cuda(), X_k.cuda(), X_v.cuda(), W_Q.cuda(), W_K.cuda(),
                            W_V.cuda(), W_O.cuda(), h, d, d, 0.125, "padding", lens)
    torch.cuda.synchronize()
    ref = oracle.mha_forward_general(f64(X_q), f64(X_k), f64(X_v), f64(W_Q), f64(W_K), f64(W_V),
                                     f64(W_O), h, d, d, 0.125, oracle.MASK_PADDING, lens, False)
    assert rel_err(f64(Y), ref) <= 1e-2


@pytest.mark.parametrize("B,T,lens,cross", [
    (5, 1408, None, False),               # 55 panels (odd): one pair's second tile has no rows
    (5, 1408, [1408, 300, 1217, 1408, 1000], False),  # 43 selected panels (odd)
    (3, 512, None, True),                 # cross: K and V over 1536 rows of X_kv per item
])
def test_qkv_projection_in_cta_pairs_exact_on_integers(B, T, lens, cross):
    """Grouped projections with many tiles run in pairs of CTAs (one 256-row
    tile, cta_group::2 MMAs, each CTA holding half of the W tile). Small
    integers are exact in bf16
    and in the fp32 accumulator, so Q, K and V must match bit for bit, also
    for a pair whose second panel is past the last one and with only the
    selected panels of a padding mask computed."""
    g = torch.Generator().manual_seed(B * T + (lens is not None) + 2 * cross)
    d_model, h, d_h, d_vh = 256, 16, 128, 128  # 24 N tiles of 256 per M panel: > 608 tiles
    n_k = 3 * T if cross else T
    X = torch.randint(-2, 3, (B, T, d_model), generator=g).bfloat16()
    Xkv = torch.randint(-2, 3, (B, n_k, d_model), generator=g).bfloat16() if cross else None
    WQ = torch.randint(-2, 3, (d_model, h * d_h), generator=g).bfloat16()
    WK = torch.randint(-2, 3, (d_model, h * d_h), generator=g).bfloat16()
    WV = torch.randint(-2, 3, (d_model, h * d_vh), generator=g).bfloat16()
    mask = "padding" if lens is not None else "none"
    Q, K, V = mha.qkv_projection(X.cuda(), None if Xkv is None else Xkv.cuda(), WQ.cuda(),
                                 WK.cuda(), WV.cuda(), h, d_h, d_vh, mask=mask, valid_len=lens)
    torch.cuda.synchronize()
    src_kv = Xkv if cross else X
    for name, got, src, Wt, d, n in (("Q", Q, X, WQ, d_h, T), ("K", K, src_kv, WK, d_h, n_k),
                                     ("V", V, src_kv, WV, d_vh, n_k)):
        ref = (f64(src) @ f64(Wt)).reshape(B, n, h, d).transpose(0, 2, 1, 3)
        got = f64(got)
        for b in range(B):
            rows = n if lens is None else min(n, -(-lens[b] // 128) * 128)
            assert np.array_equal(got[b, :, :rows], ref[b, :, :rows]), (name, b)
