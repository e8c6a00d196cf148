"""GPU parity of mha_attention_decode (new query rows over a key/value cache,
split over the keys and merged with the summary merge) against the oracle's
dense restatement, through the C ABI."""

import numpy as np
import pytest
import torch

import oracle
from head_scaled_dot_gb300 import mha, workloads
from helpers import TOL, f64, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return mha.load()


CASES = [
    # dtype, B, h, n_q, n_k, d_h, d_vh, cache lengths, causal_tail
    ("bf16", 3, 4, 1, 4096, 128, 128, [1, 4096, 2500], False),
    ("bf16", 2, 3, 3, 1000, 64, 64, [3, 777], True),
    ("bf16", 2, 2, 8, 600, 96, 40, [600, 9], False),
    ("bf16", 1, 2, 11, 700, 256, 256, [513], True),
    ("f32", 2, 3, 1, 3000, 64, 64, [2999, 1], False),
    ("f32", 2, 2, 5, 900, 36, 20, [5, 900], True),
    ("f32", 1, 1, 9, 1, 128, 128, None, False),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "%s_B%d_h%d_nq%d_nk%d_d%d_%d_%s" % (
    c[0], c[1], c[2], c[3], c[4], c[5], c[6], "tail" if c[8] else "all"))
def test_decode_matches_oracle(case):
    dtype, B, h, n_q, n_k, d_h, d_vh, lens, tail = case
    g = torch.Generator().manual_seed(n_k + d_h + n_q)
    tdt = workloads.torch_dtype(dtype)
    Q = torch.randn((B, h, n_q, d_h), generator=g).to(tdt)
    K = torch.randn((B, h, n_k, d_h), generator=g).to(tdt)
    V = torch.randn((B, h, n_k, d_vh), generator=g).to(tdt)
    c = d_h ** -0.5
    Z = mha.attention_decode(Q.cuda(), K.cuda(), V.cuda(), c, lens, tail)
    torch.cuda.synchronize()
    ref = oracle.attention_decode(f64(Q), f64(K), f64(V), c, lens, tail)
    got = f64(Z)
    assert np.isfinite(got).all()
    assert rel_err(got, ref) <= TOL[dtype]


def test_decode_workload_full_size():
    """The decode workload the benchmark times: B=16, h=8, d=128, one new row
    per sequence over a cache of capacity 8192 holding 4096..8192 positions."""
    w = workloads.DECODE
    inp = workloads.make_decode_inputs(w)
    Z = mha.attention_decode(inp["Q"].cuda(), inp["K"].cuda(), inp["V"].cuda(), w.c,
                             inp["cache_len"], False)
    torch.cuda.synchronize()
    ref = oracle.attention_decode(f64(inp["Q"]), f64(inp["K"]), f64(inp["V"]), w.c,
                                  inp["cache_len"], False)
    assert rel_err(f64(Z), ref) <= TOL["bf16"]


def test_decode_is_the_attention_step_with_a_padding_mask():
    """One new row per sequence seeing its whole cache is mha_attention with
    n_q = 1 and a padding mask on the keys (two different kernels)."""
    B, h, n_k, d = 4, 2, 1500, 64
    g = torch.Generator().manual_seed(5)
    Q = torch.randn((B, h, 1, d), generator=g).bfloat16().cuda()
    K = torch.randn((B, h, n_k, d), generator=g).bfloat16().cuda()
    V = torch.randn((B, h, n_k, d), generator=g).bfloat16().cuda()
    lens = [1500, 1, 700, 129]
    Zd = mha.attention_decode(Q, K, V, 0.125, lens, False)
    Za = mha.attention(Q, K, V, 0.125, "padding", lens, self_attention=False)
    torch.cuda.synchronize()
    assert rel_err(f64(Zd), f64(Za)) <= TOL["bf16"]


def test_decode_workspace_contents_do_not_matter():
    B, h, n_q, n_k, d = 2, 2, 2, 900, 64
    g = torch.Generator().manual_seed(6)
    Q = torch.randn((B, h, n_q, d), generator=g).bfloat16().cuda()
    K = torch.randn((B, h, n_k, d), generator=g).bfloat16().cuda()
    V = torch.randn((B, h, n_k, d), generator=g).bfloat16().cuda()
    ws = torch.full((mha.decode_workspace_size(B, n_q, n_k, h, d),), 0xFF, dtype=torch.uint8,
                    device="cuda")
    Z1 = mha.attention_decode(Q, K, V, 0.125, [900, 400], True, workspace=ws).clone()
    ws.fill_(0x7F)
    Z2 = mha.attention_decode(Q, K, V, 0.125, [900, 400], True, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(Z1, Z2)
