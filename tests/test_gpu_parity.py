"""GPU parity: the CUDA path through the C ABI against the fp64 oracle on the
same seeded inputs.

Bar: max|Y - Y_ref| / max|Y_ref| over computed rows <= 1e-2 for bf16 and
<= 1e-4 for fp32; padded query rows must be exactly zero.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from head_scaled_dot_gb300 import mha, workloads
from helpers import (TOL, computed_rows, f64, lens_list, oracle_attention_heads, oracle_forward,
                     rel_err, to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return mha.load()


def run(w, inp, **kw):
    t = to_dev(inp)
    Y = mha.forward(t["X_q"], t["X_kv"], t["W_Q"], t["W_K"], t["W_V"], t["W_O"], w.h, w.d_h,
                    w.d_vh, w.c, w.mask, inp["valid_len"], **kw)
    torch.cuda.synchronize()
    return Y


def check_full(w, inp, Y):
    ref = oracle_forward(w, inp)
    got = f64(Y)
    assert np.isfinite(got).all()
    rows = computed_rows(w, inp)
    assert np.all(got[~rows] == 0.0), "padded query rows must be exactly zero"
    err = rel_err(got[rows], ref[rows])
    assert err <= TOL[w.dtype], "rel err %.3e > %.0e" % (err, TOL[w.dtype])
    return err


# ---------------------------------------------------------------------------
# The five workloads at full size
# ---------------------------------------------------------------------------

NAMED = {"general_dims": workloads.GENERAL_DIMS, "small_dims": workloads.SMALL_DIMS,
         "simt_dims": workloads.SIMT_DIMS}


def workload(idx):
    return NAMED[idx] if idx in NAMED else workloads.WORKLOADS[idx]


@pytest.mark.parametrize("idx", [0, 1, "small_dims", "simt_dims"])
def test_workload_full_compare(idx):
    w = workload(idx)
    inp = workloads.make_inputs(w)
    check_full(w, inp, run(w, inp))


def sample_rows(w, L, rng, n=24):
    hi = L if (L is not None and not w.cross) else w.n_q
    cand = {0, 1, hi - 1, hi // 2, min(127, hi - 1), min(128, hi - 1)}
    cand |= set(rng.integers(0, hi, n).tolist())
    return sorted(c for c in cand if 0 <= c < hi)


@pytest.mark.parametrize("idx", [2, 3, 4, "general_dims"])
def test_workload_sampled_rows(idx):
    w = workload(idx)
    inp = workloads.make_inputs(w)
    got = f64(run(w, inp))
    assert np.isfinite(got).all()
    rows_ok = computed_rows(w, inp)
    assert np.all(got[~rows_ok] == 0.0)
    lens = lens_list(inp)
    rng = np.random.default_rng(w.seed)
    batches = range(w.B) if w.B <= 4 else sorted(set([0, w.B - 1] + rng.integers(0, w.B, 2).tolist()))
    worst = 0.0
    for b in batches:
        L = None if lens is None else lens[b]
        rows = sample_rows(w, L, rng)
        Yr, _ = oracle.mha_rows(f64(inp["X_q"]), f64(inp["X_kv"]), f64(inp["W_Q"]),
                                f64(inp["W_K"]), f64(inp["W_V"]), f64(inp["W_O"]), w.h, w.d_h,
                                w.d_vh, w.c, oracle.MASK_NAMES[w.mask], lens, b, rows)
        worst = max(worst, rel_err(got[b, rows], Yr))
    assert worst <= TOL[w.dtype], "rel err %.3e" % worst


@pytest.mark.parametrize("idx", [2, 3, 4, "general_dims", "small_dims", "simt_dims"])
def test_workload_full_attention_step(idx):
    """Every element of Z at full size, in the launch configuration of the
    benchmark: the attention step on the GPU's own bf16 Q, K, V (from the
    GPU's projection) against the oracle's dense attention of exactly those
    values, one (batch item, head) at a time. Padded query rows must be
    exactly zero; the metric is max|Z - Z_ref| / max|Z_ref| over the computed
    rows of the whole Z."""
    w = workload(idx)
    inp = workloads.make_inputs(w)
    t = to_dev(inp)
    lens = lens_list(inp)
    Q, K, V = mha.qkv_projection(t["X_q"], t["X_kv"], t["W_Q"], t["W_K"], t["W_V"], w.h, w.d_h,
                                 w.d_vh)
    Z = mha.attention(Q, K, V, w.c, w.mask, lens, self_attention=not w.cross)
    torch.cuda.synchronize()
    ref = oracle_attention_heads(Q, K, V, w.c, w.mask, lens, not w.cross)
    got = f64(Z)
    assert np.isfinite(got).all()
    rows = computed_rows(w, inp)
    assert np.all(got[~rows] == 0.0), "padded query rows must be exactly zero"
    err = rel_err(got[rows], ref[rows])
    assert err <= TOL[w.dtype], "rel err %.3e > %.0e" % (err, TOL[w.dtype])


# ---------------------------------------------------------------------------
# Small and ragged shapes: several tiles plus a ragged tail, all masks
# ---------------------------------------------------------------------------

SHAPES = [
    # B, n_q, n_k, d_model, h, d_h, d_vh, d_o, mask, cross, lengths
    (2, 200, 200, 128, 2, 64, 64, 128, "causal", False, None),
    (1, 1, 1, 64, 1, 64, 64, 64, "none", False, None),
    (3, 130, 130, 256, 2, 128, 128, 192, "causal_padding", False, [1, 129, 130]),
    (2, 77, 300, 64, 3, 64, 128, 136, "padding", True, [1, 300]),
    (1, 256, 256, 512, 4, 128, 64, 512, "none", False, None),
    (2, 100, 100, 64, 1, 64, 64, 64, "causal", False, None),
    (2, 383, 383, 192, 2, 64, 64, 64, "padding", False, [383, 200]),
    (1, 129, 517, 128, 2, 128, 128, 128, "none", True, None),
]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s[:8])) + "_" + s[8])
def test_small_shapes(shape, dtype):
    B, n_q, n_k, d_model, h, d_h, d_vh, d_o, mask, cross, lens = shape
    w = workloads.Workload(name="small", B=B, n_q=n_q, n_k=n_k, d_model=d_model, h=h, d_h=d_h,
                           d_vh=d_vh, d_o=d_o, mask=mask, dtype=dtype, cross=cross,
                           c=1 / math.sqrt(d_h), seed=1000 + n_q)
    inp = workloads.make_inputs(w, lengths=lens)
    check_full(w, inp, run(w, inp))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("mask", ["causal_padding", "padding"])
def test_largest_padded_batch(mask, dtype):
    """MHA_MAX_PADDED_BATCH (1024) batch items, each with its own valid length
    (1 to 40 of 40 positions): the launch parameters' length tables are full,
    and the GEMMs' zero-filled padding panels and the attention's units span
    every batch item."""
    B, T = 1024, 40
    w = workloads.Workload(name="max_batch", B=B, n_q=T, n_k=T, d_model=64, h=1, d_h=64,
                           d_vh=64, d_o=64, mask=mask, dtype=dtype, cross=False,
                           c=1 / math.sqrt(64), seed=21)
    lens = [1 + (37 * b) % T for b in range(B)]
    inp = workloads.make_inputs(w, lengths=lens)
    check_full(w, inp, run(w, inp))


# c = 0.9 is 7x the usual 1/sqrt(64): with Q and K stored in bf16 the score
# error grows with c |q| |k|, past the 1e-2 bar, so that case runs in fp32 only.
@pytest.mark.parametrize("dtype,c", [("bf16", 0.0), ("bf16", -0.2), ("bf16", 0.3),
                                     ("f32", 0.0), ("f32", -0.2), ("f32", 0.9)])
def test_scale_special_cases(c, dtype):
    w = workloads.Workload(name="scale", B=2, n_q=160, n_k=160, d_model=128, h=2, d_h=64,
                           d_vh=64, d_o=128, mask="causal", dtype=dtype, cross=False, c=c, seed=7)
    inp = workloads.make_inputs(w)
    check_full(w, inp, run(w, inp))


# ---------------------------------------------------------------------------
# Step by step, in the audit order: Q/K/V, then Z, then Y
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_steps_against_oracle_intermediates(dtype):
    w = workloads.Workload(name="steps", B=2, n_q=192, n_k=320, d_model=256, h=3, d_h=64,
                           d_vh=128, d_o=64, mask="padding", dtype=dtype, cross=True,
                           c=0.11, seed=5)
    inp = workloads.make_inputs(w, lengths=[100, 320])
    t = to_dev(inp)
    ref_Y, inter = oracle_forward(w, inp, return_intermediates=True)
    Q, K, V = mha.qkv_projection(t["X_q"], t["X_kv"], t["W_Q"], t["W_K"], t["W_V"], w.h, w.d_h,
                                 w.d_vh)
    for name, got in (("Q", Q), ("K", K), ("V", V)):
        assert rel_err(f64(got), inter[name]) <= TOL[dtype], name
    Z = mha.attention(Q, K, V, w.c, w.mask, lens_list(inp), self_attention=False)
    assert rel_err(f64(Z), inter["Z"]) <= TOL[dtype]
    Y = mha.output_projection(Z, t["W_O"], w.h, w.d_vh)
    torch.cuda.synchronize()
    assert rel_err(f64(Y), ref_Y) <= TOL[dtype]


# head sizes of 72..128 run in the 128-wide tensor-core kernels, the columns
# past d_h / d_vh read as zeros
@pytest.mark.parametrize("d", [(64, 64), (128, 128), (64, 128), (128, 64),
                               (96, 96), (72, 120), (128, 80), (64, 96), (112, 64)])
@pytest.mark.parametrize("mask", ["none", "causal", "causal_padding"])
def test_attention_step_alone(d, mask):
    """The attention kernel on bf16 Q, K, V given directly; the oracle sees the
    same bf16 values."""
    d_h, d_vh = d
    B, h, n = 2, 3, 333
    g = torch.Generator().manual_seed(d_h + d_vh + len(mask))
    Q = torch.randn((B, h, n, d_h), generator=g).bfloat16()
    K = torch.randn((B, h, n, d_h), generator=g).bfloat16()
    V = torch.randn((B, h, n, d_vh), generator=g).bfloat16()
    lens = [333, 150] if "padding" in mask else None
    c = 1 / math.sqrt(d_h)
    Z = mha.attention(Q.cuda(), K.cuda(), V.cuda(), c, mask, lens, self_attention=True)
    torch.cuda.synchronize()
    got = f64(Z)
    ref = np.zeros((B, n, h * d_vh))
    for b in range(B):
        L = None if lens is None else lens[b]
        rows = oracle.query_rows_computed(oracle.MASK_NAMES[mask], n, L, True)
        allowed = oracle.allowed_keys(oracle.MASK_NAMES[mask], n, n, L)
        for i in range(h):
            H, _ = oracle.attention(f64(Q[b, i]), f64(K[b, i]), f64(V[b, i]), c, allowed, rows)
            ref[b, :, i * d_vh:(i + 1) * d_vh] = H
    assert np.isfinite(got).all()
    assert rel_err(got, ref) <= 1e-2


@pytest.mark.parametrize("d", [(64, 64), (128, 128), (96, 96)])
@pytest.mark.parametrize("mask", ["none", "causal", "padding", "causal_padding"])
def test_attention_more_units_than_sms(d, mask):
    """More tile pairs than SMs, so that CTAs take several units in turn: the
    barrier phases carried from unit to unit, tiles with no rows (valid length
    at most 128 into the pair) and pairs that are all padding."""
    d_h, d_vh = d
    B, h, n = 24, 4, 700  # 3 tile pairs per (batch item, head): 288 units
    g = torch.Generator().manual_seed(7 * d_h + len(mask))
    Q = torch.randn((B, h, n, d_h), generator=g).bfloat16()
    K = torch.randn((B, h, n, d_h), generator=g).bfloat16()
    V = torch.randn((B, h, n, d_vh), generator=g).bfloat16()
    lens = None
    if "padding" in mask:
        lens = [700, 1, 128, 129, 255, 256, 257, 300, 511, 512, 513, 699] * 2
    c = 1 / math.sqrt(d_h)
    Z = mha.attention(Q.cuda(), K.cuda(), V.cuda(), c, mask, lens, self_attention=True)
    torch.cuda.synchronize()
    got = f64(Z)
    ref = np.zeros((B, n, h * d_vh))
    for b in range(B):
        L = None if lens is None else lens[b]
        rows = oracle.query_rows_computed(oracle.MASK_NAMES[mask], n, L, True)
        allowed = oracle.allowed_keys(oracle.MASK_NAMES[mask], n, n, L)
        for i in range(h):
            H, _ = oracle.attention(f64(Q[b, i]), f64(K[b, i]), f64(V[b, i]), c, allowed, rows)
            ref[b, :, i * d_vh:(i + 1) * d_vh] = H
        if L is not None:
            assert np.all(got[b, L:] == 0.0), "padded query rows must be exactly zero"
    assert np.isfinite(got).all()
    assert rel_err(got, ref) <= 1e-2
    # a second call on the same buffers gives the same bits
    Z2 = mha.attention(Q.cuda(), K.cuda(), V.cuda(), c, mask, lens, self_attention=True)
    torch.cuda.synchronize()
    assert torch.equal(Z.cpu(), Z2.cpu())


@pytest.mark.parametrize("d", [(64, 64), (128, 128)])
@pytest.mark.parametrize("n", [600, 640])
def test_attention_last_round_split_into_single_tiles(d, n):
    """198 tile pairs without a mask on a GPU of 152 SMs: the 46 pairs of the
    last, partly filled round run as 92 single-tile units (n = 600: the second
    tile of each last pair has no rows at all)."""
    d_h, d_vh = d
    B, h = 22, 3
    g = torch.Generator().manual_seed(n + d_h)
    Q = torch.randn((B, h, n, d_h), generator=g).bfloat16()
    K = torch.randn((B, h, n, d_h), generator=g).bfloat16()
    V = torch.randn((B, h, n, d_vh), generator=g).bfloat16()
    c = 1 / math.sqrt(d_h)
    Z = torch.full((B, n, h * d_vh), float("nan"), dtype=torch.bfloat16, device="cuda")
    mha.attention(Q.cuda(), K.cuda(), V.cuda(), c, "none", None, self_attention=True, out=Z)
    torch.cuda.synchronize()
    got = f64(Z)
    ref = np.zeros((B, n, h * d_vh))
    allowed = oracle.allowed_keys(oracle.MASK_NAMES["none"], n, n, None)
    for b in range(B):
        for i in range(h):
            H, _ = oracle.attention(f64(Q[b, i]), f64(K[b, i]), f64(V[b, i]), c, allowed)
            ref[b, :, i * d_vh:(i + 1) * d_vh] = H
    assert np.isfinite(got).all(), "every row written exactly once"
    assert rel_err(got, ref) <= 1e-2


# ---------------------------------------------------------------------------
# Statements of the pages checked on the GPU
# ---------------------------------------------------------------------------

def test_zero_output_projection_gives_exact_zero():
    w = workloads.WORKLOADS[1].with_(B=1, n_q=256, n_k=256)
    inp = workloads.make_inputs(w)
    inp["W_O"] = torch.zeros_like(inp["W_O"])
    assert torch.count_nonzero(run(w, inp)).item() == 0


def test_batch_items_are_independent():
    w = workloads.WORKLOADS[2].with_(B=3, n_q=256, n_k=256)
    inp = workloads.make_inputs(w)
    Y1 = run(w, inp).clone()
    inp2 = dict(inp)
    inp2["X_q"] = inp["X_q"].clone()
    inp2["X_q"][1] = -inp2["X_q"][1]
    Y2 = run(w, inp2)
    assert torch.equal(Y1[0], Y2[0]) and torch.equal(Y1[2], Y2[2])
    assert not torch.equal(Y1[1], Y2[1])


def test_head_permutation_with_matching_w_o_blocks():
    w = workloads.WORKLOADS[1].with_(B=1, n_q=256, n_k=256, d_model=256, h=4, d_o=256)
    inp = workloads.make_inputs(w)
    perm = [2, 0, 3, 1]
    d = w.d_h
    cols = lambda W: torch.cat([W[:, p * d:(p + 1) * d] for p in perm], dim=1)
    inp2 = dict(inp, W_Q=cols(inp["W_Q"]), W_K=cols(inp["W_K"]), W_V=cols(inp["W_V"]),
                W_O=torch.cat([inp["W_O"][p * d:(p + 1) * d] for p in perm], dim=0))
    assert rel_err(f64(run(w, inp)), f64(run(w, inp2))) <= 1e-2


def test_workspace_contents_on_entry_do_not_matter():
    w = workloads.WORKLOADS[3].with_(B=2, n_q=300, n_k=300, d_model=256, h=2, d_o=256)
    inp = workloads.make_inputs(w, lengths=[300, 131])
    t = to_dev(inp)
    nbytes = mha.workspace_size(w.B, w.n_q, w.n_k, w.d_model, w.h, w.d_h, w.d_vh, w.d_o, w.dtype)
    ws = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device="cuda")  # NaN bit patterns
    Y = mha.forward(t["X_q"], None, t["W_Q"], t["W_K"], t["W_V"], t["W_O"], w.h, w.d_h, w.d_vh,
                    w.c, w.mask, inp["valid_len"], workspace=ws)
    torch.cuda.synchronize()
    check_full(w, inp, Y)


# ---------------------------------------------------------------------------
# Failure detection without a fault: a wait that nothing completes
# ---------------------------------------------------------------------------

def test_bounded_wait_reports_timeout_and_context_survives():
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    mha.selftest_wait_timeout(err, 2_000_000)  # 2 ms
    torch.cuda.synchronize()
    assert mha.get_device_error(err) == 6  # MHA_ERR_DEVICE_TIMEOUT
    assert mha.get_device_error(err) == 0  # read resets the word
    w = workloads.WORKLOADS[1].with_(B=1, n_q=128, n_k=128)
    inp = workloads.make_inputs(w)
    check_full(w, inp, run(w, inp))


# ---------------------------------------------------------------------------
# The general form: separate key and value inputs of their own widths, and
# head sizes beyond 64 / 128 ("Multi-head attention and self-attention",
# Definition)
# ---------------------------------------------------------------------------

GENERAL = [
    # B, n_q, n_k, d_q, d_k, d_v, h, d_h, d_vh, d_o, mask, self_attention, lens
    (2, 130, 200, 64, 96, 40, 3, 64, 64, 72, "padding", False, [1, 200]),   # tensor cores
    (2, 150, 150, 64, 64, 64, 2, 128, 64, 64, "causal", True, None),        # tensor cores
    (2, 77, 140, 48, 32, 56, 3, 32, 48, 40, "none", False, None),          # tensor cores (as 64)
    (2, 90, 90, 48, 48, 48, 3, 24, 16, 40, "causal_padding", True, [90, 30]),  # CUDA cores
    (1, 100, 100, 96, 96, 96, 2, 96, 96, 96, "causal_padding", True, [61]),  # tensor cores (bf16)
    (1, 70, 90, 256, 128, 64, 2, 256, 256, 64, "padding", False, [45]),     # d = 256
]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("shape", GENERAL, ids=lambda s: "x".join(map(str, s[:10])) + "_" + s[10])
def test_general_form(shape, dtype):
    B, n_q, n_k, d_q, d_k, d_v, h, d_h, d_vh, d_o, mask, self_attn, lens = shape
    g = torch.Generator().manual_seed(n_q * 7 + d_h)
    tdt = workloads.torch_dtype(dtype)
    rnd = lambda *s, scale=1.0: (torch.randn(s, generator=g) * scale).to(tdt)
    X_q = rnd(B, n_q, d_q)
    if self_attn:
        X_k = X_v = X_q
    else:
        X_k, X_v = rnd(B, n_k, d_k), rnd(B, n_k, d_v)
    W_Q = rnd(d_q, h * d_h, scale=d_q ** -0.5)
    W_K = rnd(d_k, h * d_h, scale=d_k ** -0.5)
    W_V = rnd(d_v, h * d_vh, scale=d_v ** -0.5)
    W_O = rnd(h * d_vh, d_o, scale=(h * d_vh) ** -0.5)
    c = 1 / math.sqrt(d_h)
    dev = lambda t: t.cuda()
    Y = mha.forward_general(dev(X_q), dev(X_k), dev(X_v), dev(W_Q), dev(W_K), dev(W_V),
                            dev(W_O), h, d_h, d_vh, c, mask, lens, self_attention=self_attn)
    torch.cuda.synchronize()
    ref = oracle.mha_forward_general(f64(X_q), f64(X_k), f64(X_v), f64(W_Q), f64(W_K), f64(W_V),
                                     f64(W_O), h, d_h, d_vh, c, oracle.MASK_NAMES[mask], lens,
                                     self_attn)
    got = f64(Y)
    assert np.isfinite(got).all()
    rows = np.ones((B, n_q), dtype=bool)
    if self_attn and lens is not None:
        for b in range(B):
            rows[b, lens[b]:] = False
        assert np.all(got[~rows] == 0.0)
    assert rel_err(got[rows], ref[rows]) <= TOL[dtype]


@pytest.mark.parametrize("dtype,d", [("bf16", 64), ("bf16", 96), ("f32", 64)])
def test_head_gate_zeroes_a_head_like_its_w_o_block(dtype, d):
    """Head zeroing at the named location (the head's block of the
    concatenation, before W_O) equals zeroing that head's rows of W_O, and the
    gates match the oracle's."""
    B, n, d_model, h = 2, 140, 128, 4
    g = torch.Generator().manual_seed(300 + d)
    tdt = workloads.torch_dtype(dtype)
    rnd = lambda *s, scale=1.0: (torch.randn(s, generator=g) * scale).to(tdt)
    X = rnd(B, n, d_model)
    W_Q, W_K = rnd(d_model, h * d, scale=d_model ** -0.5), rnd(d_model, h * d, scale=d_model ** -0.5)
    W_V = rnd(d_model, h * d, scale=d_model ** -0.5)
    W_O = rnd(h * d, d_model, scale=(h * d) ** -0.5)
    gate = [1.0, 0.0, 0.5, 1.0]
    c = 1 / math.sqrt(d)
    dev = lambda t: t.cuda()
    Yg = mha.forward_general(dev(X), dev(X), dev(X), dev(W_Q), dev(W_K), dev(W_V), dev(W_O), h, d,
                             d, c, "causal", None, self_attention=True, head_gate=gate)
    W_O0 = W_O.clone()
    W_O0[d:2 * d] = 0
    Yw = mha.forward_general(dev(X), dev(X), dev(X), dev(W_Q), dev(W_K), dev(W_V), dev(W_O0),
                             h, d, d, c, "causal", None, self_attention=True,
                             head_gate=[1.0, 1.0, 0.5, 1.0])
    torch.cuda.synchronize()
    ref = oracle.mha_forward_general(f64(X), f64(X), f64(X), f64(W_Q), f64(W_K), f64(W_V),
                                     f64(W_O), h, d, d, c, oracle.MASK_CAUSAL, None, True,
                                     head_gate=gate)
    assert rel_err(f64(Yg), ref) <= TOL[dtype]
    # zeroing by gate or by W_O rows: the Z blocks that reach W_O differ only
    # in head 1, whose W_O rows are zero in the second call
    assert rel_err(f64(Yg), f64(Yw)) <= TOL[dtype]


@pytest.mark.parametrize("dtype,d", [("bf16", 64), ("bf16", 128), ("f32", 64)])
def test_more_heads_than_gate_slots_without_a_gate(dtype, d):
    """h = 1025 heads (one past the per-head gate table) with no gate: every
    head, the last ones included, is scaled by exactly 1."""
    B, h, n = 1, 1025, 130
    g = torch.Generator().manual_seed(1025 + d)
    tdt = workloads.torch_dtype(dtype)
    Q = torch.randn((B, h, n, d), generator=g).to(tdt)
    K = torch.randn((B, h, n, d), generator=g).to(tdt)
    V = torch.randn((B, h, n, d), generator=g).to(tdt)
    c = 1 / math.sqrt(d)
    Z = mha.attention(Q.cuda(), K.cuda(), V.cuda(), c, "causal", None, self_attention=True)
    torch.cuda.synchronize()
    ref = oracle_attention_heads(Q, K, V, c, "causal", None, True)
    assert rel_err(f64(Z), ref) <= TOL[dtype]


@pytest.mark.parametrize("d", [(64, 64), (128, 128)])
def test_schedule_of_one_shape_with_new_lengths(d):
    """The host keeps the attention schedule of recent (shape, lengths)
    calls. The same shape with other valid lengths (here every few calls,
    returning to earlier lengths) must be computed for its own lengths: the
    kernels read the lengths of the call, whatever schedule is reused."""
    d_h, d_vh = d
    B, h, n = 10, 4, 900
    g = torch.Generator().manual_seed(900 + d_h)
    Q = torch.randn((B, h, n, d_h), generator=g).bfloat16()
    K = torch.randn((B, h, n, d_h), generator=g).bfloat16()
    V = torch.randn((B, h, n, d_vh), generator=g).bfloat16()
    c = 1 / math.sqrt(d_h)
    sets = [[900, 1, 129, 256, 257, 500, 640, 641, 899, 384],
            [300, 900, 900, 2, 700, 128, 513, 65, 900, 880],
            [900] * 10]
    Qd, Kd, Vd = Q.cuda(), K.cuda(), V.cuda()
    for lens in sets + sets[:2]:
        Z = mha.attention(Qd, Kd, Vd, c, "causal_padding", lens, self_attention=True)
        torch.cuda.synchronize()
        ref = oracle_attention_heads(Q, K, V, c, "causal_padding", lens, True)
        got = f64(Z)
        for b, L in enumerate(lens):
            assert np.all(got[b, L:] == 0.0)
        assert rel_err(got, ref) <= 1e-2, lens
