"""GPU parity of the split over the keys: the keys of each (query tile,
head) cut into ranges on separate thread blocks, each range summarised on
its own and the summaries merged ("Stable summary of an attention key block",
Definition: the summary of a union of disjoint key sets is the merge of
theirs). Compared element by element with the fp64 oracle's dense attention
of the same bf16 Q, K, V; bar max|Z - Z_ref| / max|Z_ref| <= 1e-2."""

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


def oracle_z(Q, K, V, c, mask, lens, self_attention):
    B, h, n_q, _ = Q.shape
    n_k, d_vh = K.shape[2], V.shape[3]
    ref = np.zeros((B, n_q, h * d_vh))
    for b in range(B):
        L = None if lens is None else lens[b]
        rows = oracle.query_rows_computed(oracle.MASK_NAMES[mask], n_q, L, self_attention)
        allowed = oracle.allowed_keys(oracle.MASK_NAMES[mask], n_q, n_k, L)
        for i in range(h):
            H, _ = oracle.attention(f64(Q[b, i]), f64(K[b, i]), f64(V[b, i]), c, allowed, rows)
            ref[b, :, i * d_vh:(i + 1) * d_vh] = H
    return ref


def draw(B, h, n_q, n_k, d_h, d_vh, seed):
    g = torch.Generator().manual_seed(seed)
    Q = torch.randn((B, h, n_q, d_h), generator=g).bfloat16()
    K = torch.randn((B, h, n_k, d_h), generator=g).bfloat16()
    V = torch.randn((B, h, n_k, d_vh), generator=g).bfloat16()
    return Q, K, V


@pytest.mark.parametrize("w", workloads.LONG_KEYS, ids=lambda w: w.name)
def test_long_key_workload_full_size(w):
    """16 (batch item, head) query tiles against 32768 keys at full size: the
    automatic choice splits the keys (nine ranges of 29 blocks on 152 SMs);
    every element of Z against the oracle on the GPU's own Q, K, V, and every
    row of Y against the oracle's whole forward pass."""
    grid, rec = mha.attention_plan(w.B, w.n_q, w.n_k, w.h, w.d_h, w.d_vh, w.mask, None,
                                   not w.cross, torch.cuda.get_device_properties(0)
                                   .multi_processor_count, nsplit=0)
    assert len(rec) > w.B * w.h and np.any(rec[:, 5] > 0), "the keys are split"
    inp = workloads.make_inputs(w)
    t = to_dev(inp)
    Q, K, V = mha.qkv_projection(t["X_q"], t["X_kv"], t["W_Q"], t["W_K"], t["W_V"], w.h, w.d_h,
                                 w.d_vh)
    Z = mha.attention_split(Q, K, V, w.c, w.mask, None, self_attention=False, nsplit=0)
    torch.cuda.synchronize()
    ref = oracle_attention_heads(Q, K, V, w.c, w.mask, None, False)
    got = f64(Z)
    assert np.isfinite(got).all()
    assert rel_err(got, ref) <= TOL["bf16"]
    # the whole forward pass (which takes the same split) against the oracle
    Y = mha.forward(t["X_q"], t["X_kv"], t["W_Q"], t["W_K"], t["W_V"], t["W_O"], w.h, w.d_h,
                    w.d_vh, w.c, w.mask, None)
    torch.cuda.synchronize()
    ref_y = oracle_forward(w, inp)
    assert rel_err(f64(Y), ref_y) <= TOL["bf16"]


@pytest.mark.parametrize("d", [(64, 64), (128, 128), (96, 72)])
@pytest.mark.parametrize("mask", ["none", "causal", "padding", "causal_padding"])
@pytest.mark.parametrize("nsplit", [2, 3, 64])
def test_forced_split_all_masks(d, mask, nsplit):
    """A split fixed by the caller on ragged sizes: ranges past a valid length
    or past the causal diagonal are empty summaries; padded query rows stay
    exactly zero."""
    d_h, d_vh = d
    B, h, n = 3, 2, 333 if "causal" in mask else 300
    n_k = n if "causal" in mask else 1000
    self_attention = "causal" in mask
    Q, K, V = draw(B, h, n, n_k, d_h, d_vh, 100 * nsplit + d_h + len(mask))
    lens = [n_k, 1, 129] if "padding" in mask else None
    c = 1 / math.sqrt(d_h)
    Z = mha.attention_split(Q.cuda(), K.cuda(), V.cuda(), c, mask, lens,
                            self_attention=self_attention, nsplit=nsplit)
    torch.cuda.synchronize()
    got = f64(Z)
    ref = oracle_z(Q, K, V, c, mask, lens, self_attention)
    assert np.isfinite(got).all()
    if lens is not None and self_attention:
        for b, L in enumerate(lens):
            assert np.all(got[b, L:] == 0.0), "padded query rows must be exactly zero"
    assert rel_err(got, ref) <= TOL["bf16"]


@pytest.mark.parametrize("d", [(128, 128), (64, 128), (96, 72)])
@pytest.mark.parametrize("shape", [(128, 1000, "none", False), (1, 777, "padding", False),
                                   (64, 3000, "padding", False), (120, 120, "causal", True),
                                   (100, 100, "causal_padding", True)],
                         ids=lambda s: "%dx%d_%s" % s[:3])
@pytest.mark.parametrize("nsplit", [0, 2, 5])
def test_single_tile_split(d, shape, nsplit):
    """At most 128 query rows with the keys split: every unit holds a single
    query tile (the second tile of each pair has no rows), for both attention
    kernels' head sizes and the masks of self- and cross-attention."""
    d_h, d_vh = d
    n_q, n_k, mask, self_attention = shape
    B, h = 2, 3
    Q, K, V = draw(B, h, n_q, n_k, d_h, d_vh, 7 * nsplit + d_h + n_q)
    lens = [n_k, max(1, n_k // 3)] if "padding" in mask else None
    c = 1 / math.sqrt(d_h)
    Z = mha.attention_split(Q.cuda(), K.cuda(), V.cuda(), c, mask, lens,
                            self_attention=self_attention, nsplit=nsplit)
    torch.cuda.synchronize()
    got = f64(Z)
    ref = oracle_z(Q, K, V, c, mask, lens, self_attention)
    assert np.isfinite(got).all()
    if lens is not None and self_attention:
        for b, L in enumerate(lens):
            assert np.all(got[b, L:] == 0.0), "padded query rows must be exactly zero"
    assert rel_err(got, ref) <= TOL["bf16"]


def test_workload_one_shape_split_in_two():
    """The B=4, T=1024, h=12, d=64 workload's attention step with its keys cut
    in two ranges: every element against the oracle."""
    w = workloads.WORKLOADS[1]
    Q, K, V = draw(w.B, w.h, w.n_q, w.n_k, w.d_h, w.d_vh, 21)
    Z = mha.attention_split(Q.cuda(), K.cuda(), V.cuda(), w.c, "none", None, nsplit=2)
    torch.cuda.synchronize()
    ref = oracle_attention_heads(Q, K, V, w.c, "none", None, True)
    assert rel_err(f64(Z), ref) <= TOL["bf16"]


def test_split_calls_in_a_row_are_identical_and_ignore_stale_scratch():
    """The merge adds the ranges in range order whichever thread block
    finishes last, so the result is the same bits call after call; the
    scratch's contents on entry (here NaN bytes, then the last call's) do not
    matter."""
    B, h, n_q, n_k = 2, 4, 200, 5000
    Q, K, V = draw(B, h, n_q, n_k, 64, 64, 5)
    Q, K, V = Q.cuda(), K.cuda(), V.cuda()
    nbytes = mha.attention_split_workspace_size(B, n_q, n_k, h, 64, 64, 7)
    ws = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device="cuda")
    Z1 = mha.attention_split(Q, K, V, 0.125, "none", None, False, nsplit=7, workspace=ws)
    Z2 = mha.attention_split(Q, K, V, 0.125, "none", None, False, nsplit=7, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(Z1, Z2)
    ref = oracle_z(Q.cpu(), K.cpu(), V.cpu(), 0.125, "none", None, False)
    assert rel_err(f64(Z1), ref) <= TOL["bf16"]


def test_automatic_split_matches_the_forced_one():
    w = workloads.LONG_KEYS[1]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    grid, rec = mha.attention_plan(w.B, w.n_q, 8192, w.h, w.d_h, w.d_vh, "none", None, False,
                                   sms, nsplit=0)
    nsplit = len(rec) // (w.B * w.h)
    assert nsplit > 1
    Q, K, V = draw(w.B, w.h, w.n_q, 8192, w.d_h, w.d_vh, 9)
    Q, K, V = Q.cuda(), K.cuda(), V.cuda()
    Za = mha.attention_split(Q, K, V, w.c, "none", None, False, nsplit=0)
    Zf = mha.attention_split(Q, K, V, w.c, "none", None, False, nsplit=nsplit)
    Zn = mha.attention(Q, K, V, w.c, "none", None, self_attention=False)
    torch.cuda.synchronize()
    assert torch.equal(Za, Zf)
    ref = oracle_z(Q.cpu(), K.cpu(), V.cpu(), w.c, "none", None, False)
    assert rel_err(f64(Za), ref) <= TOL["bf16"]
    assert rel_err(f64(Zn), ref) <= TOL["bf16"]
