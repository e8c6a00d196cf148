"""Pins for the oracle: each test ties it to something other than itself.

The pins are the worked example printed on the pages, closed forms, the
invariants the pages state, special cases that reduce to a library routine
(scipy's softmax, torch's CPU multi-head attention in float64) and brute force
on tiny inputs. A plausible slip in the oracle (a dropped scale, a transposed
weight, a wrong head order, an off-by-one mask, a softmax over the wrong axis)
fails at least one of them.
"""

import itertools
import json
import math
import os
import random

import numpy as np
import pytest
import scipy.special
import torch

import oracle as O


def rng(seed):
    return np.random.default_rng(seed)


def rand_layer(seed, B=2, n_q=7, n_k=7, d_model=12, h=3, d_h=4, d_vh=4, d_o=12,
               cross=False):
    r = rng(seed)
    X_q = r.standard_normal((B, n_q, d_model))
    X_kv = r.standard_normal((B, n_k, d_model)) if cross else None
    s = 1 / math.sqrt(d_model)
    W_Q = r.standard_normal((d_model, h * d_h)) * s
    W_K = r.standard_normal((d_model, h * d_h)) * s
    W_V = r.standard_normal((d_model, h * d_vh)) * s
    W_O = r.standard_normal((h * d_vh, d_o)) * s
    return X_q, X_kv, W_Q, W_K, W_V, W_O


# ---------------------------------------------------------------------------
# The worked example ("Self-Attention & Multi-Head", two tokens by hand)
# ---------------------------------------------------------------------------

def test_worked_example_matches_printed_values(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "worked_example_two_tokens.json")))
    q = np.array([g["q1"]])
    K = np.array(g["keys"])
    V = np.array(g["values"])
    c = 1 / math.sqrt(g["d_k"])
    S = O.scores(q, K, 1.0)
    np.testing.assert_array_equal(S[0], g["raw_scores"])
    Sc = O.scores(q, K, c)

    def close(val, printed):
        tol = 0.5 * 10.0 ** (-printed["printed_decimals"]) + 1e-12
        np.testing.assert_allclose(val, printed["values"], rtol=0, atol=tol)

    close(Sc[0], g["scaled_scores"])
    close(np.exp(Sc[0]), g["exp_scaled_scores"])
    assert abs(np.exp(Sc[0]).sum() - g["exp_sum"]["value"]) <= 0.005 + 1e-12
    H, A = O.attention(q, K, V, c, np.ones((1, 2), dtype=bool))
    close(A[0], g["weights"])
    close(H[0], g["output"])
    # closed form: weights = (sigma(sqrt 2), 1 - sigma(sqrt 2)) exactly
    w1 = 1.0 / (1.0 + math.exp(-math.sqrt(2.0)))
    np.testing.assert_allclose(A[0], [w1, 1 - w1], rtol=0, atol=1e-15)
    np.testing.assert_allclose(H[0], [w1, 1 - w1], rtol=0, atol=1e-15)


# ---------------------------------------------------------------------------
# Block summary and merge ("Stable summary of an attention key block")
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(6))
def test_merge_over_any_partition_and_order_equals_softmax(seed):
    r = rng(seed)
    n, d, v = 23, 5, 3
    Q = r.standard_normal((n, d))
    K = r.standard_normal((n, d)) * 3.0  # wide score range: the max matters
    V = r.standard_normal((n, v))
    c = 0.7
    S = O.scores(Q, K, c)
    allowed = r.random((n, n)) < 0.6
    allowed[np.arange(n), r.integers(0, n, n)] = True  # every row nonempty
    for i in range(n):
        keys = list(range(n))
        random.Random(seed * 100 + i).shuffle(keys)
        cuts = sorted(r.choice(np.arange(1, n), size=r.integers(0, 6), replace=False))
        blocks = [np.array(b) for b in np.split(np.array(keys), cuts)]
        got = O.attention_row_by_blocks(S[i], V, allowed[i], blocks)
        A_i = np.flatnonzero(allowed[i])
        ref = scipy.special.softmax(S[i, A_i]) @ V[A_i]
        np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)


def test_merge_identity_and_symmetry():
    r = rng(7)
    s = r.standard_normal(9) * 4
    V = r.standard_normal((9, 2))
    a = O.block_summary(s, V, [0, 3, 5])
    b = O.block_summary(s, V, [1, 2, 8])
    assert O.merge(O.BOTTOM, a) is a and O.merge(a, O.BOTTOM) is a
    assert O.block_summary(s, V, []) is O.BOTTOM
    ab, ba = O.merge(a, b), O.merge(b, a)
    assert ab[0] == ba[0]
    np.testing.assert_allclose(ab[1], ba[1], rtol=1e-15)
    np.testing.assert_allclose(ab[2], ba[2], rtol=1e-15)
    # the merged summary is the summary of the union (same m, l, z)
    u = O.block_summary(s, V, [0, 1, 2, 3, 5, 8])
    assert ab[0] == u[0]
    np.testing.assert_allclose(ab[1], u[1], rtol=1e-14)
    np.testing.assert_allclose(ab[2], u[2], rtol=1e-14)
    # m is the exact max; l >= 1 since the max term contributes e^0
    assert a[0] == s[[0, 3, 5]].max() and a[1] >= 1.0
    with pytest.raises(O.EmptyAllowedRow):
        O.summary_output(O.BOTTOM)


# ---------------------------------------------------------------------------
# Library pins: scipy softmax and torch's float64 CPU multi-head attention
# ---------------------------------------------------------------------------

def test_single_head_unmasked_is_scipy_softmax_times_v():
    r = rng(11)
    Q, K, V = r.standard_normal((6, 4)), r.standard_normal((9, 4)), r.standard_normal((9, 3))
    c = 0.37
    H, A = O.attention(Q, K, V, c, np.ones((6, 9), dtype=bool))
    ref = scipy.special.softmax(c * Q @ K.T, axis=1)
    np.testing.assert_allclose(A, ref, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(H, ref @ V, rtol=1e-13, atol=1e-15)


def _torch_mha(X_q, X_kv, W_Q, W_K, W_V, W_O, h, d_h, c, mask, valid_len):
    """torch's own multi-head attention (x W^T convention, scale 1/sqrt(d_h)),
    fed with our row-major weights transposed and W_Q pre-scaled so that its
    fixed scale becomes c."""
    Xq = torch.from_numpy(X_q).transpose(0, 1)  # (n_q, B, d)
    Xkv = Xq if X_kv is None else torch.from_numpy(X_kv).transpose(0, 1)
    n_q, n_k, d_model = Xq.shape[0], Xkv.shape[0], Xq.shape[2]
    WQ = torch.from_numpy(W_Q * (c * math.sqrt(d_h))).T.contiguous()
    attn_mask = None
    if mask in (O.MASK_CAUSAL, O.MASK_CAUSAL_PADDING):
        attn_mask = torch.ones(n_q, n_k, dtype=torch.bool).triu(1)
    kpm = None
    if mask in (O.MASK_PADDING, O.MASK_CAUSAL_PADDING):
        kpm = torch.arange(n_k)[None, :] >= torch.as_tensor(valid_len)[:, None]
    out, _ = torch.nn.functional.multi_head_attention_forward(
        Xq, Xkv, Xkv, d_model, h, None, None, None, None, False, 0.0,
        torch.from_numpy(W_O).T.contiguous(), None, training=False,
        key_padding_mask=kpm, need_weights=False, attn_mask=attn_mask,
        use_separate_proj_weight=True, q_proj_weight=WQ,
        k_proj_weight=torch.from_numpy(W_K).T.contiguous(),
        v_proj_weight=torch.from_numpy(W_V).T.contiguous())
    return out.transpose(0, 1).numpy()


@pytest.mark.parametrize("mask", [O.MASK_NONE, O.MASK_CAUSAL, O.MASK_PADDING,
                                  O.MASK_CAUSAL_PADDING])
@pytest.mark.parametrize("cross", [False, True])
def test_matches_torch_multi_head_attention(mask, cross):
    h, d_h = 3, 5
    d_model = h * d_h
    B, n = 3, 9
    X_q, X_kv, W_Q, W_K, W_V, W_O = rand_layer(
        5 + mask + 10 * cross, B=B, n_q=n, n_k=n, d_model=d_model, h=h, d_h=d_h,
        d_vh=d_h, d_o=d_model, cross=cross)
    c = 0.61
    valid_len = [9, 4, 1] if mask in (O.MASK_PADDING, O.MASK_CAUSAL_PADDING) else None
    Y = O.mha_forward(X_q, X_kv, W_Q, W_K, W_V, W_O, h, d_h, d_h, c, mask, valid_len)
    ref = _torch_mha(X_q, X_kv, W_Q, W_K, W_V, W_O, h, d_h, c, mask, valid_len)
    for b in range(B):
        rows = np.ones(n, dtype=bool)
        if valid_len is not None and not cross:
            rows[valid_len[b]:] = False
            # padded query rows are not computed and are exactly zero
            assert np.all(Y[b, ~rows] == 0.0)
        np.testing.assert_allclose(Y[b, rows], ref[b, rows], rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------------------
# Statements of the pages
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("mask", [O.MASK_NONE, O.MASK_CAUSAL, O.MASK_PADDING])
def test_separate_and_combined_projections_agree(mask):
    h, d_h, d_vh = 3, 4, 5
    X_q, X_kv, W_Q, W_K, W_V, W_O = rand_layer(21, h=h, d_h=d_h, d_vh=d_vh, d_o=6)
    valid_len = [5, 7] if mask == O.MASK_PADDING else None
    Y = O.mha_forward(X_q, None, W_Q, W_K, W_V, W_O, h, d_h, d_vh, 0.5, mask, valid_len)
    sep = O.mha_forward_separate(
        X_q, None,
        [W_Q[:, i * d_h:(i + 1) * d_h] for i in range(h)],
        [W_K[:, i * d_h:(i + 1) * d_h] for i in range(h)],
        [W_V[:, i * d_vh:(i + 1) * d_vh] for i in range(h)],
        W_O, 0.5, mask, valid_len)
    np.testing.assert_allclose(Y, sep, rtol=1e-13, atol=1e-14)


def test_head_permutation_with_inverse_w_o_blocks_preserves_output():
    h, d_h, d_vh = 4, 3, 2
    X_q, _, W_Q, W_K, W_V, W_O = rand_layer(31, h=h, d_h=d_h, d_vh=d_vh, d_o=5)
    perm = [2, 0, 3, 1]

    def cols(W, d):
        return np.concatenate([W[:, p * d:(p + 1) * d] for p in perm], axis=1)

    W_O_p = np.concatenate([W_O[p * d_vh:(p + 1) * d_vh] for p in perm], axis=0)
    Y = O.mha_forward(X_q, None, W_Q, W_K, W_V, W_O, h, d_h, d_vh, 0.8, O.MASK_CAUSAL)
    Yp = O.mha_forward(X_q, None, cols(W_Q, d_h), cols(W_K, d_h), cols(W_V, d_vh),
                       W_O_p, h, d_h, d_vh, 0.8, O.MASK_CAUSAL)
    np.testing.assert_allclose(Y, Yp, rtol=1e-13, atol=1e-14)
    # without permuting W_O the output changes: the head order matters
    Yw = O.mha_forward(X_q, None, cols(W_Q, d_h), cols(W_K, d_h), cols(W_V, d_vh),
                       W_O, h, d_h, d_vh, 0.8, O.MASK_CAUSAL)
    assert np.abs(Yw - Y).max() > 1e-3


def test_zero_output_projection_gives_zero():
    X_q, _, W_Q, W_K, W_V, W_O = rand_layer(41)
    Y = O.mha_forward(X_q, None, W_Q, W_K, W_V, np.zeros_like(W_O), 3, 4, 4, 0.5)
    assert np.all(Y == 0.0)


def test_zero_scale_gives_mean_of_allowed_values():
    r = rng(51)
    Q, K, V = r.standard_normal((6, 3)), r.standard_normal((6, 3)), r.standard_normal((6, 2))
    H, _ = O.attention(Q, K, V, 0.0, O.allowed_keys(O.MASK_NONE, 6, 6))
    np.testing.assert_allclose(H, np.tile(V.mean(axis=0), (6, 1)), rtol=1e-14)
    H, _ = O.attention(Q, K, V, 0.0, O.allowed_keys(O.MASK_CAUSAL, 6, 6))
    prefix = np.cumsum(V, axis=0) / np.arange(1, 7)[:, None]
    np.testing.assert_allclose(H, prefix, rtol=1e-14)
    H, _ = O.attention(Q, K, V, 0.0, O.allowed_keys(O.MASK_PADDING, 6, 6, 4))
    np.testing.assert_allclose(H, np.tile(V[:4].mean(axis=0), (6, 1)), rtol=1e-14)


def test_causal_first_row_is_first_value_exactly():
    r = rng(52)
    Q, K, V = r.standard_normal((5, 3)), r.standard_normal((5, 3)), r.standard_normal((5, 4))
    H, A = O.attention(Q, K, V, 1.3, O.allowed_keys(O.MASK_CAUSAL, 5, 5))
    assert np.array_equal(H[0], V[0]) and A[0, 0] == 1.0


def test_constant_values_and_shifted_keys():
    r = rng(53)
    Q, K = r.standard_normal((5, 3)), r.standard_normal((7, 3))
    vrow = r.standard_normal(4)
    V = np.tile(vrow, (7, 1))
    H, _ = O.attention(Q, K, V, 0.9, O.allowed_keys(O.MASK_NONE, 5, 7))
    np.testing.assert_allclose(H, np.tile(vrow, (5, 1)), rtol=1e-14)
    # adding one vector u to every key adds c q_i.u to a whole row of scores
    V = r.standard_normal((7, 4))
    u = r.standard_normal(3) * 5
    H1, A1 = O.attention(Q, K, V, 0.9, O.allowed_keys(O.MASK_NONE, 5, 7))
    H2, A2 = O.attention(Q, K + u, V, 0.9, O.allowed_keys(O.MASK_NONE, 5, 7))
    np.testing.assert_allclose(A1, A2, rtol=1e-12)
    np.testing.assert_allclose(H1, H2, rtol=1e-12)


@pytest.mark.parametrize("mask,L", [(O.MASK_CAUSAL, None), (O.MASK_PADDING, 3),
                                    (O.MASK_CAUSAL_PADDING, 4)])
def test_forbidden_weights_exact_zero_and_rows_sum_to_one(mask, L):
    r = rng(54)
    n = 8
    Q, K, V = r.standard_normal((n, 3)), r.standard_normal((n, 3)), r.standard_normal((n, 2))
    allowed = O.allowed_keys(mask, n, n, L)
    _, A = O.attention(Q, K, V, 2.0, allowed)
    assert np.all(A[~allowed] == 0.0)
    assert np.all(A[allowed] > 0.0)
    np.testing.assert_allclose(A.sum(axis=1), 1.0, rtol=0, atol=1e-14)
    i, j = np.indices((n, n))
    if mask in (O.MASK_CAUSAL, O.MASK_CAUSAL_PADDING):
        assert not np.any(allowed & (j > i))
        assert np.all(allowed[j <= np.minimum(i, (L or n) - 1)])
    if L is not None:
        assert not np.any(allowed[:, L:])


def test_projection_ablations_w_v_and_w_o_leave_weights_unchanged():
    r = rng(55)
    X = r.standard_normal((6, 4))
    WQ, WK = r.standard_normal((4, 3)), r.standard_normal((4, 3))
    allowed = O.allowed_keys(O.MASK_NONE, 6, 6)
    _, A1 = O.attention(X @ WQ, X @ WK, X @ r.standard_normal((4, 2)), 0.5, allowed)
    _, A2 = O.attention(X @ WQ, X @ WK, X @ r.standard_normal((4, 2)), 0.5, allowed)
    np.testing.assert_array_equal(A1, A2)
    _, A3 = O.attention(X @ r.standard_normal((4, 3)), X @ WK, X, 0.5, allowed)
    assert np.abs(A3 - A1).max() > 1e-3


def test_empty_allowed_row_is_rejected():
    X_q, _, W_Q, W_K, W_V, W_O = rand_layer(61)
    with pytest.raises(O.EmptyAllowedRow):
        O.mha_forward(X_q, None, W_Q, W_K, W_V, W_O, 3, 4, 4, 0.5, O.MASK_PADDING, [0, 3])
    with pytest.raises(O.EmptyAllowedRow):
        O.mha_forward(X_q, None, W_Q, W_K, W_V, W_O, 3, 4, 4, 0.5, O.MASK_PADDING, [3, 8])
    allowed = np.ones((3, 3), dtype=bool)
    allowed[1] = False
    with pytest.raises(O.EmptyAllowedRow):
        O.attention_weights(np.zeros((3, 3)), allowed)


def test_batch_items_are_independent():
    X_q, X_kv, W_Q, W_K, W_V, W_O = rand_layer(71, B=3, cross=True)
    Y = O.mha_forward(X_q, X_kv, W_Q, W_K, W_V, W_O, 3, 4, 4, 0.5)
    X_q2, X_kv2 = X_q.copy(), X_kv.copy()
    X_q2[1] += 3.0
    X_kv2[1] *= -2.0
    Y2 = O.mha_forward(X_q2, X_kv2, W_Q, W_K, W_V, W_O, 3, 4, 4, 0.5)
    np.testing.assert_array_equal(Y[[0, 2]], Y2[[0, 2]])
    assert np.abs(Y[1] - Y2[1]).max() > 1e-3


def test_parameter_count_is_four_d_squared_when_widths_match():
    for d, h in [(768, 12), (1024, 16), (2048, 16)]:
        assert O.parameter_count(d, h, d // h, d // h) == 4 * d * d


def test_sampled_rows_match_full_forward():
    X_q, X_kv, W_Q, W_K, W_V, W_O = rand_layer(81, B=2, n_q=9, n_k=9)
    L = [9, 5]
    Y, inter = O.mha_forward(X_q, None, W_Q, W_K, W_V, W_O, 3, 4, 4, 0.4,
                             O.MASK_CAUSAL_PADDING, L, return_intermediates=True)
    for b in range(2):
        rows = [0, 3, 4, 8]
        Yr, Zr = O.mha_rows(X_q, None, W_Q, W_K, W_V, W_O, 3, 4, 4, 0.4,
                            O.MASK_CAUSAL_PADDING, L, b, rows)
        np.testing.assert_allclose(Yr, Y[b, rows], rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(Zr, inter["Z"][b, rows], rtol=1e-13, atol=1e-15)


# ---------------------------------------------------------------------------
# Brute force with scalar loops on tiny shapes
# ---------------------------------------------------------------------------

def _brute(X_q, X_kv, W_Q, W_K, W_V, W_O, h, d_h, d_vh, c, allowed_fn):
    X_kv = X_q if X_kv is None else X_kv
    B, n_q, dm = X_q.shape
    n_k = X_kv.shape[1]
    d_o = W_O.shape[1]
    Y = np.zeros((B, n_q, d_o))
    for b in range(B):
        for i in range(n_q):
            z = []
            for hd in range(h):
                q = [math.fsum(X_q[b, i, t] * W_Q[t, hd * d_h + r] for t in range(dm))
                     for r in range(d_h)]
                keys = [j for j in range(n_k) if allowed_fn(b, i, j)]
                s = {}
                for j in keys:
                    k = [math.fsum(X_kv[b, j, t] * W_K[t, hd * d_h + r] for t in range(dm))
                         for r in range(d_h)]
                    s[j] = c * math.fsum(q[r] * k[r] for r in range(d_h))
                m = max(s.values())
                e = {j: math.exp(s[j] - m) for j in keys}
                tot = math.fsum(e.values())
                for r in range(d_vh):
                    vr = {j: math.fsum(X_kv[b, j, t] * W_V[t, hd * d_vh + r] for t in range(dm))
                          for j in keys}
                    z.append(math.fsum(e[j] * vr[j] for j in keys) / tot)
            for o in range(d_o):
                Y[b, i, o] = math.fsum(z[f] * W_O[f, o] for f in range(len(z)))
    return Y


@pytest.mark.parametrize("case", list(itertools.product(["none", "causal", "cross"], [0, 1])))
def test_brute_force_tiny(case):
    kind, seed = case
    h, d_h, d_vh = 2, 3, 2
    cross = kind == "cross"
    X_q, X_kv, W_Q, W_K, W_V, W_O = rand_layer(
        90 + seed, B=2, n_q=3, n_k=4 if cross else 3, d_model=3, h=h, d_h=d_h,
        d_vh=d_vh, d_o=3, cross=cross)
    mask = O.MASK_CAUSAL if kind == "causal" else O.MASK_NONE
    Y = O.mha_forward(X_q, X_kv, W_Q, W_K, W_V, W_O, h, d_h, d_vh, 0.75, mask)
    ref = _brute(X_q, X_kv, W_Q, W_K, W_V, W_O, h, d_h, d_vh, 0.75,
                 (lambda b, i, j: j <= i) if kind == "causal" else (lambda b, i, j: True))
    np.testing.assert_allclose(Y, ref, rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------------------
# The general form: separate query, key and value inputs of their own widths
# ("Multi-head attention and self-attention", Definition: Q in R^{n_q x d_q},
# K in R^{n_k x d_k}, V in R^{n_k x d_v})
# ---------------------------------------------------------------------------

def rand_general(seed, B, n_q, n_k, d_q, d_k, d_v, h, d_h, d_vh, d_o):
    r = rng(seed)
    X_q = r.standard_normal((B, n_q, d_q))
    X_k = r.standard_normal((B, n_k, d_k))
    X_v = r.standard_normal((B, n_k, d_v))
    W_Q = r.standard_normal((d_q, h * d_h)) / math.sqrt(d_q)
    W_K = r.standard_normal((d_k, h * d_h)) / math.sqrt(d_k)
    W_V = r.standard_normal((d_v, h * d_vh)) / math.sqrt(d_v)
    W_O = r.standard_normal((h * d_vh, d_o)) / math.sqrt(h * d_vh)
    return X_q, X_k, X_v, W_Q, W_K, W_V, W_O


def _brute_general(X_q, X_k, X_v, W_Q, W_K, W_V, W_O, h, d_h, d_vh, c, allowed_fn):
    B, n_q, d_q = X_q.shape
    n_k, d_k, d_v = X_k.shape[1], X_k.shape[2], X_v.shape[2]
    d_o = W_O.shape[1]
    Y = np.zeros((B, n_q, d_o))
    for b in range(B):
        for i in range(n_q):
            z = []
            for hd in range(h):
                q = [math.fsum(X_q[b, i, t] * W_Q[t, hd * d_h + r] for t in range(d_q))
                     for r in range(d_h)]
                keys = [j for j in range(n_k) if allowed_fn(b, i, j)]
                s = {}
                for j in keys:
                    k = [math.fsum(X_k[b, j, t] * W_K[t, hd * d_h + r] for t in range(d_k))
                         for r in range(d_h)]
                    s[j] = c * math.fsum(q[r] * k[r] for r in range(d_h))
                m = max(s.values())
                e = {j: math.exp(s[j] - m) for j in keys}
                tot = math.fsum(e.values())
                for r in range(d_vh):
                    vr = {j: math.fsum(X_v[b, j, t] * W_V[t, hd * d_vh + r] for t in range(d_v))
                          for j in keys}
                    z.append(math.fsum(e[j] * vr[j] for j in keys) / tot)
            for o in range(d_o):
                Y[b, i, o] = math.fsum(z[f] * W_O[f, o] for f in range(len(z)))
    return Y


@pytest.mark.parametrize("kind", ["none", "causal", "padding"])
def test_general_form_brute_force_tiny(kind):
    h, d_h, d_vh = 2, 3, 2
    n_q, n_k = (3, 3) if kind == "causal" else (3, 4)
    X_q, X_k, X_v, W_Q, W_K, W_V, W_O = rand_general(
        140 + len(kind), B=2, n_q=n_q, n_k=n_k, d_q=3, d_k=4, d_v=2, h=h, d_h=d_h, d_vh=d_vh,
        d_o=3)
    mask = {"none": O.MASK_NONE, "causal": O.MASK_CAUSAL, "padding": O.MASK_PADDING}[kind]
    valid_len = [2, 4] if kind == "padding" else None
    Y = O.mha_forward_general(X_q, X_k, X_v, W_Q, W_K, W_V, W_O, h, d_h, d_vh, 0.8, mask,
                              valid_len)
    if kind == "causal":
        fn = lambda b, i, j: j <= i
    elif kind == "padding":
        fn = lambda b, i, j: j < valid_len[b]
    else:
        fn = lambda b, i, j: True
    ref = _brute_general(X_q, X_k, X_v, W_Q, W_K, W_V, W_O, h, d_h, d_vh, 0.8, fn)
    np.testing.assert_allclose(Y, ref, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("mask", [O.MASK_NONE, O.MASK_CAUSAL, O.MASK_PADDING])
def test_general_form_matches_torch_with_separate_key_and_value_inputs(mask):
    """torch's multi-head attention takes key and value tensors of their own
    widths (kdim, vdim); its query width, head sizes and output width are tied
    to embed_dim = h d_h, so those are chosen that way here."""
    h, d_h = 3, 4
    E = h * d_h
    B, n = 2, 6
    d_k, d_v = 7, 5
    X_q, X_k, X_v, W_Q, W_K, W_V, W_O = rand_general(
        150 + mask, B=B, n_q=n, n_k=n, d_q=E, d_k=d_k, d_v=d_v, h=h, d_h=d_h, d_vh=d_h, d_o=E)
    c = 0.47
    valid_len = [6, 2] if mask == O.MASK_PADDING else None
    Y = O.mha_forward_general(X_q, X_k, X_v, W_Q, W_K, W_V, W_O, h, d_h, d_h, c, mask,
                              valid_len)
    Xq = torch.from_numpy(X_q).transpose(0, 1)
    Xk = torch.from_numpy(X_k).transpose(0, 1)
    Xv = torch.from_numpy(X_v).transpose(0, 1)
    attn_mask = torch.ones(n, n, dtype=torch.bool).triu(1) if mask == O.MASK_CAUSAL else None
    kpm = None
    if mask == O.MASK_PADDING:
        kpm = torch.arange(n)[None, :] >= torch.as_tensor(valid_len)[:, None]
    out, _ = torch.nn.functional.multi_head_attention_forward(
        Xq, Xk, Xv, E, h, None, None, None, None, False, 0.0,
        torch.from_numpy(W_O).T.contiguous(), None, training=False, key_padding_mask=kpm,
        need_weights=False, attn_mask=attn_mask, use_separate_proj_weight=True,
        q_proj_weight=torch.from_numpy(W_Q * (c * math.sqrt(d_h))).T.contiguous(),
        k_proj_weight=torch.from_numpy(W_K).T.contiguous(),
        v_proj_weight=torch.from_numpy(W_V).T.contiguous())
    np.testing.assert_allclose(Y, out.transpose(0, 1).numpy(), rtol=1e-12, atol=1e-13)


def test_general_form_key_and_value_inputs_are_not_interchangeable():
    """With d_k == d_v, swapping the key and value inputs must change the output
    (the keys decide the weights, the values what is averaged)."""
    X_q, X_k, X_v, W_Q, W_K, W_V, W_O = rand_general(
        160, B=1, n_q=4, n_k=5, d_q=6, d_k=6, d_v=6, h=2, d_h=3, d_vh=3, d_o=4)
    Y1 = O.mha_forward_general(X_q, X_k, X_v, W_Q, W_K, W_V, W_O, 2, 3, 3, 0.9)
    Y2 = O.mha_forward_general(X_q, X_v, X_k, W_Q, W_K, W_V, W_O, 2, 3, 3, 0.9)
    assert np.abs(Y1 - Y2).max() > 1e-3


def test_one_key_value_input_is_the_shared_case():
    """mha_forward with X_kv equals the general form with X_k = X_v = X_kv."""
    X_q, X_kv, W_Q, W_K, W_V, W_O = rand_layer(170, cross=True, n_k=9)
    Y = O.mha_forward(X_q, X_kv, W_Q, W_K, W_V, W_O, 3, 4, 4, 0.5)
    G = O.mha_forward_general(X_q, X_kv, X_kv, W_Q, W_K, W_V, W_O, 3, 4, 4, 0.5)
    np.testing.assert_array_equal(Y, G)


# ---------------------------------------------------------------------------
# Head zeroing at a named location ("Multi-Head Attention review", "Head
# Identity and Ablation" and "Audit Order"): the gate scales head i's block of
# the concatenation, before W_O
# ---------------------------------------------------------------------------

def test_zeroing_a_head_gate_equals_zeroing_its_w_o_row_block():
    h, d_h, d_vh = 3, 4, 5
    X_q, X_k, X_v, W_Q, W_K, W_V, W_O = rand_general(
        180, B=2, n_q=6, n_k=7, d_q=5, d_k=6, d_v=4, h=h, d_h=d_h, d_vh=d_vh, d_o=8)
    for i in range(h):
        gate = [1.0] * h
        gate[i] = 0.0
        Yg = O.mha_forward_general(X_q, X_k, X_v, W_Q, W_K, W_V, W_O, h, d_h, d_vh, 0.7,
                                   head_gate=gate)
        W_O0 = W_O.copy()
        W_O0[i * d_vh:(i + 1) * d_vh] = 0.0
        Yw = O.mha_forward_general(X_q, X_k, X_v, W_Q, W_K, W_V, W_O0, h, d_h, d_vh, 0.7)
        np.testing.assert_allclose(Yg, Yw, rtol=1e-13, atol=1e-15)


def test_head_gates_scale_each_heads_contribution_linearly():
    h, d_h, d_vh = 2, 3, 3
    X_q, X_k, X_v, W_Q, W_K, W_V, W_O = rand_general(
        181, B=1, n_q=5, n_k=5, d_q=4, d_k=4, d_v=4, h=h, d_h=d_h, d_vh=d_vh, d_o=4)
    f = lambda g: O.mha_forward_general(X_q, X_k, X_v, W_Q, W_K, W_V, W_O, h, d_h, d_vh, 0.5,
                                        O.MASK_CAUSAL, head_gate=g)
    np.testing.assert_allclose(f([1.0, 1.0]), f(None), rtol=0, atol=0)
    np.testing.assert_allclose(f([1.0, 1.0]), f([1.0, 0.0]) + f([0.0, 1.0]), rtol=1e-13,
                               atol=1e-15)
    np.testing.assert_allclose(f([2.5, -1.0]), 2.5 * f([1.0, 0.0]) - f([0.0, 1.0]),
                               rtol=1e-12, atol=1e-14)
    assert np.all(f([0.0, 0.0]) == 0.0)


# ---------------------------------------------------------------------------
# New rows over a key/value cache (autoregressive generation)
# ---------------------------------------------------------------------------

def test_decode_allowed_sets_reduce_to_the_causal_and_padding_masks():
    # the rows are the whole sequence: the tail-causal sets are the causal mask
    for n in (1, 4, 9):
        np.testing.assert_array_equal(O.decode_allowed(n, n, n, True),
                                      O.allowed_keys(O.MASK_CAUSAL, n, n))
    # the rows see the whole cache: the padding mask of the cache length
    np.testing.assert_array_equal(O.decode_allowed(3, 10, 7, False),
                                  O.allowed_keys(O.MASK_PADDING, 3, 10, 7))
    # one new row: both readings agree (it is the last position)
    np.testing.assert_array_equal(O.decode_allowed(1, 10, 7, True),
                                  O.decode_allowed(1, 10, 7, False))
    # tail rows: row i sees the first L - n_q + i + 1 keys
    a = O.decode_allowed(3, 10, 6, True)
    assert [int(r.sum()) for r in a] == [4, 5, 6]


def test_decode_rows_equal_the_last_rows_of_causal_self_attention():
    """The n_q newest rows over a cache equal the last n_q rows of causal
    self-attention over the whole sequence."""
    r = rng(190)
    B, h, n, d = 2, 3, 11, 4
    Q = r.standard_normal((B, h, n, d))
    K = r.standard_normal((B, h, n, d))
    V = r.standard_normal((B, h, n, d))
    full = np.zeros((B, n, h * d))
    for b in range(B):
        for i in range(h):
            H, _ = O.attention(Q[b, i], K[b, i], V[b, i], 0.6, O.allowed_keys(O.MASK_CAUSAL, n, n))
            full[b, :, i * d:(i + 1) * d] = H
    for n_q in (1, 3):
        Z = O.attention_decode(Q[:, :, n - n_q:], K, V, 0.6, [n, n], causal_tail=True)
        np.testing.assert_allclose(Z, full[:, n - n_q:], rtol=1e-13, atol=1e-15)
    with pytest.raises(O.EmptyAllowedRow):
        O.attention_decode(Q[:, :, :3], K, V, 0.6, [2, 5], causal_tail=True)
