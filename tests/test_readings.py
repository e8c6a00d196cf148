"""Readings of the block-summary Definition ("Stable summary of an attention
key block", alphabetamath.cc) that the CUDA kernels rely on, checked on the
CPU against the oracle.

Stale maximum. The Definition's m is the exact maximum of the summarised
scores. The kernels keep a running m that they raise only when a block's
maximum exceeds it by more than 2^8 (scores scaled by log2(e), exponentials
taken base 2). Otherwise the block's terms are taken against the older m.
The triple (m~, l~, z~) with m~ <= m equals e^{m - m~} (m, l, z) in its last
two coordinates, so z~ / l~ = z / l, and every term 2^{x - m~} stays at most
2^8. The model below is written from that reading, not from the kernel
source. It must give the oracle's output over any block order and with
masked keys, and its terms must respect the bound."""

import math

import numpy as np
import pytest

from oracle import mha_oracle as O

LOG2E = 1.0 / math.log(2.0)
TAU = 8.0  # log2 of the allowed growth before m is raised


def stale_fold(s_row, V, allowed_row, blocks, tau=TAU):
    """z / l of one row folded block by block with a stale running max.
    Returns (output, largest term seen, number of times m was raised)."""
    x = np.where(allowed_row, s_row * LOG2E, -np.inf)  # log2 units, masked
    m, l, z = -np.inf, 0.0, np.zeros(V.shape[1])
    biggest, raises = 0.0, 0
    for blk in blocks:
        xb = x[blk]
        mb = xb.max()
        if mb == -np.inf:  # all keys of the block forbidden: the empty summary
            continue
        if m == -np.inf or mb > m + tau:
            m_new = max(m, mb)
            raises += 1
        else:
            m_new = m
        alpha = 0.0 if m == -np.inf else 2.0 ** (m - m_new)
        p = np.where(np.isfinite(xb), 2.0 ** (xb - m_new), 0.0)
        biggest = max(biggest, p.max())
        l = l * alpha + p.sum()
        z = z * alpha + p @ V[blk]
        m = m_new
    return z / l, biggest, raises


def blocks_of(n, size, order):
    b = [np.arange(i, min(i + size, n)) for i in range(0, n, size)]
    return [b[i] for i in order(len(b))]


@pytest.mark.parametrize("seed", range(5))
@pytest.mark.parametrize("order", ["forward", "reverse", "shuffled"])
def test_stale_maximum_gives_the_exact_softmax(seed, order):
    r = np.random.default_rng(seed)
    n_q, n_k, d, dv = 9, 70, 6, 4
    Q = r.standard_normal((n_q, d))
    K = r.standard_normal((n_k, d)) * (1 + seed)  # from narrow to wide score ranges
    V = r.standard_normal((n_k, dv))
    c = 0.8
    allowed = r.random((n_q, n_k)) < 0.7
    allowed[:, r.integers(0, n_k)] = True
    allowed[0, 16:32] = False  # a block fully forbidden for row 0
    H, _ = O.attention(Q, K, V, c, allowed)
    S = O.scores(Q, K, c)
    pick = {"forward": lambda k: range(k), "reverse": lambda k: reversed(range(k)),
            "shuffled": lambda k: r.permutation(k)}[order]
    for i in range(n_q):
        out, biggest, _ = stale_fold(S[i], V, allowed[i], blocks_of(n_k, 16, pick))
        assert np.allclose(out, H[i], rtol=1e-12, atol=1e-12)
        assert biggest <= 2.0 ** TAU * (1 + 1e-15)


def test_rising_scores_raise_the_maximum_only_past_the_threshold():
    # block j's scores all equal 3 j (log2 units): the max rises by 3 per
    # block, so m is raised at block 0 and then whenever it lags by more than 8
    n_blk, size = 12, 8
    x = np.repeat(3.0 * np.arange(n_blk), size)
    s_row = x / LOG2E
    V = np.eye(n_blk * size)[:, :5]
    allowed = np.ones(n_blk * size, dtype=bool)
    out, biggest, raises = stale_fold(s_row, V, allowed, blocks_of(n_blk * size, size,
                                                                   lambda k: range(k)))
    w = 2.0 ** (x - x.max())
    assert np.allclose(out, (w @ V) / w.sum(), rtol=1e-12, atol=1e-15)
    # raised at blocks 0, 3 (9 > 0 + 8), 6 (18 > 9 + 8), 9 (27 > 18 + 8)
    assert raises == 4
    assert biggest <= 2.0 ** TAU


def test_exact_threshold_does_not_raise():
    # a block whose max is exactly m + 8 is taken against the old m: term 2^8
    s_row = np.array([0.0, 8.0]) / LOG2E
    V = np.array([[1.0], [2.0]])
    out, biggest, raises = stale_fold(s_row, V, np.ones(2, dtype=bool), [np.array([0]),
                                                                         np.array([1])])
    assert raises == 1 and biggest == 2.0 ** 8
    w = np.array([1.0, 256.0])
    assert np.isclose(out[0], (w @ V[:, 0]) / w.sum(), rtol=1e-15)
