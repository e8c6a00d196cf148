"""The tensor-core attention schedule, checked on the host (no GPU): the
plan mha_attention would launch (mha_attention_plan) must hand every query
tile of every (batch item, head) to exactly one CTA, whatever the sizes,
masks and SM count. A tile handed out twice would be written twice (a race);
a tile never handed out would leave rows of Z unwritten."""

import numpy as np
import pytest

from head_scaled_dot_gb300 import mha

BLK = 128


def check_plan(B, n_q, n_k, h, d, mask, lens, self_attention, sms):
    grid, rec = mha.attention_plan(B, n_q, n_k, h, d[0], d[1], mask, lens, self_attention, sms)
    n_tiles = -(-n_q // BLK)
    pairs = B * h * (-(-n_q // (2 * BLK)))
    assert rec.shape[1] == 5 and len(rec) >= pairs
    cta, b, head, q0, nt = rec.T
    # CTA by CTA, every CTA of the grid used, none past it
    assert np.all(np.diff(cta) >= 0)
    assert cta.min() == 0 and cta.max() == grid - 1
    assert len(np.unique(cta)) == grid
    # each existing query tile of each (b, head) exactly once
    assert np.all((q0 % BLK) == 0) and np.all((nt == 1) | (nt == 2))
    cover = np.zeros((B, h, n_tiles), dtype=np.int64)
    for k in range(2):
        t = q0 // BLK + k
        sel = (nt > k) & (t < n_tiles)
        np.add.at(cover, (b[sel], head[sel], t[sel]), 1)
    assert np.all(cover == 1)
    # pairs start on even tiles; single tiles come in the two halves of a pair
    assert np.all((q0[nt == 2] // BLK) % 2 == 0)
    singles = rec[nt == 1]
    if len(singles):
        assert mask == "none"  # only equal units are split
        r = pairs % sms
        assert len(singles) == 2 * r and pairs > sms and 2 * r <= sms
    # grid: one CTA per unit, or one persistent CTA per SM
    units = len(rec)
    if units <= sms:
        assert grid == units
    else:
        assert grid in (sms, units)
    if grid == sms and units > sms:
        per = np.bincount(cta, minlength=grid)
        assert per.max() - per.min() <= 1
    return grid, rec


def test_workload_one_plan_on_152_sms():
    # 4 x 12 heads x 4 tile pairs = 192 pairs on 152 SMs: the 40 pairs of the
    # partly filled second round run as 80 single tiles
    grid, rec = check_plan(4, 1024, 1024, 12, (64, 64), "none", None, True, 152)
    assert grid == 152
    assert (rec[:, 4] == 2).sum() == 152 and (rec[:, 4] == 1).sum() == 80


def test_causal_plan_puts_heavy_pairs_first():
    grid, rec = check_plan(8, 2048, 2048, 16, (64, 64), "causal", None, True, 152)
    assert grid == 152
    first = rec[np.r_[True, np.diff(rec[:, 0]) != 0]]  # each CTA's first unit
    assert first[:, 3].min() >= 2048 - 4 * 2 * BLK   # from the last four pairs of a head


SIZES = [1, 100, 128, 129, 255, 256, 257, 600, 640, 1000, 2048]


@pytest.mark.parametrize("mask", ["none", "causal", "padding", "causal_padding"])
@pytest.mark.parametrize("sms", [1, 5, 148, 152])
def test_every_tile_exactly_once(mask, sms):
    rng = np.random.default_rng(7 + sms)
    for trial in range(40):
        B = int(rng.choice([1, 2, 3, 8, 33]))
        h = int(rng.choice([1, 3, 8, 16]))
        n = int(rng.choice(SIZES))
        self_attention = bool(rng.integers(2)) or "causal" in mask
        n_q = n
        n_k = n if self_attention else int(rng.choice(SIZES))
        d = [(64, 64), (128, 128), (64, 128), (128, 64), (96, 72)][trial % 5]
        lens = [int(x) for x in rng.integers(1, n_k + 1, B)] if "padding" in mask else None
        check_plan(B, n_q, n_k, h, d, mask, lens, self_attention, sms)


def test_many_units_run_one_cta_each():
    # more units than the host simulates (65536): one CTA per unit
    grid, rec = check_plan(1024, 1024, 1024, 32, (64, 64), "causal_padding",
                           [1 + (37 * b) % 1024 for b in range(1024)], True, 152)
    assert grid == len(rec) == 1024 * 32 * 4


def test_plan_rejects_what_attention_rejects():
    def status(*a, **k):
        try:
            mha.attention_plan(*a, **k)
        except mha.MHAError as e:
            return e.status
        return 0
    assert status(2, 256, 256, 4, 64, 64, num_sms=0) == 1            # INVALID_ARG
    assert status(2, 256, 128, 4, 64, 64, "causal", self_attention=False) == 1
    assert status(2, 256, 256, 4, 96, 64) == 0                        # 96 runs as 128
    assert status(2, 256, 256, 4, 48, 64) == 2                        # UNSUPPORTED head sizes
    assert status(2, 256, 256, 4, 64, 100) == 2
    assert status(2, 256, 256, 4, 136, 64) == 2
    assert status(2, 256, 256, 4, 64, 64, "padding", [0, 10]) == 3    # EMPTY_ROW
    assert status(2, 256, 256, 4, 64, 64, "padding", [10, 257]) == 3
    assert status(1025, 8, 8, 1, 64, 64, "padding", [1] * 1025) == 2  # beyond the length table
