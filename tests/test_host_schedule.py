"""The tensor-core attention schedule, checked on the host (no GPU): the
plan mha_attention would launch (mha_attention_plan) must hand every query
tile of every (batch item, head) to exactly one CTA, whatever the sizes,
masks and SM count, and with a split over the keys every (query tile, key
block) to exactly one unit. A tile handed out twice would be written twice
(a race); a tile never handed out would leave rows of Z unwritten; a key
block in two ranges would be counted twice in the merged summary."""

import numpy as np
import pytest

from head_scaled_dot_gb300 import mha

BLK = 128


def check_plan(B, n_q, n_k, h, d, mask, lens, self_attention, sms, nsplit=1):
    grid, rec = mha.attention_plan(B, n_q, n_k, h, d[0], d[1], mask, lens, self_attention, sms,
                                   nsplit=nsplit)
    n_tiles = -(-n_q // BLK)
    n_blocks = -(-n_k // BLK)
    pairs = B * h * (-(-n_q // (2 * BLK)))
    assert rec.shape[1] == 7 and len(rec) >= pairs
    cta, b, head, q0, nt, k0, k1 = rec.T
    # CTA by CTA, every CTA of the grid used, none past it
    assert np.all(np.diff(cta) >= 0)
    assert cta.min() == 0 and cta.max() == grid - 1
    assert len(np.unique(cta)) == grid
    # key ranges: whole 128-key blocks (the last one ends at n_k)
    assert np.all(k0 % BLK == 0) and np.all(k0 < k1) and np.all(k1 <= n_k)
    assert np.all((k1 % BLK == 0) | (k1 == n_k))
    # each (existing query tile, key block) of each (b, head) exactly once
    assert np.all((q0 % BLK) == 0) and np.all((nt == 1) | (nt == 2))
    cover = np.zeros((B, h, n_tiles, n_blocks), dtype=np.int64)
    for u in range(len(rec)):
        for k in range(nt[u]):
            t = q0[u] // BLK + k
            if t < n_tiles:
                cover[b[u], head[u], t, k0[u] // BLK:-(-k1[u] // BLK)] += 1
    assert np.all(cover == 1)
    if nsplit == 1:
        assert np.all(k0 == 0) and np.all(k1 == n_k)
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


def test_few_long_tiles_split_over_the_keys():
    # 16 heads of one 128-row query tile against 32768 keys: 16 tile pairs
    # would leave 136 of 152 SMs idle; the keys are cut into nine ranges
    grid, rec = check_plan(2, 128, 32768, 8, (128, 128), "none", None, False, 152, nsplit=0)
    assert len(rec) == grid == 16 * 9
    spans = rec[:, 6] - rec[:, 5]
    assert spans.max() == 29 * BLK and spans.sum() == 16 * 32768
    # the schedule mha_attention uses (no scratch) does not split
    grid1, rec1 = check_plan(2, 128, 32768, 8, (128, 128), "none", None, False, 152, nsplit=1)
    assert len(rec1) == grid1 == 16


@pytest.mark.parametrize("cfg", [
    (4, 1024, 1024, 12, (64, 64), "none", None, True),
    (8, 2048, 2048, 16, (64, 64), "causal", None, True),
    (2, 8192, 8192, 16, (128, 128), "causal_padding", [4290, 7796], True),
    (16, 512, 4096, 8, (128, 128), "none", None, False)])
def test_full_workloads_are_not_split(cfg):
    # enough tile pairs to fill the GPU: the automatic choice keeps every
    # (query tile, head) on one thread block
    grid, rec = check_plan(*cfg, 152, nsplit=0)
    assert np.all(rec[:, 5] == 0) and np.all(rec[:, 6] == cfg[2])


@pytest.mark.parametrize("mask", ["none", "causal", "padding", "causal_padding"])
@pytest.mark.parametrize("nsplit", [0, 2, 3, 7, 64])
def test_split_covers_every_key_block_once(mask, nsplit):
    rng = np.random.default_rng(11 + nsplit)
    for trial in range(12):
        B = int(rng.choice([1, 2, 3]))
        h = int(rng.choice([1, 3, 8]))
        n = int(rng.choice(SIZES))
        self_attention = bool(rng.integers(2)) or "causal" in mask
        n_q = n
        n_k = n if self_attention else int(rng.choice(SIZES + [4000, 9000]))
        d = [(64, 64), (128, 128), (96, 72)][trial % 3]
        lens = [int(x) for x in rng.integers(1, n_k + 1, B)] if "padding" in mask else None
        grid, rec = check_plan(B, n_q, n_k, h, d, mask, lens, self_attention, 152, nsplit)
        n_blocks = -(-n_k // BLK)
        if nsplit > 1:
            # as many equal ranges of whole blocks as asked for (fewer when
            # the blocks do not divide)
            per = -(-n_blocks // min(nsplit, n_blocks))
            want = -(-n_blocks // per)
            pairs = B * h * (-(-n_q // (2 * BLK)))
            assert len(rec) == pairs * (want if want > 1 else 1)


def test_split_workspace_sizes():
    # counters (one int per query tile, rounded to 256 bytes), then one slot of
    # (64 or 128 + 2) x 128 floats per (tile, key range)
    assert mha.attention_split_workspace_size(2, 128, 32768, 8, 128, 128, 1) == 0
    assert mha.attention_split_workspace_size(2, 128, 32768, 8, 128, 128, 9) == \
        256 + 16 * 2 * 9 * 130 * 128 * 4
    # 8 key blocks asked to make 5 ranges: ranges of 2 blocks, so 4 of them
    assert mha.attention_split_workspace_size(1, 300, 1000, 2, 64, 64, 5) == \
        256 + 4 * 2 * 4 * 66 * 128 * 4
    # more ranges than key blocks: one range per block
    assert mha.attention_split_workspace_size(1, 128, 300, 1, 64, 64, 50) == \
        256 + 1 * 2 * 3 * 66 * 128 * 4
    # the automatic choice: the most it may take, none for full workloads
    assert mha.attention_split_workspace_size(2, 128, 32768, 8, 128, 128, 0) == \
        256 + 16 * 2 * 10 * 130 * 128 * 4
    assert mha.attention_split_workspace_size(8, 2048, 2048, 16, 64, 64, 0) == 0
    # head sizes off the tensor cores never split
    assert mha.attention_split_workspace_size(1, 128, 4096, 1, 24, 24, 4) == 0
    # mha_forward's workspace includes the automatic split's scratch
    base = mha.workspace_size(2, 128, 32768, 1024, 8, 128, 128, 1024, "f32")
    assert mha.workspace_size(2, 128, 32768, 1024, 8, 128, 128, 1024, "bf16") >= \
        base // 2 + mha.attention_split_workspace_size(2, 128, 32768, 8, 128, 128, 0)


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
    assert status(2, 256, 256, 4, 48, 64) == 0                        # 48 runs as 64
    assert status(2, 256, 256, 4, 24, 64) == 2                        # UNSUPPORTED head sizes
    assert status(2, 256, 256, 4, 64, 100) == 2
    assert status(2, 256, 256, 4, 136, 64) == 2
    assert status(2, 256, 256, 4, 64, 64, "padding", [0, 10]) == 3    # EMPTY_ROW
    assert status(2, 256, 256, 4, 64, 64, "padding", [10, 257]) == 3
    assert status(1025, 8, 8, 1, 64, 64, "padding", [1] * 1025) == 2  # beyond the length table
    assert status(2, 256, 256, 4, 64, 64, nsplit=-1) == 1
    assert status(2, 256, 256, 4, 64, 64, nsplit=257) == 1
