"""Shared test helpers: moving seeded inputs to the GPU, calling the oracle on
exactly the values the GPU sees, and the parity metric."""

import numpy as np
import torch

import oracle

# Parity tolerances: max|Y - Y_ref| / max|Y_ref| over computed rows.
TOL = {"bf16": 1e-2, "f32": 1e-4}


def f64(t):
    return None if t is None else t.double().cpu().numpy()


def to_dev(inp, device="cuda:0"):
    return {k: (v.to(device) if torch.is_tensor(v) and k != "valid_len" else v)
            for k, v in inp.items()}


def rel_err(got, ref, rows=None):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if rows is not None:
        got, ref = got[rows], ref[rows]
    denom = np.abs(ref).max()
    return float(np.abs(got - ref).max() / denom) if denom > 0 else float(np.abs(got).max())


def lens_list(inp):
    v = inp.get("valid_len")
    return None if v is None else [int(x) for x in v]


def oracle_forward(w, inp, return_intermediates=False):
    return oracle.mha_forward(f64(inp["X_q"]), f64(inp["X_kv"]), f64(inp["W_Q"]),
                              f64(inp["W_K"]), f64(inp["W_V"]), f64(inp["W_O"]), w.h, w.d_h,
                              w.d_vh, w.c, oracle.MASK_NAMES[w.mask], lens_list(inp),
                              return_intermediates=return_intermediates)


def computed_rows(w, inp):
    """Boolean (B, n_q): rows that are real queries (padded self-attention rows
    are excluded from the error metric and must be exactly zero)."""
    rows = np.ones((w.B, w.n_q), dtype=bool)
    lens = lens_list(inp)
    if lens is not None and not w.cross:
        for b, L in enumerate(lens):
            rows[b, L:] = False
    return rows
