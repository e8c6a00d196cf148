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


def _oracle_head(args):
    """One (batch item, head) of the oracle's dense attention, for a worker
    process: (b, i, Q, K, V, c, mask, L, self_attention) -> (b, i, H)."""
    b, i, Q, K, V, c, mask, L, self_attention = args
    n_q, n_k = Q.shape[0], K.shape[0]
    rows = oracle.query_rows_computed(mask, n_q, L, self_attention)
    allowed = oracle.allowed_keys(mask, n_q, n_k, L)
    H, _ = oracle.attention(Q, K, V, c, allowed, rows)
    return b, i, H


def oracle_attention_heads(Q, K, V, c, mask, lens, self_attention, workers=None):
    """Z (B, n_q, h*d_vh) in float64 from head-split Q, K, V (torch tensors of
    any dtype, on any device): the oracle's dense attention of every
    (batch item, head), heads concatenated in order.

    The heads run in a pool of spawned worker processes (the elementwise
    steps of the oracle use one core each); spawn, not fork, because the
    calling process may already hold a CUDA context."""
    import multiprocessing as mp
    import os

    B, h, n_q, _ = Q.shape
    d_vh = V.shape[3]
    mk = oracle.MASK_NAMES[mask]
    Qc, Kc, Vc = Q.cpu(), K.cpu(), V.cpu()
    jobs = [(b, i, Qc[b, i].double().numpy(), Kc[b, i].double().numpy(),
             Vc[b, i].double().numpy(), float(c), mk,
             None if lens is None else int(lens[b]), bool(self_attention))
            for b in range(B) for i in range(h)]
    Z = np.zeros((B, n_q, h * d_vh))
    n = workers or max(1, min(16, os.cpu_count() or 1, len(jobs)))
    keys = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")
    saved = {k: os.environ.get(k) for k in keys}
    for k in keys:
        os.environ[k] = "1"  # the workers' BLAS: one thread each
    try:
        with mp.get_context("spawn").Pool(n) as pool:
            for b, i, H in pool.imap_unordered(_oracle_head, jobs):
                Z[b, :, i * d_vh:(i + 1) * d_vh] = H
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    return Z
