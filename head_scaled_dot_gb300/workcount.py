"""Work counts of one multi-head attention forward pass (floating-point
operations), as the benchmark reports them. Counting only: no kernel or oracle
arithmetic lives here."""


def flops(w, valid_len=None):
    """Work counts of one forward pass, in floating-point operations.

    attention core: 4 * n_q * n_k * d_h per (batch item, head), halved under a
    causal mask; projections: 2 * rows * d_in * width per GEMM. With
    `valid_len` (padding masks) the effective count uses the valid rows: for
    each batch item L_b query rows (self-attention), L_b keys, and L_b^2 / 2
    pairs under causal. Returns a dict with 'attention', 'qkv', 'out', 'total'.
    """
    B, h, d_h, d_vh = w.B, w.h, w.d_h, w.d_vh
    causal = w.mask in ("causal", "causal_padding")
    padded = w.mask in ("padding", "causal_padding") and valid_len is not None
    attn = qkv = out = 0.0
    for b in range(B):
        if padded:
            L = int(valid_len[b])
            nq = L if not w.cross else w.n_q
            nk = L
        else:
            nq, nk = w.n_q, w.n_k
        pairs = nq * nk / 2.0 if causal else float(nq) * nk
        attn += 2.0 * h * pairs * (d_h + d_vh)
        nq_rows = nq if not w.cross else w.n_q
        nk_rows = nk if not w.cross else w.n_k
        qkv += 2.0 * nq_rows * w.d_model * h * d_h
        qkv += 2.0 * nk_rows * w.d_model * h * (d_h + d_vh)
        out += 2.0 * nq_rows * h * d_vh * w.d_o
    return {"attention": attn, "qkv": qkv, "out": out, "total": attn + qkv + out}
