"""Oracle for the multi-head attention forward pass: plain fp64 CPU code.

TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check of the package
entry module and the CPU-baseline leg of the benchmark may import this module.
The product path (the CUDA library and its Python binding) never calls it, and
this module imports nothing from the product package.

What it computes, with the page each step follows:

* "Multi-head attention and self-attention" (alphabetamath.cc,
  def-multihead-self-attention, Definition): head i is
  H_i = Attn(Q W_i^Q, K W_i^K, V W_i^V); MHA = Concat_feature(H_1..H_h) W^O.
  Self-attention is Q = K = V = X.
* "Stable summary of an attention key block" (alphabetamath.cc,
  def-attention-block-summary, Definition): scores s_ij = c * sum_r Q_ir K_jr
  over a nonempty allowed key set A_i; the summary (m, l, z) of a key set, the
  empty state (bottom) and the merge (star). z / l is the attention output.
* "Multi-Head Attention review" (llmprimer.com, sections "The Complete
  Multi-Head Operation" and "Separate and Combined Projections"): batch-major
  shapes, combined projection matrices W_Q, W_K : d_model x (h d_k),
  W_V : d_model x (h d_v) with the head blocks side by side, the head split
  (B,T,h d_k) -> (B,T,h,d_k) -> (B,h,T,d_k), concatenation in head order and
  Y = Z W_O with W_O : (h d_v, d_model).
* "From Attention to Self-Attention review" (llmprimer.com, sections "The
  Complete Layer" and "Causal and padding masks"): the mask is applied before
  the row softmax; a causal mask removes future positions, a padding mask
  removes artificial positions; no projection biases.
* "Self-Attention & Multi-Head" (ailu.in): the five steps project, score,
  scale, normalise, aggregate; softmax along each query row.

Every array is float64. Masked positions get weight exactly 0 (they are removed
from the allowed set, never given a large negative score). A query row whose
allowed set is empty is rejected with EmptyAllowedRow, following the nonempty
condition of the block-summary Definition.

Readings where the pages leave a step open (each one is also listed in the
design notes of the repository):

* the scale is a free constant c (block-summary Definition); the workloads use
  c = 1/sqrt(d_k) as in the other pages;
* causal: A_i = {j : j <= i}, defined only when n_q == n_k;
* padding with per-sequence valid length L_b: A_i = {j : j < L_b}; in
  self-attention the query rows i >= L_b are padding too, they are not
  computed and their rows of Z and Y are 0 (0 times W_O is 0, no biases);
  in cross-attention the padding applies to keys only;
* causal + padding: A_i = {j : j <= i and j < L_b};
* the empty state is the identity of the merge: bottom * S = S * bottom = S.
"""

import math

import numpy as np

MASK_NONE = 0
MASK_CAUSAL = 1
MASK_PADDING = 2
MASK_CAUSAL_PADDING = 3

MASK_NAMES = {
    "none": MASK_NONE,
    "causal": MASK_CAUSAL,
    "padding": MASK_PADDING,
    "causal_padding": MASK_CAUSAL_PADDING,
}


class EmptyAllowedRow(ValueError):
    """A query row has no allowed key (block-summary Definition: A_i must be
    nonempty)."""


# ---------------------------------------------------------------------------
# Masks: "From Attention to Self-Attention review", "Causal and padding masks"
# ---------------------------------------------------------------------------

def _has_causal(mask):
    return mask in (MASK_CAUSAL, MASK_CAUSAL_PADDING)


def _has_padding(mask):
    return mask in (MASK_PADDING, MASK_CAUSAL_PADDING)


def query_rows_computed(mask, n_q, valid_len_b, self_attention):
    """Boolean (n_q,): which query rows are real positions.

    Only self-attention with a padding mask has padded query rows (i >= L_b);
    every other case computes every row.
    """
    rows = np.ones(n_q, dtype=bool)
    if _has_padding(mask) and self_attention:
        rows[np.arange(n_q) >= valid_len_b] = False
    return rows


def allowed_keys(mask, n_q, n_k, valid_len_b=None):
    """Boolean (n_q, n_k) matrix whose row i is the allowed key set A_i.

    Causal: j <= i (needs n_q == n_k). Padding: j < L_b. Both: the
    intersection. None: every key.
    """
    allowed = np.ones((n_q, n_k), dtype=bool)
    i = np.arange(n_q)[:, None]
    j = np.arange(n_k)[None, :]
    if _has_causal(mask):
        if n_q != n_k:
            raise ValueError("a causal mask needs n_q == n_k")
        allowed &= j <= i
    if _has_padding(mask):
        if valid_len_b is None:
            raise ValueError("a padding mask needs the valid length")
        allowed &= j < valid_len_b
    return allowed


# ---------------------------------------------------------------------------
# Scaled dot-product attention, dense, one head
# ---------------------------------------------------------------------------

def scores(Q, K, c):
    """S = c Q K^T: s_ij = c * sum_r Q_ir K_jr (block-summary Definition;
    'Self-Attention & Multi-Head' steps Score and Scale)."""
    return c * (Q @ K.T)


def attention_weights(S, allowed, rows=None):
    """Row softmax of the scores over each allowed set, exact zeros elsewhere.

    For each computed row i: m = max_{j in A_i} s_ij, w_j = exp(s_ij - m) for
    j in A_i and 0 otherwise, weights = w / sum(w). Rows not in `rows` are left
    all zero. Raises EmptyAllowedRow for a computed row with an empty A_i.
    """
    n_q = S.shape[0]
    if rows is None:
        rows = np.ones(n_q, dtype=bool)
    empty = rows & ~allowed.any(axis=1)
    if empty.any():
        raise EmptyAllowedRow(
            "query row %d has no allowed key" % int(np.flatnonzero(empty)[0]))
    use = allowed & rows[:, None]
    masked = np.where(use, S, -np.inf)
    m = masked.max(axis=1, keepdims=True)
    m = np.where(np.isfinite(m), m, 0.0)
    w = np.where(use, np.exp(masked - m), 0.0)
    l = w.sum(axis=1, keepdims=True)
    l = np.where(l > 0.0, l, 1.0)
    return w / l


def attention(Q, K, V, c, allowed, rows=None):
    """One head: softmax(c Q K^T restricted to A_i) V, dense.

    Returns (H, A): the (n_q, d_v) output and the (n_q, n_k) weight matrix.
    Rows not in `rows` are 0 in both.
    """
    A = attention_weights(scores(Q, K, c), allowed, rows)
    return A @ V, A


# ---------------------------------------------------------------------------
# Stable block summary and its merge: "Stable summary of an attention key
# block", Definition
# ---------------------------------------------------------------------------

BOTTOM = None  # the summary of the empty set: no numeric coordinates


def block_summary(s_row, V, S_idx):
    """Summary (m, l, z) of the nonempty key set S_idx for one query row.

    m = max_{j in S} s_ij, l = sum_{j in S} exp(s_ij - m),
    z = sum_{j in S} exp(s_ij - m) v_j. The empty set gives BOTTOM.
    """
    S_idx = np.asarray(S_idx, dtype=np.int64)
    if S_idx.size == 0:
        return BOTTOM
    s = s_row[S_idx]
    m = s.max()
    e = np.exp(s - m)
    return (m, e.sum(), e @ V[S_idx])


def merge(sig_S, sig_T):
    """The merge of two summaries of disjoint nonempty key sets.

    m' = max(m_S, m_T), l' = e^{m_S - m'} l_S + e^{m_T - m'} l_T and
    z' = e^{m_S - m'} z_S + e^{m_T - m'} z_T. BOTTOM is the identity.
    """
    if sig_S is BOTTOM:
        return sig_T
    if sig_T is BOTTOM:
        return sig_S
    m_S, l_S, z_S = sig_S
    m_T, l_T, z_T = sig_T
    m = max(m_S, m_T)
    a = math.exp(m_S - m)
    b = math.exp(m_T - m)
    return (m, a * l_S + b * l_T, a * z_S + b * z_T)


def summary_output(sig):
    """Attention output on the summarised set: third coordinate over second."""
    if sig is BOTTOM:
        raise EmptyAllowedRow("the empty key set has no attention output")
    _, l, z = sig
    return z / l


def attention_row_by_blocks(s_row, V, allowed_row, blocks):
    """Output of one query row folded block by block with the merge.

    `blocks` is a sequence of key-index arrays (a partition of range(n_k) in
    any order). Each block is cut down to its allowed keys, summarised, and
    merged into the running summary.
    """
    allowed_row = np.asarray(allowed_row, dtype=bool)
    running = BOTTOM
    for blk in blocks:
        blk = np.asarray(blk, dtype=np.int64)
        running = merge(running, block_summary(s_row, V, blk[allowed_row[blk]]))
    return summary_output(running)


# ---------------------------------------------------------------------------
# Multi-head attention forward pass
# ---------------------------------------------------------------------------

def _f64(a):
    return np.asarray(a, dtype=np.float64)


def mha_forward_general(X_q, X_k, X_v, W_Q, W_K, W_V, W_O, h, d_h, d_vh, c,
                        mask=MASK_NONE, valid_len=None, self_attention=False,
                        head_gate=None, return_intermediates=False):
    """The general form of the 'Multi-head attention and self-attention'
    Definition: query, key and value inputs are separate matrices, each with
    its own width,
        head i = Attn(X_q W_i^Q, X_k W_i^K, X_v W_i^V),
        Y = Concat_feature(head_1 .. head_h) W^O.

    Batch-major arguments, all converted to float64:
      X_q (B, n_q, d_q); X_k (B, n_k, d_k); X_v (B, n_k, d_v);
      W_Q (d_q, h*d_h), W_K (d_k, h*d_h), W_V (d_v, h*d_vh): head i owns the
      column block [i*d, (i+1)*d) (combined projections);
      W_O (h*d_vh, d_o): row block [i*d_vh, (i+1)*d_vh) belongs to head i;
      valid_len: B integers for the padding masks, else None;
      self_attention: the query rows are positions of the same sequence, so
      rows i >= valid_len are padding queries (their output rows are 0);
      head_gate: h numbers or None. Head i's block of the concatenation is
      multiplied by head_gate[i] before W_O: the head-zeroing location of the
      'Multi-Head Attention review' ("Head Identity and Ablation", "Audit
      Order": head zeroing at an explicitly named location).

    Returns Y (B, n_q, d_o) and, when asked, a dict with the head-split
    Q, K (B, h, n, d_h), V (B, h, n_k, d_vh) and the concatenated
    Z (B, n_q, h*d_vh).
    """
    X_q, X_k, X_v = _f64(X_q), _f64(X_k), _f64(X_v)
    W_Q, W_K, W_V, W_O = _f64(W_Q), _f64(W_K), _f64(W_V), _f64(W_O)
    B, n_q, d_q = X_q.shape
    n_k, d_k = X_k.shape[1], X_k.shape[2]
    d_v = X_v.shape[2]
    d_o = W_O.shape[1]
    assert X_k.shape[0] == B and X_v.shape[:2] == (B, n_k)
    assert W_Q.shape == (d_q, h * d_h) and W_K.shape == (d_k, h * d_h)
    assert W_V.shape == (d_v, h * d_vh) and W_O.shape == (h * d_vh, d_o)
    if _has_padding(mask):
        if valid_len is None or len(valid_len) != B:
            raise ValueError("a padding mask needs one valid length per batch item")
        for L in valid_len:
            if not 1 <= int(L) <= n_k:
                raise EmptyAllowedRow("valid length %d outside [1, %d]" % (int(L), n_k))

    Qh = np.zeros((B, h, n_q, d_h))
    Kh = np.zeros((B, h, n_k, d_h))
    Vh = np.zeros((B, h, n_k, d_vh))
    Z = np.zeros((B, n_q, h * d_vh))
    for b in range(B):
        L = int(valid_len[b]) if _has_padding(mask) else None
        rows = query_rows_computed(mask, n_q, L, self_attention)
        allowed = allowed_keys(mask, n_q, n_k, L)
        # combined projections, then the head split (B,T,h d)->(B,T,h,d)->(B,h,T,d)
        Qb = (X_q[b] @ W_Q).reshape(n_q, h, d_h).transpose(1, 0, 2)
        Kb = (X_k[b] @ W_K).reshape(n_k, h, d_h).transpose(1, 0, 2)
        Vb = (X_v[b] @ W_V).reshape(n_k, h, d_vh).transpose(1, 0, 2)
        Qh[b], Kh[b], Vh[b] = Qb, Kb, Vb
        heads = []
        for i in range(h):
            H_i, _ = attention(Qb[i], Kb[i], Vb[i], c, allowed, rows)
            heads.append(H_i)
        if head_gate is not None:
            heads = [float(head_gate[i]) * heads[i] for i in range(h)]
        # concatenate along the feature axis in head order
        Z[b] = np.concatenate(heads, axis=1)
    Y = Z @ W_O
    if return_intermediates:
        return Y, {"Q": Qh, "K": Kh, "V": Vh, "Z": Z}
    return Y


def mha_forward(X_q, X_kv, W_Q, W_K, W_V, W_O, h, d_h, d_vh, c,
                mask=MASK_NONE, valid_len=None, return_intermediates=False):
    """Y = Concat_i(softmax(c (X_q W_i^Q)(X_kv W_i^K)^T + M)(X_kv W_i^V)) W_O:
    mha_forward_general with one key/value input X_kv (B, n_k, d_model), or
    X_kv None for self-attention (X_kv := X_q, padded query rows are 0)."""
    self_attention = X_kv is None
    X_kv = X_q if self_attention else X_kv
    return mha_forward_general(X_q, X_kv, X_kv, W_Q, W_K, W_V, W_O, h, d_h, d_vh, c, mask,
                               valid_len, self_attention, None, return_intermediates)


def mha_forward_separate(X_q, X_kv, W_Q_list, W_K_list, W_V_list, W_O, c,
                         mask=MASK_NONE, valid_len=None):
    """The same layer written with one matrix per head (the 'Multi-head
    attention and self-attention' Definition): H_i = Attn(X W_i^Q, X W_i^K,
    X W_i^V), Y = Concat_feature(H_1..H_h) W^O. No combined matrices and no
    reshape: used to check the combined form and its head split."""
    self_attention = X_kv is None
    X_q = _f64(X_q)
    X_kv = X_q if self_attention else _f64(X_kv)
    B, n_q, _ = X_q.shape
    n_k = X_kv.shape[1]
    out = []
    for b in range(B):
        L = int(valid_len[b]) if _has_padding(mask) else None
        rows = query_rows_computed(mask, n_q, L, self_attention)
        allowed = allowed_keys(mask, n_q, n_k, L)
        heads = []
        for WQ_i, WK_i, WV_i in zip(W_Q_list, W_K_list, W_V_list):
            H_i, _ = attention(X_q[b] @ _f64(WQ_i), X_kv[b] @ _f64(WK_i),
                               X_kv[b] @ _f64(WV_i), c, allowed, rows)
            heads.append(H_i)
        out.append(np.concatenate(heads, axis=1) @ _f64(W_O))
    return np.stack(out)


def mha_rows(X_q, X_kv, W_Q, W_K, W_V, W_O, h, d_h, d_vh, c, mask, valid_len,
             b, rows):
    """Y[b, rows, :] and Z[b, rows, :] for a few query rows of one batch item.

    The same arithmetic as mha_forward restricted to the requested rows, so a
    full-size workload can be checked on sampled outputs. Returns (Y, Z), each
    with one row per requested index; padded query rows are 0.
    """
    self_attention = X_kv is None
    Xq_b = _f64(X_q[b])
    Xkv_b = Xq_b if self_attention else _f64(X_kv[b])
    W_Q, W_K, W_V, W_O = _f64(W_Q), _f64(W_K), _f64(W_V), _f64(W_O)
    n_q = Xq_b.shape[0]
    n_k = Xkv_b.shape[0]
    rows = np.asarray(rows, dtype=np.int64)
    L = int(valid_len[b]) if _has_padding(mask) else None
    computed = query_rows_computed(mask, n_q, L, self_attention)[rows]
    allowed = allowed_keys(mask, n_q, n_k, L)[rows]
    Qr = (Xq_b[rows] @ W_Q).reshape(len(rows), h, d_h).transpose(1, 0, 2)
    Kb = (Xkv_b @ W_K).reshape(n_k, h, d_h).transpose(1, 0, 2)
    Vb = (Xkv_b @ W_V).reshape(n_k, h, d_vh).transpose(1, 0, 2)
    heads = []
    for i in range(h):
        H_i, _ = attention(Qr[i], Kb[i], Vb[i], c, allowed, computed)
        heads.append(H_i)
    Z = np.concatenate(heads, axis=1)
    return Z @ W_O, Z


def decode_allowed(n_q, n_k, cache_len, causal_tail):
    """Allowed key sets of n_q new query rows over a cache holding cache_len
    positions ('From Attention to Self-Attention review': autoregressive
    generation; a causal mask removes future positions, a padding mask the
    positions that are not part of the sequence). Without causal_tail every
    row sees keys 0 .. cache_len-1; with it the rows are the last n_q
    positions of the sequence and row i sees keys j <= cache_len - n_q + i."""
    allowed = np.zeros((n_q, n_k), dtype=bool)
    for i in range(n_q):
        last = cache_len - n_q + i if causal_tail else cache_len - 1
        allowed[i, :last + 1] = True
    return allowed


def attention_decode(Q, K, V, c, cache_len=None, causal_tail=False):
    """Z (B, n_q, h*d_vh) of head-split Q (B, h, n_q, d_h) over the cache K
    (B, h, n_k, d_h), V (B, h, n_k, d_vh): each head by the dense definition
    (attention), the heads concatenated in order."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    B, h, n_q, _ = Q.shape
    n_k, d_vh = V.shape[2], V.shape[3]
    Z = np.zeros((B, n_q, h * d_vh))
    for b in range(B):
        L = n_k if cache_len is None else int(cache_len[b])
        if not 1 <= L <= n_k or (causal_tail and L < n_q):
            raise EmptyAllowedRow("cache length %d" % L)
        allowed = decode_allowed(n_q, n_k, L, causal_tail)
        for i in range(h):
            H, _ = attention(Q[b, i], K[b, i], V[b, i], c, allowed)
            Z[b, :, i * d_vh:(i + 1) * d_vh] = H
    return Z


# ---------------------------------------------------------------------------
# Work counts (the formulas the benchmark reports)
# ---------------------------------------------------------------------------

def parameter_count(d_model, h, d_k, d_v):
    """Projection parameters without biases: 2 d_model h d_k + 2 d_model h d_v
    ('Multi-Head Attention review', 'Parameter and Work Conventions').
    The W_O term is h d_v x d_model."""
    return 2 * d_model * h * d_k + 2 * d_model * h * d_v
