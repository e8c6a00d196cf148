"""Seeded synthetic inputs for the multi-head attention forward pass.

This module only draws random inputs; it holds none of the layer's arithmetic.
The CUDA path, the oracle, the tests and the benchmark all take their inputs
from here, so both sides of every comparison see the same values.

Recipe (one torch CPU generator per call, seeded; draw order fixed):
  X_q ~ N(0, 1) of shape (B, n_q, d_model); for cross-attention then
  X_kv ~ N(0, 1) of shape (B, n_k, d_model); then W_Q, W_K (d_model, h*d_h),
  W_V (d_model, h*d_vh), W_O (h*d_vh, d_o), each N(0, 1/d_model); then, for
  the padding masks, one valid length per batch item, uniform on the integers
  [ceil(n_k/2), n_k]. Values are drawn in float32 and then rounded to the
  compute type (bf16 rounds to nearest even), so the oracle receives exactly
  the rounded values the GPU sees.
"""

import math
from dataclasses import dataclass, replace

import torch

MASKS = ("none", "causal", "padding", "causal_padding")
DTYPES = ("f32", "bf16")


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    n_q: int
    n_k: int
    d_model: int
    h: int
    d_h: int
    d_vh: int
    d_o: int
    mask: str
    dtype: str
    cross: bool
    c: float
    seed: int

    def with_(self, **kw):
        return replace(self, **kw)


def _w(name, B, T, d_model, h, d, mask, dtype, c, seed):
    return Workload(name=name, B=B, n_q=T, n_k=T, d_model=d_model, h=h, d_h=d,
                    d_vh=d, d_o=d_model, mask=mask, dtype=dtype, cross=False,
                    c=c, seed=seed)


# The five workloads of the benchmark and the parity suite; seed = index.
WORKLOADS = [
    _w("self_f32_B1_T128_d256_h4_dh64_none", 1, 128, 256, 4, 64, "none", "f32", 1 / 8, 0),
    _w("self_bf16_B4_T1024_d768_h12_dh64_none", 4, 1024, 768, 12, 64, "none", "bf16", 1 / 8, 1),
    _w("self_bf16_B8_T2048_d1024_h16_dh64_causal", 8, 2048, 1024, 16, 64, "causal", "bf16", 1 / 8, 2),
    _w("self_bf16_B2_T8192_d2048_h16_dh128_causal_padding", 2, 8192, 2048, 16, 128,
       "causal_padding", "bf16", 1 / math.sqrt(128), 3),
    Workload(name="cross_bf16_B16_nq512_nk4096_d1024_h8_dh128_none", B=16, n_q=512,
             n_k=4096, d_model=1024, h=8, d_h=128, d_vh=128, d_o=1024, mask="none",
             dtype="bf16", cross=True, c=1 / math.sqrt(128), seed=4),
]


# A general head size (d_h = 96, neither 64 nor 128): the attention step runs
# in the 128-wide tensor-core kernel with the columns past 96 read as zeros.
# Measured beside the five above (not a benchmark headline); seed 6.
GENERAL_DIMS = _w("self_bf16_B4_T1024_d768_h8_dh96_none", 4, 1024, 768, 8, 96, "none", "bf16",
                  1 / math.sqrt(96), 6)


# A small head (d_h = 32): bf16 heads of 32..64 run in the 64-wide
# tensor-core kernel, the columns past d_h read as zeros; seed 9.
SMALL_DIMS = _w("self_bf16_B4_T1024_d768_h24_dh32_none", 4, 1024, 768, 24, 32, "none", "bf16",
                1 / math.sqrt(32), 9)


# A head size off the tensor cores (d_h = 24): the attention step runs in the
# CUDA-core kernel. Measured beside the others against the fp32 FMA peak;
# seed 10.
SIMT_DIMS = _w("self_bf16_B4_T1024_d768_h32_dh24_none", 4, 1024, 768, 32, 24, "none", "bf16",
               1 / math.sqrt(24), 10)


# Few query rows against many keys (the cross-attention workload's heads with
# n_q of 64 or 128 and n_k = 32768, 16 (batch item, head) pairs): 16 query
# tile pairs would fill 16 of the SMs, so the attention step splits the keys
# over thread blocks and merges the summaries. Seeds 7 and 8.
LONG_KEYS = [
    Workload(name="cross_bf16_B2_nq%d_nk32768_d1024_h8_dh128_none" % n_q, B=2, n_q=n_q,
             n_k=32768, d_model=1024, h=8, d_h=128, d_vh=128, d_o=1024, mask="none",
             dtype="bf16", cross=True, c=1 / math.sqrt(128), seed=seed)
    for n_q, seed in ((128, 7), (64, 8))
]


def torch_dtype(dtype):
    return {"f32": torch.float32, "bf16": torch.bfloat16}[dtype]


def make_inputs(w, lengths=None):
    """Draw the inputs of workload `w` on the CPU.

    Returns a dict of CPU tensors in the compute dtype: X_q, X_kv (None for
    self-attention), W_Q, W_K, W_V, W_O, and valid_len (int32, or None when the
    mask has no padding). `lengths` overrides the drawn valid lengths.
    """
    g = torch.Generator().manual_seed(int(w.seed))
    std = 1.0 / math.sqrt(w.d_model)
    X_q = torch.randn((w.B, w.n_q, w.d_model), generator=g)
    X_kv = torch.randn((w.B, w.n_k, w.d_model), generator=g) if w.cross else None
    W_Q = torch.randn((w.d_model, w.h * w.d_h), generator=g) * std
    W_K = torch.randn((w.d_model, w.h * w.d_h), generator=g) * std
    W_V = torch.randn((w.d_model, w.h * w.d_vh), generator=g) * std
    W_O = torch.randn((w.h * w.d_vh, w.d_o), generator=g) * std
    valid_len = None
    if w.mask in ("padding", "causal_padding"):
        lo = max(1, (w.n_k + 1) // 2)
        valid_len = torch.randint(lo, w.n_k + 1, (w.B,), generator=g).to(torch.int32)
        if lengths is not None:
            valid_len = torch.as_tensor(lengths, dtype=torch.int32).clone()
    dt = torch_dtype(w.dtype)
    out = {
        "X_q": X_q.to(dt),
        "X_kv": None if X_kv is None else X_kv.to(dt),
        "W_Q": W_Q.to(dt),
        "W_K": W_K.to(dt),
        "W_V": W_V.to(dt),
        "W_O": W_O.to(dt),
        "valid_len": valid_len,
    }
    return out



@dataclass(frozen=True)
class DecodeWorkload:
    """New query rows over a key/value cache (head-split tensors)."""
    name: str
    B: int
    h: int
    n_q: int
    n_k: int
    d_h: int
    d_vh: int
    dtype: str
    c: float
    seed: int
    causal_tail: bool = False


# The decode workload of the benchmark: one new row per sequence over a cache
# of capacity 8192, the sizes of the cross-attention workload's heads.
DECODE = DecodeWorkload(name="decode_bf16_B16_h8_dh128_nq1_cache8192", B=16, h=8, n_q=1,
                        n_k=8192, d_h=128, d_vh=128, dtype="bf16", c=1 / math.sqrt(128),
                        seed=5)


def make_decode_inputs(w, lengths=None):
    """Draw Q (B, h, n_q, d_h), K (B, h, n_k, d_h), V (B, h, n_k, d_vh), each
    N(0, 1), then one cache length per batch item, uniform on the integers
    [ceil(n_k/2), n_k] (at least n_q with causal_tail); in this order, from one
    torch CPU generator seeded with w.seed, rounded to the compute type."""
    g = torch.Generator().manual_seed(int(w.seed))
    Q = torch.randn((w.B, w.h, w.n_q, w.d_h), generator=g)
    K = torch.randn((w.B, w.h, w.n_k, w.d_h), generator=g)
    V = torch.randn((w.B, w.h, w.n_k, w.d_vh), generator=g)
    lo = max(1, (w.n_k + 1) // 2, w.n_q if w.causal_tail else 1)
    cache_len = torch.randint(lo, w.n_k + 1, (w.B,), generator=g).to(torch.int32)
    if lengths is not None:
        cache_len = torch.as_tensor(lengths, dtype=torch.int32).clone()
    dt = torch_dtype(w.dtype)
    return {"Q": Q.to(dt), "K": K.to(dt), "V": V.to(dt),
            "cache_len": [int(x) for x in cache_len]}
