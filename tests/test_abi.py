"""The C ABI on the CPU: the library loads, exports every symbol the header
declares, and rejects bad arguments on the host before touching CUDA."""

import ctypes
import math
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mha.h")


@pytest.fixture(scope="module")
def lib():
    from head_scaled_dot_gb300 import mha
    if not os.path.exists(mha.LIB_PATH):
        from head_scaled_dot_gb300 import build
        build.build()
    return mha.load()


def declared_functions():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"MHA_API\s+[\w\s\*]+?\b(mha_\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["mha_forward", "mha_workspace_size", "mha_status_string", "mha_get_device_error",
              "mha_qkv_projection", "mha_attention", "mha_output_projection"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from head_scaled_dot_gb300 import mha
    names = declared_functions()
    assert set(names) == set(mha.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    from head_scaled_dot_gb300 import mha
    for code in range(7):
        s = mha.status_string(code)
        assert s and s != "unknown status"
    assert mha.status_string(99) == "unknown status"


def test_workspace_size_is_linear_in_sequence_lengths(lib):
    from head_scaled_dot_gb300 import mha
    ws = lambda nq, nk: mha.workspace_size(2, nq, nk, 256, 4, 64, 64, 256, "bf16")
    base = ws(1024, 1024)
    # doubling both lengths at most doubles the bytes (plus alignment): no n_q*n_k term
    assert ws(2048, 2048) <= 2 * base + 4096
    assert ws(8192, 8192) <= 8 * base + 4 * 8192
    # Q, K, V, Z after the 256-byte header, then the automatic split's scratch
    # (bounded whatever the lengths: at most 160 query tile pairs' summaries)
    split = mha.attention_split_workspace_size(2, 1024, 1024, 4, 64, 64, 0)
    assert 0 < split <= 160 * 2 * 66 * 128 * 4 + 256
    exact = 256 + 2 * 4 * (1024 * 64 * 3 + 1024 * 64) * 2
    assert exact + split <= base <= exact + split + 4 * 1024
    assert mha.workspace_size(2, 1024, 1024, 256, 4, 64, 64, 256, "f32") <= 2 * exact + 4096
    assert mha.workspace_size(0, 1, 1, 1, 1, 1, 1, 1, "bf16") == 0


def _fwd(lib, **kw):
    """mha_forward with plausible non-null fake pointers: every call here must be
    rejected by the host checks, which run before any CUDA call."""
    from head_scaled_dot_gb300 import mha
    a = dict(X_q=4096, X_kv=None, W_Q=8192, W_K=12288, W_V=16384, W_O=20480, Y=24576,
             B=2, n_q=64, n_k=64, d_model=128, h=2, d_h=64, d_vh=64, d_o=128, c=0.125,
             mask=0, valid_len=None, dt=1, ws=1 << 20, ws_bytes=1 << 30, stream=None)
    a.update(kw)
    P = ctypes.c_void_p
    return lib.mha_forward(P(a["X_q"]), P(a["X_kv"]), P(a["W_Q"]), P(a["W_K"]), P(a["W_V"]),
                           P(a["W_O"]), P(a["Y"]), a["B"], a["n_q"], a["n_k"], a["d_model"],
                           a["h"], a["d_h"], a["d_vh"], a["d_o"], a["c"], a["mask"],
                           a["valid_len"], a["dt"], P(a["ws"]), a["ws_bytes"], a["stream"])


def _lens(*v):
    arr = (ctypes.c_int32 * len(v))(*v)
    return ctypes.cast(arr, ctypes.c_void_p), arr


@pytest.mark.parametrize("kw,code", [
    (dict(X_q=None), 1), (dict(W_O=None), 1), (dict(Y=None), 1),
    (dict(B=0), 1), (dict(n_q=-1), 1), (dict(h=0), 1), (dict(d_o=0), 1),
    (dict(c=math.nan), 1), (dict(c=math.inf), 1), (dict(mask=7), 1), (dict(dt=5), 1),
    (dict(n_k=65), 1),                       # self-attention needs n_k == n_q
    (dict(X_kv=28672, n_k=65, mask=1), 1),   # causal needs n_q == n_k
    (dict(mask=2), 1),                       # padding without valid lengths
    (dict(d_h=300), 2), (dict(d_vh=257), 2), (dict(d_model=100), 2), (dict(d_o=12), 2),
    (dict(d_h=33), 2),                       # bf16: h*d_h must be a multiple of 8
    (dict(d_h=300, dt=0), 2),
    (dict(X_q=4097), 2),                     # bf16 pointers must be 16-byte aligned
    (dict(ws=None), 4), (dict(ws=(1 << 20) + 16), 4), (dict(ws_bytes=1000), 4),
])
def test_forward_rejects_bad_arguments_on_host(lib, kw, code):
    assert _fwd(lib, **kw) == code


def test_empty_allowed_rows_are_rejected(lib):
    for v in [(0, 64), (64, 65), (-3, 10)]:
        lens, keep = _lens(*v)
        assert _fwd(lib, mask=2, valid_len=lens) == 3
        assert _fwd(lib, mask=3, valid_len=lens) == 3
    lens, keep = _lens(*([1] * 1025))
    assert _fwd(lib, mask=2, valid_len=lens, B=1025) == 2


def test_steps_reject_bad_arguments_on_host(lib):
    P = ctypes.c_void_p
    # attention: causal with n_q != n_k, non-finite c, padding without lengths
    assert lib.mha_attention(P(16), P(32), P(48), P(64), 1, 8, 9, 1, 64, 64, 0.1, 1, None, 0,
                             1, None, None) == 1
    assert lib.mha_attention(P(16), P(32), P(48), P(64), 1, 8, 8, 1, 64, 64, math.nan, 0,
                             None, 1, 1, None, None) == 1
    assert lib.mha_attention(P(16), P(32), P(48), P(64), 1, 8, 8, 1, 64, 64, 0.1, 2, None, 1,
                             1, None, None) == 1
    assert lib.mha_output_projection(None, P(16), P(32), 1, 8, 1, 64, 64, None, 1, None,
                                     None) == 1
    assert lib.mha_output_projection(P(16), P(32), P(48), 1, 8, 1, 64, 12, None, 1, None,
                                     None) == 2
    assert lib.mha_qkv_projection(P(16), None, P(32), P(48), P(64), P(80), P(96), P(112), 1, 8,
                                  9, 64, 1, 64, 64, 0, None, 1, None, None) == 1
    # padding without lengths; a length outside [1, n_k] / [1, n_q]
    assert lib.mha_qkv_projection(P(16), None, P(32), P(48), P(64), P(80), P(96), P(112), 1, 8,
                                  8, 64, 1, 64, 64, 2, None, 1, None, None) == 1
    lens, keep = _lens(9)
    assert lib.mha_qkv_projection(P(16), None, P(32), P(48), P(64), P(80), P(96), P(112), 1, 8,
                                  8, 64, 1, 64, 64, 2, lens, 1, None, None) == 3
    assert lib.mha_output_projection(P(16), P(32), P(48), 1, 8, 1, 64, 64, lens, 1, None,
                                     None) == 3
    assert lib.mha_get_device_error(None, None) == 1
    assert lib.mha_selftest_wait_timeout(None, 1000, None) == 1


def test_split_attention_rejects_bad_arguments_on_host(lib):
    P = ctypes.c_void_p

    def split(nsplit, ws=1 << 20, ws_bytes=1 << 30, dt=1, d=64, n_k=4096, c=0.1, mask=0):
        return lib.mha_attention_split(P(16), P(32), P(48), P(64), 1, 128, n_k, 2, d, d, c,
                                       mask, None, 0, nsplit, dt, P(ws) if ws else None,
                                       ws_bytes, None, None)
    assert split(-1) == 1 and split(257) == 1                 # INVALID_ARG
    assert split(4, dt=0) == 2 and split(4, d=24) == 2        # fp32 / off the tensor cores
    assert split(4, ws=None) == 4                              # WORKSPACE: missing,
    assert split(4, ws=(1 << 20) + 16) == 4                    # misaligned,
    assert split(4, ws_bytes=1000) == 4                        # too small
    assert split(4, c=math.nan) == 1                           # the step's own checks
    assert split(4, mask=2) == 1                               # padding without lengths


def _gen(lib, **kw):
    """mha_forward_general with fake pointers; every call here must be rejected
    by the host checks."""
    a = dict(X_q=4096, X_k=28672, X_v=32768, W_Q=8192, W_K=12288, W_V=16384, W_O=20480,
             Y=24576, B=2, n_q=64, n_k=80, d_q=128, d_k=96, d_v=40, h=2, d_h=64, d_vh=64,
             d_o=128, c=0.125, mask=0, valid_len=None, self_attention=0, gate=None, dt=1,
             ws=1 << 20, ws_bytes=1 << 30, stream=None)
    a.update(kw)
    P = ctypes.c_void_p
    return lib.mha_forward_general(
        P(a["X_q"]), P(a["X_k"]), P(a["X_v"]), P(a["W_Q"]), P(a["W_K"]), P(a["W_V"]),
        P(a["W_O"]), P(a["Y"]), a["B"], a["n_q"], a["n_k"], a["d_q"], a["d_k"], a["d_v"], a["h"],
        a["d_h"], a["d_vh"], a["d_o"], a["c"], a["mask"], a["valid_len"], a["self_attention"],
        a["gate"], a["dt"], P(a["ws"]), a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(X_k=None), 1), (dict(X_v=None), 1), (dict(W_V=None), 1),
    (dict(d_q=0), 1), (dict(d_k=-2), 1), (dict(d_v=0), 1),
    (dict(self_attention=1), 1),             # self-attention needs n_q == n_k
    (dict(mask=1), 1),                       # causal needs n_q == n_k
    (dict(d_v=36), 2),                       # bf16 input widths: multiples of 8
    (dict(d_k=100), 2),
    (dict(d_h=260), 2),
    (dict(X_v=32776), 2),                    # bf16 pointers must be 16-byte aligned
    (dict(ws_bytes=10), 4),
])
def test_general_forward_rejects_bad_arguments_on_host(lib, kw, code):
    assert _gen(lib, **kw) == code


def test_head_gates_must_be_finite_and_few_enough(lib):
    bad = (ctypes.c_float * 2)(1.0, math.nan)
    assert _gen(lib, gate=ctypes.cast(bad, ctypes.c_void_p)) == 1
    many = (ctypes.c_float * 1025)(*([1.0] * 1025))
    assert _gen(lib, gate=ctypes.cast(many, ctypes.c_void_p), h=1025, d_h=8, d_vh=8) == 2


def _dec(lib, **kw):
    """mha_attention_decode with fake pointers; every call here must be
    rejected by the host checks."""
    a = dict(Q=4096, K=8192, V=12288, Z=16384, B=2, n_q=3, n_k=100, h=2, d_h=64, d_vh=64,
             c=0.125, lens=None, tail=0, dt=1, ws=1 << 20, ws_bytes=1 << 30, stream=None)
    a.update(kw)
    P = ctypes.c_void_p
    return lib.mha_attention_decode(P(a["Q"]), P(a["K"]), P(a["V"]), P(a["Z"]), a["B"],
                                    a["n_q"], a["n_k"], a["h"], a["d_h"], a["d_vh"], a["c"],
                                    a["lens"], a["tail"], a["dt"], P(a["ws"]), a["ws_bytes"],
                                    a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(Q=None), 1), (dict(Z=None), 1), (dict(n_q=0), 1), (dict(d_vh=-1), 1),
    (dict(c=math.inf), 1), (dict(dt=3), 1),
    (dict(d_h=264), 2), (dict(n_k=70000), 2), (dict(d_h=36), 2), (dict(K=8200), 2),
    (dict(ws=None), 4), (dict(ws=(1 << 20) + 8), 4), (dict(ws_bytes=64), 4),
    (dict(n_k=2, tail=1), 3),                # tail rows need n_q <= cache length
])
def test_decode_rejects_bad_arguments_on_host(lib, kw, code):
    assert _dec(lib, **kw) == code


def test_decode_rejects_cache_lengths_outside_the_cache(lib):
    for v, tail in [((0, 50), 0), ((101, 50), 0), ((2, 50), 1)]:
        lens, keep = _lens(*v)
        assert _dec(lib, lens=lens, tail=tail) == 3


def test_decode_rejects_batches_beyond_the_length_table(lib):
    """With or without cache lengths, a batch larger than the kernels' table
    of per-item lengths is refused on the host, before any launch."""
    big = 1024 + 1  # MHA_MAX_PADDED_BATCH + 1
    assert _dec(lib, B=big) == 2
    lens = (ctypes.c_int32 * big)(*([50] * big))
    assert _dec(lib, B=big, lens=ctypes.cast(lens, ctypes.c_void_p)) == 2


def test_decode_workspace_size(lib):
    from head_scaled_dot_gb300 import mha
    assert mha.decode_workspace_size(0, 1, 1, 1, 1) == 0
    a = mha.decode_workspace_size(2, 1, 1000, 4, 64)
    assert a == mha.decode_workspace_size(2, 1, 1024, 4, 64) > 0
    assert mha.decode_workspace_size(2, 3, 1000, 4, 64) == 3 * a
