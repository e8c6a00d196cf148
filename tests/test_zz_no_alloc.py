"""mha_forward_no_alloc (the allocation-free entry point, for callers that
cannot allocate device memory) against mha_forward on the same inputs.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""

import ctypes

import pytest
import torch

from head_scaled_dot_gb300 import mha, workloads
from helpers import TOL, f64, rel_err, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return mha.load()


def _case(name, mask, seed, lengths=None):
    # intermediates of B=2, T=768, h=4, d=64 in bf16: about 3 MiB, well inside 32 MiB
    w = workloads.Workload(name=name, B=2, n_q=768, n_k=768, d_model=256, h=4, d_h=64,
                           d_vh=64, d_o=256, mask=mask, dtype="bf16", cross=False,
                           c=0.125, seed=seed)
    return w, workloads.make_inputs(w, lengths=lengths)


def _both(w, inp):
    t = to_dev(inp)
    args = (t["X_q"], t["X_kv"], t["W_Q"], t["W_K"], t["W_V"], t["W_O"], w.h, w.d_h, w.d_vh,
            w.c, w.mask, inp["valid_len"])
    Y_ref = mha.forward(*args)
    Y = mha.forward_no_alloc(*args)
    torch.cuda.synchronize()
    return Y, Y_ref


def test_no_alloc_matches_forward_on_two_calls_in_a_row():
    # the second call finds the first call's intermediates in the shared
    # scratch; it must not depend on them
    for w, inp in (_case("no_alloc_causal", "causal", 31),
                   _case("no_alloc_padding", "causal_padding", 32, lengths=[700, 129])):
        Y, Y_ref = _both(w, inp)
        assert torch.isfinite(Y.float()).all()
        assert rel_err(f64(Y), f64(Y_ref)) <= TOL["bf16"]


def test_no_alloc_rejects_sizes_beyond_its_scratch():
    lib = mha.load()
    P = ctypes.c_void_p
    fake = [P(4096 * (i + 1)) for i in range(7)]
    # B=16, T=2048, h=16, d=64 needs ~128 MiB of intermediates
    st = lib.mha_forward_no_alloc(*fake[:6], fake[6], 16, 2048, 2048, 1024, 16, 64, 64, 1024,
                                  0.125, 0, None, 1, None)
    assert st == 4  # MHA_ERR_WORKSPACE
