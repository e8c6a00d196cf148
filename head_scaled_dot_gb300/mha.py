"""Python binding of the C ABI in include/mha.h (ctypes).

Argument marshalling only: every step of the forward pass runs in the CUDA
library. torch supplies device memory, the current stream and tensor
metadata. If the library has not been built, loading raises: there is no
fallback path.
"""

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmha_gb300.so")

MHA_OK = 0
STATUS_NAMES = {
    0: "MHA_OK",
    1: "MHA_ERR_INVALID_ARG",
    2: "MHA_ERR_UNSUPPORTED",
    3: "MHA_ERR_EMPTY_ROW",
    4: "MHA_ERR_WORKSPACE",
    5: "MHA_ERR_CUDA",
    6: "MHA_ERR_DEVICE_TIMEOUT",
}
MASKS = {"none": 0, "causal": 1, "padding": 2, "causal_padding": 3}
DTYPES = {"f32": 0, "bf16": 1}
TORCH_DTYPES = {torch.float32: "f32", torch.bfloat16: "bf16"}

# Symbols declared in include/mha.h.
EXPORTS = (
    "mha_workspace_size", "mha_workspace_layout", "mha_forward", "mha_qkv_projection", "mha_attention",
    "mha_output_projection", "mha_get_device_error", "mha_status_string",
    "mha_selftest_wait_timeout", "mha_kernel_launch_count", "mha_version",
    "mha_forward_no_alloc", "mha_forward_general", "mha_decode_workspace_size",
    "mha_attention_decode", "mha_attention_plan", "mha_attention_split_workspace_size",
    "mha_attention_split",
)

_lib = None


class MHAError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        super().__init__("%s: %s (%s)" % (what, STATUS_NAMES.get(status, status),
                                         status_string(status) if _lib else ""))


def load(path=LIB_PATH):
    """Loads the shared library once and declares the C signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError("libmha_gb300.so is not built (run __graft_entry__.build()): " + path)
    lib = ctypes.CDLL(path)
    P, I, F, S, U64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_uint64
    lib.mha_workspace_size.restype = S
    lib.mha_workspace_size.argtypes = [I] * 8 + [I]
    lib.mha_workspace_layout.restype = I
    lib.mha_workspace_layout.argtypes = [I] * 6 + [I, ctypes.POINTER(S)]
    lib.mha_forward.restype = I
    lib.mha_forward.argtypes = [P] * 7 + [I] * 8 + [F, I, P, I, P, S, P]
    lib.mha_forward_general.restype = I
    lib.mha_forward_general.argtypes = [P] * 8 + [I] * 10 + [F, I, P, I, P, I, P, S, P]
    lib.mha_decode_workspace_size.restype = S
    lib.mha_decode_workspace_size.argtypes = [I] * 5
    lib.mha_attention_decode.restype = I
    lib.mha_attention_decode.argtypes = [P] * 4 + [I] * 6 + [F, P, I, I, P, S, P]
    lib.mha_forward_no_alloc.restype = I
    lib.mha_forward_no_alloc.argtypes = [P] * 7 + [I] * 8 + [F, I, P, I, P]
    lib.mha_qkv_projection.restype = I
    lib.mha_qkv_projection.argtypes = [P] * 8 + [I] * 7 + [I, P, I, P, P]
    lib.mha_attention.restype = I
    lib.mha_attention.argtypes = [P] * 4 + [I] * 6 + [F, I, P, I, I, P, P]
    lib.mha_output_projection.restype = I
    lib.mha_output_projection.argtypes = [P] * 3 + [I] * 5 + [P, I, P, P]
    lib.mha_get_device_error.restype = I
    lib.mha_get_device_error.argtypes = [P, P]
    lib.mha_status_string.restype = ctypes.c_char_p
    lib.mha_status_string.argtypes = [I]
    lib.mha_selftest_wait_timeout.restype = I
    lib.mha_selftest_wait_timeout.argtypes = [P, U64, P]
    lib.mha_kernel_launch_count.restype = U64
    lib.mha_kernel_launch_count.argtypes = []
    lib.mha_version.restype = ctypes.c_char_p
    lib.mha_version.argtypes = []
    lib.mha_attention_plan.restype = I
    lib.mha_attention_plan.argtypes = [I] * 6 + [I, P, I, I, I, P, P, S, P]
    lib.mha_attention_split_workspace_size.restype = S
    lib.mha_attention_split_workspace_size.argtypes = [I] * 7
    lib.mha_attention_split.restype = I
    lib.mha_attention_split.argtypes = [P] * 4 + [I] * 6 + [F, I, P, I, I, I, P, S, P, P]
    _lib = lib
    return lib


def status_string(status):
    return load().mha_status_string(int(status)).decode()


def _ptr(t):
    """Device pointer of a tensor (or an int / c_void_p passed through)."""
    if t is None:
        return None
    if isinstance(t, ctypes.c_void_p):
        return t
    if isinstance(t, int):
        return ctypes.c_void_p(t)
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status, what):
    if status != MHA_OK:
        raise MHAError(status, what)


def _lens(valid_len, B):
    """Host int32 array of valid lengths (or None) and the object keeping it alive."""
    if valid_len is None:
        return None, None
    arr = (ctypes.c_int32 * B)(*[int(x) for x in list(valid_len)[:B]])
    return ctypes.cast(arr, ctypes.c_void_p), arr


def workspace_size(B, n_q, n_k, d_model, h, d_h, d_vh, d_o, dtype):
    return int(load().mha_workspace_size(B, n_q, n_k, d_model, h, d_h, d_vh, d_o, DTYPES[dtype]))


def workspace_layout(B, n_q, n_k, h, d_h, d_vh, dtype):
    """Byte offsets of the error word, Q, K, V, Z and the total size."""
    off = (ctypes.c_size_t * 6)()
    _check(load().mha_workspace_layout(B, n_q, n_k, h, d_h, d_vh, DTYPES[dtype], off),
           "mha_workspace_layout")
    return dict(zip(("err", "q", "k", "v", "z", "total"), [int(x) for x in off]))


def attention_plan(B, n_q, n_k, h, d_h, d_vh, mask="none", valid_len=None,
                   self_attention=True, num_sms=152, nsplit=1):
    """The tensor-core attention schedule for a GPU with num_sms SMs (host
    only): (grid, records), records an int32 array of rows (cta, b, head, q0,
    ntiles, key0, key1), CTA by CTA in processing order. nsplit: 1 the
    schedule of mha_attention, 0 that of mha_forward (automatic split over
    the keys), n > 1 a split into n key ranges."""
    import numpy as np
    lib = load()
    lens_arg, keep = _lens(valid_len, B)
    grid = ctypes.c_int32()
    n = ctypes.c_size_t()
    args = (B, n_q, n_k, h, d_h, d_vh, MASKS[mask], lens_arg, 1 if self_attention else 0,
            int(nsplit), num_sms, ctypes.byref(grid))
    _check(lib.mha_attention_plan(*args, None, 0, ctypes.byref(n)), "mha_attention_plan")
    rec = (ctypes.c_int32 * (7 * max(1, n.value)))()
    _check(lib.mha_attention_plan(*args, rec, n.value, ctypes.byref(n)), "mha_attention_plan")
    del keep
    return grid.value, np.ctypeslib.as_array(rec).reshape(-1, 7)[:n.value].copy()


def attention_split_workspace_size(B, n_q, n_k, h, d_h, d_vh, nsplit=0):
    return int(load().mha_attention_split_workspace_size(B, n_q, n_k, h, d_h, d_vh, int(nsplit)))


def launch_count():
    return int(load().mha_kernel_launch_count())


def forward(X_q, X_kv, W_Q, W_K, W_V, W_O, h, d_h, d_vh, c, mask="none", valid_len=None,
            out=None, workspace=None, stream=None, check=True):
    """Y = MHA(X_q, X_kv) on the GPU. Tensors: CUDA, contiguous, one dtype
    (float32 or bfloat16). X_kv None means self-attention. Returns Y
    (B, n_q, d_o); with check=True the device error word is read back
    (one stream synchronisation)."""
    lib = load()
    B, n_q, d_model = X_q.shape
    n_k = n_q if X_kv is None else X_kv.shape[1]
    d_o = W_O.shape[1]
    dt = TORCH_DTYPES[X_q.dtype]
    if out is None:
        out = torch.empty((B, n_q, d_o), dtype=X_q.dtype, device=X_q.device)
    ws_bytes = workspace_size(B, n_q, n_k, d_model, h, d_h, d_vh, d_o, dt)
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=X_q.device)
    lens, keep = _lens(valid_len, B)
    st = lib.mha_forward(_ptr(X_q), _ptr(X_kv), _ptr(W_Q), _ptr(W_K), _ptr(W_V), _ptr(W_O),
                         _ptr(out), B, n_q, n_k, d_model, h, d_h, d_vh, d_o, float(c),
                         MASKS[mask], lens, DTYPES[dt], _ptr(workspace),
                         workspace.numel() * workspace.element_size(), _stream(stream))
    del keep
    _check(st, "mha_forward")
    if check:
        _check(lib.mha_get_device_error(_ptr(workspace), _stream(stream)), "mha_forward (device)")
    return out


def forward_general(X_q, X_k, X_v, W_Q, W_K, W_V, W_O, h, d_h, d_vh, c, mask="none",
                    valid_len=None, self_attention=False, head_gate=None, out=None,
                    workspace=None, stream=None, check=True):
    """mha_forward_general: separate query, key and value inputs of their own
    widths, X_q (B, n_q, d_q), X_k (B, n_k, d_k), X_v (B, n_k, d_v); head_gate
    (h floats, or None) scales each head's output block before W_O (0 ablates
    the head). Returns Y (B, n_q, d_o)."""
    lib = load()
    B, n_q, d_q = X_q.shape
    n_k, d_k = X_k.shape[1], X_k.shape[2]
    d_v = X_v.shape[2]
    d_o = W_O.shape[1]
    dt = TORCH_DTYPES[X_q.dtype]
    if out is None:
        out = torch.empty((B, n_q, d_o), dtype=X_q.dtype, device=X_q.device)
    ws_bytes = workspace_size(B, n_q, n_k, d_q, h, d_h, d_vh, d_o, dt)
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=X_q.device)
    lens, keep = _lens(valid_len, B)
    gate = None
    if head_gate is not None:
        gate = (ctypes.c_float * h)(*[float(x) for x in head_gate])
    st = lib.mha_forward_general(_ptr(X_q), _ptr(X_k), _ptr(X_v), _ptr(W_Q), _ptr(W_K),
                                 _ptr(W_V), _ptr(W_O), _ptr(out), B, n_q, n_k, d_q, d_k, d_v, h,
                                 d_h, d_vh, d_o, float(c), MASKS[mask], lens,
                                 int(bool(self_attention)),
                                 None if gate is None else ctypes.cast(gate, ctypes.c_void_p),
                                 DTYPES[dt], _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _stream(stream))
    del keep, gate
    _check(st, "mha_forward_general")
    if check:
        _check(lib.mha_get_device_error(_ptr(workspace), _stream(stream)),
               "mha_forward_general (device)")
    return out


NO_ALLOC_SCRATCH_BYTES = 32 << 20


def forward_no_alloc(X_q, X_kv, W_Q, W_K, W_V, W_O, h, d_h, d_vh, c, mask="none",
                     valid_len=None, out=None, stream=None):
    """mha_forward_no_alloc: the forward pass with the library's own fixed
    32 MiB device scratch instead of a workspace (for callers that cannot
    allocate). `out` (B, n_q, d_o) is the only buffer the caller provides."""
    lib = load()
    B, n_q, d_model = X_q.shape
    n_k = n_q if X_kv is None else X_kv.shape[1]
    d_o = W_O.shape[1]
    dt = TORCH_DTYPES[X_q.dtype]
    if out is None:
        out = torch.empty((B, n_q, d_o), dtype=X_q.dtype, device=X_q.device)
    lens, keep = _lens(valid_len, B)
    st = lib.mha_forward_no_alloc(_ptr(X_q), _ptr(X_kv), _ptr(W_Q), _ptr(W_K), _ptr(W_V),
                                  _ptr(W_O), _ptr(out), B, n_q, n_k, d_model, h, d_h, d_vh, d_o,
                                  float(c), MASKS[mask], lens, DTYPES[dt], _stream(stream))
    del keep
    _check(st, "mha_forward_no_alloc")
    return out


def qkv_projection(X_q, X_kv, W_Q, W_K, W_V, h, d_h, d_vh, mask="none", valid_len=None,
                   out=None, dev_error=None, stream=None):
    """Step 1: head-split Q (B,h,n_q,d_h), K (B,h,n_k,d_h), V (B,h,n_k,d_vh).
    With a padding mask only the rows the attention step reads are written
    (below valid_len[b] rounded up to 128). out: (Q, K, V) to write into."""
    lib = load()
    B, n_q, d_model = X_q.shape
    n_k = n_q if X_kv is None else X_kv.shape[1]
    dt = TORCH_DTYPES[X_q.dtype]
    kw = dict(dtype=X_q.dtype, device=X_q.device)
    if out is None:
        out = (torch.empty((B, h, n_q, d_h), **kw), torch.empty((B, h, n_k, d_h), **kw),
               torch.empty((B, h, n_k, d_vh), **kw))
    Q, K, V = out
    lens, keep = _lens(valid_len, B)
    st = lib.mha_qkv_projection(_ptr(X_q), _ptr(X_kv), _ptr(W_Q), _ptr(W_K), _ptr(W_V),
                                _ptr(Q), _ptr(K), _ptr(V), B, n_q, n_k, d_model, h, d_h, d_vh,
                                MASKS[mask], lens, DTYPES[dt], _ptr(dev_error), _stream(stream))
    del keep
    _check(st, "mha_qkv_projection")
    return Q, K, V


def attention(Q, K, V, c, mask="none", valid_len=None, self_attention=True, out=None,
              dev_error=None, stream=None):
    """Step 2: Z (B, n_q, h*d_vh) from head-split Q, K, V."""
    lib = load()
    B, h, n_q, d_h = Q.shape
    n_k, d_vh = V.shape[2], V.shape[3]
    dt = TORCH_DTYPES[Q.dtype]
    if out is None:
        out = torch.empty((B, n_q, h * d_vh), dtype=Q.dtype, device=Q.device)
    lens, keep = _lens(valid_len, B)
    st = lib.mha_attention(_ptr(Q), _ptr(K), _ptr(V), _ptr(out), B, n_q, n_k, h, d_h, d_vh,
                           float(c), MASKS[mask], lens, int(bool(self_attention)), DTYPES[dt],
                           _ptr(dev_error), _stream(stream))
    del keep
    _check(st, "mha_attention")
    return out


def attention_split(Q, K, V, c, mask="none", valid_len=None, self_attention=True, nsplit=0,
                    out=None, workspace=None, dev_error=None, stream=None):
    """mha_attention_split: step 2 with the keys of each query tile cut into
    nsplit ranges on separate thread blocks, their summaries merged (0: the
    automatic choice)."""
    lib = load()
    B, h, n_q, d_h = Q.shape
    n_k, d_vh = V.shape[2], V.shape[3]
    dt = TORCH_DTYPES[Q.dtype]
    if out is None:
        out = torch.empty((B, n_q, h * d_vh), dtype=Q.dtype, device=Q.device)
    if workspace is None:
        nbytes = attention_split_workspace_size(B, n_q, n_k, h, d_h, d_vh, nsplit)
        workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=Q.device)
    lens, keep = _lens(valid_len, B)
    st = lib.mha_attention_split(_ptr(Q), _ptr(K), _ptr(V), _ptr(out), B, n_q, n_k, h, d_h,
                                 d_vh, float(c), MASKS[mask], lens, int(bool(self_attention)),
                                 int(nsplit), DTYPES[dt], _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _ptr(dev_error),
                                 _stream(stream))
    del keep
    _check(st, "mha_attention_split")
    return out


def output_projection(Z, W_O, h, d_vh, valid_len=None, out=None, dev_error=None, stream=None):
    """Step 3: Y = Z W_O. valid_len (self-attention padding): the rows
    i >= valid_len[b] are padded query rows, zero in Z and written as zeros."""
    lib = load()
    B, n_q, _ = Z.shape
    d_o = W_O.shape[1]
    dt = TORCH_DTYPES[Z.dtype]
    if out is None:
        out = torch.empty((B, n_q, d_o), dtype=Z.dtype, device=Z.device)
    lens, keep = _lens(valid_len, B)
    st = lib.mha_output_projection(_ptr(Z), _ptr(W_O), _ptr(out), B, n_q, h, d_vh, d_o, lens,
                                   DTYPES[dt], _ptr(dev_error), _stream(stream))
    del keep
    _check(st, "mha_output_projection")
    return out


def decode_workspace_size(B, n_q, n_k, h, d_vh):
    return int(load().mha_decode_workspace_size(B, n_q, n_k, h, d_vh))


def attention_decode(Q, K, V, c, cache_len=None, causal_tail=False, out=None, workspace=None,
                     stream=None):
    """mha_attention_decode: Z (B, n_q, h*d_vh) for the new query rows Q
    (B, h, n_q, d_h) over the cache K (B, h, n_k, d_h), V (B, h, n_k, d_vh)
    holding cache_len[b] valid positions."""
    lib = load()
    B, h, n_q, d_h = Q.shape
    n_k, d_vh = V.shape[2], V.shape[3]
    dt = TORCH_DTYPES[Q.dtype]
    if out is None:
        out = torch.empty((B, n_q, h * d_vh), dtype=Q.dtype, device=Q.device)
    if workspace is None:
        workspace = torch.empty(decode_workspace_size(B, n_q, n_k, h, d_vh), dtype=torch.uint8,
                                device=Q.device)
    lens, keep = _lens(cache_len, B)
    st = lib.mha_attention_decode(_ptr(Q), _ptr(K), _ptr(V), _ptr(out), B, n_q, n_k, h, d_h,
                                  d_vh, float(c), lens, int(bool(causal_tail)), DTYPES[dt],
                                  _ptr(workspace), workspace.numel() * workspace.element_size(),
                                  _stream(stream))
    del keep
    _check(st, "mha_attention_decode")
    return out


def get_device_error(error_word, stream=None):
    """Reads and resets a device error word; returns the status code."""
    return int(load().mha_get_device_error(_ptr(error_word), _stream(stream)))


def selftest_wait_timeout(dev_error, limit_ns, stream=None):
    _check(load().mha_selftest_wait_timeout(_ptr(dev_error), int(limit_ns), _stream(stream)),
           "mha_selftest_wait_timeout")
