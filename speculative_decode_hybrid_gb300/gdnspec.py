"""Python binding of libgdnspec (the C ABI declared in include/gdnspec.h).

Argument marshalling only: every step of the path runs in the library's
CUDA kernels. Device arrays are torch CUDA tensors (PyTorch provides the
memory and the stream); the functions keep the C names and raise GdnError on
a non-zero status. There is no CPU fallback: if the library is missing or
cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
# GDNSPEC_LIB selects another build of the library (e.g. the bounds-checking
# _lib/libgdnspec_debug.so) for the whole process.
LIB_PATH = os.environ.get("GDNSPEC_LIB") or os.path.join(_HERE, "_lib", "libgdnspec.so")

GDN_F32 = 0
GDN_BF16 = 1

GDN_OK = 0
GDN_ERR_NULL = 1
GDN_ERR_DIMS = 2
GDN_ERR_ALIGN = 3
GDN_ERR_DTYPE = 4
GDN_ERR_TREE_ROOT = 5
GDN_ERR_TREE_PARENT = 6
GDN_ERR_TREE_DEPTH = 7
GDN_ERR_TREE_TRUNCATED = 8
GDN_ERR_TREE_NOT_CHAIN = 9
GDN_ERR_WORKSPACE = 10
GDN_ERR_CUDA = 11
GDN_ERR_FLAGS = 12

GDN_VERIFY_STATE_READY = 0x1

GDN_DEV_TOKEN_RANGE = 0x1
GDN_DEV_NAN_LOGIT = 0x2
GDN_DEV_NODE_RANGE = 0x4
GDN_DEV_TREE = 0x8
GDN_DEV_SCHED = 0x10
GDN_DEV_BOUNDS = 0x20

GDN_MAX_TOKENS = 64
GDN_MAX_CONV_K = 8
GDN_MAX_TOPK = 32
GDN_WY_MAX_TOKENS = 16

EXPORTED = ("gdn_verify_span", "gdn_tree_verify", "spec_accept_greedy",
            "spec_accept_workspace_bytes", "gdn_rollback_restore", "gdn_tree_check",
            "gdn_status_str", "gdn_verify_span_nockpt", "gdn_commit_replay", "spec_topk",
            "spec_topk_workspace_bytes", "gdn_verify_span_wy", "gdn_commit_wy", "gdn_verify_span_ex",
            "gdn_tree_verify_ex", "gdn_verify_span_pipelined", "gdn_tree_verify_pipelined")


class GdnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: status {status} ({status_str(status)})")


class gdn_dims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("layers", ctypes.c_int32),
                ("h_k", ctypes.c_int32), ("h_v", ctypes.c_int32),
                ("d_k", ctypes.c_int32), ("d_v", ctypes.c_int32),
                ("conv_ch", ctypes.c_int32), ("conv_k", ctypes.c_int32),
                ("in_dtype", ctypes.c_int32), ("q_scale", ctypes.c_float)]


def make_dims(batch, layers, h_k, h_v, d_k, d_v, conv_k, in_dtype, q_scale=1.0, conv_ch=None) -> gdn_dims:
    if conv_ch is None:
        conv_ch = 2 * h_k * d_k + h_v * d_v
    return gdn_dims(batch, layers, h_k, h_v, d_k, d_v, conv_ch, conv_k, in_dtype, float(q_scale))


_lock = threading.Lock()
_lib = None


def load(path: Optional[str] = None):
    """Load libgdnspec.so (built by speculative_decode_hybrid_gb300.build)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"libgdnspec.so not found at {p}: build it first "
                "(python -m speculative_decode_hybrid_gb300.build); there is no fallback path")
        lib = ctypes.CDLL(p)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        dp = ctypes.POINTER(gdn_dims)
        lib.gdn_verify_span.argtypes = [dp, i32] + [vp] * 9 + [vp, vp]
        lib.gdn_tree_verify.argtypes = [dp, i32, vp, vp] + [vp] * 9 + [vp, vp]
        u32 = ctypes.c_uint32
        lib.gdn_verify_span_ex.argtypes = [dp, i32] + [vp] * 9 + [vp, u32, vp]
        lib.gdn_tree_verify_ex.argtypes = [dp, i32, vp, vp] + [vp] * 9 + [vp, u32, vp]
        lib.gdn_verify_span_pipelined.argtypes = [dp, i32] + [vp] * 9 + [vp, u32, vp, vp]
        lib.gdn_tree_verify_pipelined.argtypes = [dp, i32, vp, vp] + [vp] * 9 + [vp, u32, vp, vp]
        lib.spec_accept_greedy.argtypes = [i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, sz, vp, vp]
        lib.spec_accept_workspace_bytes.argtypes = [i32, i32]
        lib.spec_accept_workspace_bytes.restype = sz
        lib.gdn_rollback_restore.argtypes = [dp, i32, vp, vp, vp, vp, vp, vp, vp]
        lib.spec_topk.argtypes = [i32, i32, i32, vp, vp, vp, vp, sz, vp, vp]
        lib.spec_topk_workspace_bytes.argtypes = [i32, i32]
        lib.spec_topk_workspace_bytes.restype = sz
        lib.gdn_verify_span_nockpt.argtypes = [dp, i32] + [vp] * 7 + [vp, vp]
        lib.gdn_commit_replay.argtypes = [dp, i32] + [vp] * 9
        lib.gdn_verify_span_wy.argtypes = [dp, i32] + [vp] * 7 + [vp, vp]
        lib.gdn_commit_wy.argtypes = [dp, i32] + [vp] * 9
        lib.gdn_tree_check.argtypes = [vp, i32, i32, i32, i32]
        lib.gdn_status_str.argtypes = [ctypes.c_int]
        lib.gdn_status_str.restype = ctypes.c_char_p
        for f in ("gdn_verify_span", "gdn_tree_verify", "gdn_verify_span_ex", "gdn_tree_verify_ex",
                  "gdn_verify_span_pipelined", "gdn_tree_verify_pipelined", "spec_accept_greedy",
                  "gdn_rollback_restore", "gdn_tree_check", "gdn_verify_span_nockpt",
                  "gdn_commit_replay", "spec_topk", "gdn_verify_span_wy", "gdn_commit_wy"):
            getattr(lib, f).restype = ctypes.c_int
        _lib = lib
        return lib


def status_str(status: int) -> str:
    try:
        return load().gdn_status_str(int(status)).decode()
    except Exception:  # library missing: still describe the code
        return "status %d" % status


def _ptr(t) -> Optional[int]:
    """Raw pointer of a tensor / numpy array / int / None."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if hasattr(t, "data_ptr"):
        return t.data_ptr()
    if hasattr(t, "ctypes"):
        return t.ctypes.data
    raise TypeError(f"cannot take a pointer of {type(t)}")


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ok(rc: int, what: str):
    if rc != GDN_OK:
        raise GdnError(rc, what)


def gdn_verify_span(dims: gdn_dims, n_tok: int, x, a, b, conv_w, ssm_in, conv_in,
                    ssm_ckpt, conv_ckpt, out, dev_status=None, stream=None, flags: int = 0,
                    x_ready=None) -> None:
    """gdn_verify_span; gdn_verify_span_ex when flags (GDN_VERIFY_*) are given;
    gdn_verify_span_pipelined when x_ready (device int32 [batch][layers]) is."""
    args = (ctypes.byref(dims), int(n_tok), _ptr(x), _ptr(a), _ptr(b), _ptr(conv_w), _ptr(ssm_in),
            _ptr(conv_in), _ptr(ssm_ckpt), _ptr(conv_ckpt), _ptr(out), _ptr(dev_status))
    if x_ready is not None:
        _ok(load().gdn_verify_span_pipelined(*args, int(flags), _ptr(x_ready), _stream(stream)),
            "gdn_verify_span_pipelined")
    elif flags:
        _ok(load().gdn_verify_span_ex(*args, int(flags), _stream(stream)), "gdn_verify_span_ex")
    else:
        _ok(load().gdn_verify_span(*args, _stream(stream)), "gdn_verify_span")


def gdn_tree_verify(dims: gdn_dims, n_nodes: int, parent_host, parent_dev, x, a, b, conv_w, ssm_in,
                    conv_in, ssm_ckpt, conv_ckpt, out, dev_status=None, stream=None, flags: int = 0,
                    x_ready=None) -> None:
    """gdn_tree_verify; gdn_tree_verify_ex when flags (GDN_VERIFY_*) are given;
    gdn_tree_verify_pipelined when x_ready (device int32 [batch][layers]) is."""
    import numpy as np
    ph = None
    if parent_host is not None:
        ph = np.ascontiguousarray(parent_host, dtype=np.int32)
    args = (ctypes.byref(dims), int(n_nodes), _ptr(ph), _ptr(parent_dev), _ptr(x), _ptr(a), _ptr(b),
            _ptr(conv_w), _ptr(ssm_in), _ptr(conv_in), _ptr(ssm_ckpt), _ptr(conv_ckpt), _ptr(out),
            _ptr(dev_status))
    if x_ready is not None:
        _ok(load().gdn_tree_verify_pipelined(*args, int(flags), _ptr(x_ready), _stream(stream)),
            "gdn_tree_verify_pipelined")
    elif flags:
        _ok(load().gdn_tree_verify_ex(*args, int(flags), _stream(stream)), "gdn_tree_verify_ex")
    else:
        _ok(load().gdn_tree_verify(*args, _stream(stream)), "gdn_tree_verify")


def spec_accept_workspace_bytes(batch: int, n_nodes: int) -> int:
    return int(load().spec_accept_workspace_bytes(int(batch), int(n_nodes)))


def spec_accept_greedy(batch: int, n_nodes: int, vocab: int, logits, tokens, parent_dev,
                       argmax_out, accept_len, accept_node, workspace, workspace_bytes: int,
                       dev_status=None, stream=None) -> None:
    rc = load().spec_accept_greedy(int(batch), int(n_nodes), int(vocab), _ptr(logits), _ptr(tokens),
                                   _ptr(parent_dev), _ptr(argmax_out), _ptr(accept_len),
                                   _ptr(accept_node), _ptr(workspace), int(workspace_bytes),
                                   _ptr(dev_status), _stream(stream))
    _ok(rc, "spec_accept_greedy")


def gdn_rollback_restore(dims: gdn_dims, n_tok: int, accept_node_dev, ssm_ckpt, conv_ckpt,
                         ssm_state, conv_state, dev_status=None, stream=None) -> None:
    rc = load().gdn_rollback_restore(ctypes.byref(dims), int(n_tok), _ptr(accept_node_dev),
                                     _ptr(ssm_ckpt), _ptr(conv_ckpt), _ptr(ssm_state),
                                     _ptr(conv_state), _ptr(dev_status), _stream(stream))
    _ok(rc, "gdn_rollback_restore")


def gdn_verify_span_nockpt(dims: gdn_dims, n_tok: int, x, a, b, conv_w, ssm_in, conv_in, out,
                           dev_status=None, stream=None) -> None:
    rc = load().gdn_verify_span_nockpt(ctypes.byref(dims), int(n_tok), _ptr(x), _ptr(a), _ptr(b),
                                       _ptr(conv_w), _ptr(ssm_in), _ptr(conv_in), _ptr(out),
                                       _ptr(dev_status), _stream(stream))
    _ok(rc, "gdn_verify_span_nockpt")


def gdn_commit_replay(dims: gdn_dims, n_tok: int, accept_len_dev, x, a, b, conv_w, ssm_state,
                      conv_state, dev_status=None, stream=None) -> None:
    rc = load().gdn_commit_replay(ctypes.byref(dims), int(n_tok), _ptr(accept_len_dev), _ptr(x), _ptr(a),
                                  _ptr(b), _ptr(conv_w), _ptr(ssm_state), _ptr(conv_state),
                                  _ptr(dev_status), _stream(stream))
    _ok(rc, "gdn_commit_replay")


def gdn_verify_span_wy(dims: gdn_dims, n_tok: int, x, a, b, conv_w, ssm_in, conv_in, out,
                       dev_status=None, stream=None) -> None:
    rc = load().gdn_verify_span_wy(ctypes.byref(dims), int(n_tok), _ptr(x), _ptr(a), _ptr(b),
                                   _ptr(conv_w), _ptr(ssm_in), _ptr(conv_in), _ptr(out),
                                   _ptr(dev_status), _stream(stream))
    _ok(rc, "gdn_verify_span_wy")


def gdn_commit_wy(dims: gdn_dims, n_tok: int, accept_len_dev, x, a, b, conv_w, ssm_state,
                  conv_state, dev_status=None, stream=None) -> None:
    rc = load().gdn_commit_wy(ctypes.byref(dims), int(n_tok), _ptr(accept_len_dev), _ptr(x), _ptr(a),
                              _ptr(b), _ptr(conv_w), _ptr(ssm_state), _ptr(conv_state),
                              _ptr(dev_status), _stream(stream))
    _ok(rc, "gdn_commit_wy")


def spec_topk_workspace_bytes(rows: int, k: int) -> int:
    return int(load().spec_topk_workspace_bytes(int(rows), int(k)))


def spec_topk(rows: int, vocab: int, k: int, logits, idx_out, val_out, workspace, workspace_bytes: int,
              dev_status=None, stream=None) -> None:
    rc = load().spec_topk(int(rows), int(vocab), int(k), _ptr(logits), _ptr(idx_out), _ptr(val_out),
                          _ptr(workspace), int(workspace_bytes), _ptr(dev_status), _stream(stream))
    _ok(rc, "spec_topk")


def gdn_tree_check(parent_host, batch: int, n_nodes: int, require_chain: bool = False,
                   max_depth: int = 0) -> int:
    """Host-only geometry check; returns the status code (does not raise)."""
    import numpy as np
    ph = None if parent_host is None else np.ascontiguousarray(parent_host, dtype=np.int32)
    return int(load().gdn_tree_check(_ptr(ph), int(batch), int(n_nodes), int(bool(require_chain)),
                                     int(max_depth)))


GDN_STATIC_SCRATCH_BYTES = 1 << 20


def spec_accept_greedy_static(batch: int, n_nodes: int, vocab: int, logits, tokens, parent_dev,
                              argmax_out, accept_len, accept_node, dev_status=None, stream=None) -> None:
    """spec_accept_greedy without a workspace argument, for callers that
    cannot allocate device memory: the library's fixed 1 MiB device scratch
    is used instead. All calls share that scratch, so calls that may overlap
    on the GPU must be serialised by the caller; make the first call on a
    device before any stream capture (it looks up the scratch's address)."""
    lib = load()
    f = lib.spec_accept_greedy_static
    if not getattr(f, "_gdn_typed", False):
        vp, i32 = ctypes.c_void_p, ctypes.c_int32
        f.argtypes = [i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp]
        f.restype = ctypes.c_int
        f._gdn_typed = True
    rc = f(int(batch), int(n_nodes), int(vocab), _ptr(logits), _ptr(tokens), _ptr(parent_dev),
           _ptr(argmax_out), _ptr(accept_len), _ptr(accept_node), _ptr(dev_status), _stream(stream))
    _ok(rc, "spec_accept_greedy_static")
