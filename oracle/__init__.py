"""CPU oracle for GDN span verify + greedy acceptance + rollback.

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package. The CUDA
product path never imports it and shares no code with it.

The arithmetic lives in ``gdn_oracle.c`` (plain C, every value in double);
this module only marshals numpy arrays to it. ``build()`` compiles it with
gcc. Parity is pinned by closed forms, invariants, library routines and
brute force in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIB = os.path.join(_HERE, "_gdn_oracle.so")
_lock = threading.Lock()
_lib = None

ORA_OK = 0
ORA_ERR_ARG = 1
ORA_ERR_TREE = 2


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile the oracle shared library (gcc, no FMA contraction)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            i32, dbl, lng = ctypes.c_int, ctypes.c_double, ctypes.c_longlong
            vp = ctypes.c_void_p
            lib.ora_conv1d_silu.argtypes = [i32, i32, vp, vp, vp, vp, vp]
            lib.ora_l2norm.argtypes = [i32, vp]
            lib.ora_l2norm.restype = None
            lib.ora_gdn_delta_rule.argtypes = [i32, i32, i32] + [vp] * 8
            lib.ora_gdn_delta_rule_explicit.argtypes = [i32, i32, i32] + [vp] * 8
            lib.ora_tree_depths.argtypes = [i32, vp, vp]
            lib.ora_gdn_verify_layer.argtypes = [i32] * 6 + [vp] * 7 + [dbl, vp, vp, vp]
            lib.ora_argmax_f32.argtypes = [i32, vp]
            lib.ora_accept_greedy.argtypes = [i32, i32, vp, vp, vp, vp, vp, vp]
            lib.ora_restore.argtypes = [lng, i32, vp, vp]
            lib.ora_topk_f32.argtypes = [i32, vp, i32, vp, vp]
            for f in ("ora_conv1d_silu", "ora_gdn_delta_rule", "ora_gdn_delta_rule_explicit",
                      "ora_tree_depths", "ora_gdn_verify_layer", "ora_argmax_f32",
                      "ora_accept_greedy", "ora_restore", "ora_topk_f32"):
                getattr(lib, f).restype = ctypes.c_int
            _lib = lib
    return _lib


def _d(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc != ORA_OK:
        raise OracleError(f"{what}: oracle status {rc}")


def conv1d_silu(w, state, x):
    """Causal conv1d + SiLU of one channel over a chain.
    w [K], state [K-1] (oldest first), x [T] -> (y [T], state_after [T][K-1])."""
    w, x = _d(w), _d(x)
    K, T = w.shape[0], x.shape[0]
    state = _d(state) if K > 1 else np.zeros(0)
    y = np.zeros(T)
    st = np.zeros((T, max(K - 1, 0)))
    _check(_load().ora_conv1d_silu(K, T, _p(w), _p(state), _p(x), _p(y), _p(st)), "conv1d_silu")
    return y, st


def l2norm(v):
    v = _d(v).copy()
    _load().ora_l2norm(v.shape[0], _p(v))
    return v


def delta_rule(q, k, v, a, b, S0, explicit: bool = False):
    """Gated delta rule of one head, inputs fed straight to the recurrence.
    q,k [T][d_k]; v [T][d_v]; a,b [T]; S0 [d_v][d_k] -> (S [T][d_v][d_k], o [T][d_v])."""
    q, k, v, a, b, S0 = map(_d, (q, k, v, a, b, S0))
    T, d_k = q.shape
    d_v = v.shape[1]
    S = np.zeros((T, d_v, d_k))
    o = np.zeros((T, d_v))
    f = _load().ora_gdn_delta_rule_explicit if explicit else _load().ora_gdn_delta_rule
    _check(f(d_k, d_v, T, _p(q), _p(k), _p(v), _p(a), _p(b), _p(S0), _p(S), _p(o)), "delta_rule")
    return S, o


def tree_depths(parent):
    parent = np.ascontiguousarray(parent, dtype=np.int32)
    depth = np.zeros(parent.shape[0], dtype=np.int32)
    rc = _load().ora_tree_depths(parent.shape[0], _p(parent), _p(depth))
    return rc, depth


def verify_layer(h_k, h_v, d_k, d_v, K, x, a, b, w, ssm_in, conv_in, *,
                 parent=None, q_scale: float = 1.0):
    """Verify one (request, layer) over N-1 processed nodes.

    x [T][C]; a,b [T][H_v]; w [C][K]; ssm_in [H_v][d_v][d_k]; conv_in [C][K-1];
    parent [N] (tree) or None (chain). Returns (ssm_ckpt [T][H_v][d_v][d_k],
    conv_ckpt [T][C][K-1], out [T][H_v][d_v]) in float64."""
    x, a, b, w, ssm_in = map(_d, (x, a, b, w, ssm_in))
    conv_in = _d(conv_in) if K > 1 else np.zeros(0)
    T, C = x.shape
    N = T + 1
    par = None
    if parent is not None:
        par = np.ascontiguousarray(parent, dtype=np.int32)
        if par.shape[0] != N:
            raise OracleError("parent length must be T + 1")
    ck = np.zeros((T, h_v, d_v, d_k))
    cc = np.zeros((T, C, max(K - 1, 0)))
    out = np.zeros((T, h_v, d_v))
    rc = _load().ora_gdn_verify_layer(
        h_k, h_v, d_k, d_v, K, N, _p(par) if par is not None else None,
        _p(x), _p(a), _p(b), _p(w), _p(ssm_in), _p(conv_in), float(q_scale),
        _p(ck), _p(cc), _p(out))
    _check(rc, "verify_layer")
    return ck, cc, out


def argmax_f32(row):
    row = np.ascontiguousarray(row, dtype=np.float32)
    return int(_load().ora_argmax_f32(row.shape[0], _p(row)))


def accept_greedy(logits, tokens, parent=None):
    """Greedy acceptance of one request. logits [N][V] fp32; tokens [N];
    parent [N] or None. Returns (argmax [N] int32, accept_len, accept_node)."""
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    N, V = logits.shape
    par = np.ascontiguousarray(parent, dtype=np.int32) if parent is not None else None
    am = np.zeros(N, dtype=np.int32)
    kl = np.zeros(1, dtype=np.int32)
    kn = np.zeros(1, dtype=np.int32)
    rc = _load().ora_accept_greedy(N, V, _p(logits), _p(tokens),
                                   _p(par) if par is not None else None,
                                   _p(am), _p(kl), _p(kn))
    _check(rc, "accept_greedy")
    return am, int(kl[0]), int(kn[0])


def restore(ckpt, node: int, state):
    """state <- ckpt[node-1] (node > 0); node 0 leaves state unchanged.
    ckpt [T][...]; state [...] float64. Returns the new state."""
    state = _d(state).copy()
    ckpt = _d(ckpt)
    n = state.size
    _check(_load().ora_restore(n, int(node), _p(ckpt), _p(state)), "restore")
    return state


def verify_request(wl, r: int, layers=None, q_scale: float = 1.0):
    """Run the oracle over request r of a workload (all or some layers).
    Returns lists of per-layer (ssm_ckpt, conv_ckpt, out)."""
    s = wl.shape
    layers = range(s.layers) if layers is None else layers
    par = wl.parent[r] if wl.parent is not None else None
    res = []
    for y in layers:
        res.append(verify_layer(s.h_k, s.h_v, s.d_k, s.d_v, s.conv_k,
                                wl.x_f[r, y], wl.a_f[r, y], wl.b_f[r, y],
                                wl.conv_w_f[y], wl.ssm0[r, y], wl.conv0[r, y],
                                parent=par, q_scale=q_scale))
    return res


def topk_f32(row, k: int):
    """Top-k of a row: NaN first, then larger values, lower index on ties.
    Returns (idx [k] int32, val [k] float32)."""
    row = np.ascontiguousarray(row, dtype=np.float32)
    idx = np.zeros(k, dtype=np.int32)
    val = np.zeros(k, dtype=np.float32)
    _check(_load().ora_topk_f32(row.shape[0], _p(row), int(k), _p(idx), _p(val)), "topk_f32")
    return idx, val
