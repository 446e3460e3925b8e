"""CPU-only checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects bad calls on the host before anything is queued
(no GPU needed: every call here fails validation before any CUDA call)."""
import ctypes
import os
import re

import numpy as np
import pytest

from golden_cases import tree_geometry_cases
from speculative_decode_hybrid_gb300 import build as B
from speculative_decode_hybrid_gb300 import gdnspec as G

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdnspec.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return G.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w \*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while")))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("gdn_verify_span", "gdn_tree_verify", "spec_accept_greedy", "gdn_rollback_restore"):
        assert n in names
    assert set(G.EXPORTED) <= set(names)


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n
        assert isinstance(getattr(lib, n), ctypes._CFuncPtr)


def test_status_strings(lib):
    for code in range(0, 13):
        s = G.status_str(code)
        assert s and s != "unknown status", code
    assert G.status_str(999) == "unknown status"


@pytest.mark.parametrize("case", tree_geometry_cases(), ids=lambda c: c[0])
def test_tree_check_golden(lib, case):
    name, mode, parent, want = case
    expect = {"ok": G.GDN_OK, "root": G.GDN_ERR_TREE_ROOT, "parent": G.GDN_ERR_TREE_PARENT,
              "truncated": G.GDN_ERR_TREE_TRUNCATED, "not_chain": G.GDN_ERR_TREE_NOT_CHAIN,
              "null": G.GDN_ERR_NULL}[want]
    n = 2 if parent is None else len(parent)
    arr = None if parent is None else np.array(parent, dtype=np.int32)
    if parent is not None and len(parent) == 0:
        arr = np.zeros(1, dtype=np.int32)
    rc = G.gdn_tree_check(arr, 1, n, require_chain=(mode == "chain"))
    assert rc == expect, (name, rc)


def test_tree_check_depth_and_batch(lib):
    chain = np.arange(-1, 17, dtype=np.int32)     # 18 nodes, depth 17
    assert G.gdn_tree_check(chain, 1, 18, max_depth=17) == G.GDN_OK
    assert G.gdn_tree_check(chain, 1, 18, max_depth=16) == G.GDN_ERR_TREE_DEPTH
    two = np.stack([chain, chain.copy()])
    two[1, 5] = 7
    assert G.gdn_tree_check(two, 1, 18) == G.GDN_OK          # only the first request checked
    assert G.gdn_tree_check(two, 2, 18) == G.GDN_ERR_TREE_PARENT
    assert G.gdn_tree_check(chain, 0, 18) == G.GDN_ERR_DIMS


FAKE = 0x10000  # a 16-byte aligned non-NULL address that is never dereferenced


def _dims(**kw):
    d = dict(batch=1, layers=2, h_k=2, h_v=4, d_k=64, d_v=64, conv_k=4, in_dtype=G.GDN_F32)
    d.update(kw)
    return G.make_dims(**d)


def _verify(lib, dims, n_tok, **ptrs):
    p = dict(x=FAKE, a=FAKE, b=FAKE, w=FAKE, ssm_in=FAKE, conv_in=FAKE, ck=FAKE, cc=FAKE, out=FAKE)
    p.update(ptrs)
    return lib.gdn_verify_span(ctypes.byref(dims) if dims is not None else None, n_tok, p["x"], p["a"],
                               p["b"], p["w"], p["ssm_in"], p["conv_in"], p["ck"], p["cc"], p["out"],
                               p.get("ds"), None)


@pytest.mark.parametrize("bad", [
    dict(d_k=96), dict(d_k=32), dict(d_v=8), dict(d_v=72), dict(h_v=3), dict(conv_k=0), dict(conv_k=9),
    dict(batch=0), dict(layers=0), dict(batch=300, layers=300), dict(conv_ch=1000)])
def test_verify_rejects_bad_dims(lib, bad):
    assert _verify(lib, _dims(**bad), 4) == G.GDN_ERR_DIMS


def test_verify_rejects_before_launch(lib):
    assert _verify(lib, None, 4) == G.GDN_ERR_NULL
    assert _verify(lib, _dims(), 0) == G.GDN_ERR_DIMS
    assert _verify(lib, _dims(), 65) == G.GDN_ERR_DIMS
    assert _verify(lib, _dims(in_dtype=7), 4) == G.GDN_ERR_DTYPE
    d = _dims()
    d.q_scale = float("nan")
    assert _verify(lib, d, 4) == G.GDN_ERR_DIMS
    for name in ("x", "a", "b", "w", "ssm_in", "conv_in", "ck", "cc", "out"):
        assert _verify(lib, _dims(), 4, **{name: None}) == G.GDN_ERR_NULL, name
    for name in ("ssm_in", "ck", "out", "conv_in", "cc"):
        assert _verify(lib, _dims(), 4, **{name: FAKE + 4}) == G.GDN_ERR_ALIGN, name
    assert _verify(lib, _dims(in_dtype=G.GDN_BF16), 4, x=FAKE + 1) == G.GDN_ERR_ALIGN
    assert _verify(lib, _dims(), 4, ds=FAKE + 2) == G.GDN_ERR_ALIGN
    # K == 1 needs no conv buffers, but still validates everything else
    assert _verify(lib, _dims(conv_k=1, d_v=72), 4, conv_in=None, cc=None) == G.GDN_ERR_DIMS


def test_tree_verify_rejects_bad_geometry_before_launch(lib):
    d = _dims()
    par = np.array([-1, 0, 3, 1], dtype=np.int32)  # forward parent
    rc = lib.gdn_tree_verify(ctypes.byref(d), 4, par.ctypes.data, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                             FAKE, FAKE, FAKE, FAKE, None, None)
    assert rc == G.GDN_ERR_TREE_PARENT
    par = np.array([0, 0, 1, 2], dtype=np.int32)
    rc = lib.gdn_tree_verify(ctypes.byref(d), 4, par.ctypes.data, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                             FAKE, FAKE, FAKE, FAKE, None, None)
    assert rc == G.GDN_ERR_TREE_ROOT
    rc = lib.gdn_tree_verify(ctypes.byref(d), 1, par.ctypes.data, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                             FAKE, FAKE, FAKE, FAKE, None, None)
    assert rc == G.GDN_ERR_TREE_TRUNCATED
    rc = lib.gdn_tree_verify(ctypes.byref(d), 4, None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                             FAKE, FAKE, FAKE, FAKE, None, None)
    assert rc == G.GDN_ERR_NULL


def test_accept_workspace_and_validation(lib):
    ws = G.spec_accept_workspace_bytes(1, 17)
    assert ws >= 17 * 8 and ws % 8 == 0
    assert G.spec_accept_workspace_bytes(16, 23) > G.spec_accept_workspace_bytes(1, 23)
    assert G.spec_accept_workspace_bytes(0, 17) == 0
    assert G.spec_accept_workspace_bytes(1, 66) == 0

    def call(B=1, N=17, V=1000, logits=FAKE, tokens=FAKE, am=FAKE, kl=FAKE, kn=FAKE, wsp=FAKE, wsb=None):
        wsb = ws if wsb is None else wsb
        return lib.spec_accept_greedy(B, N, V, logits, tokens, None, am, kl, kn, wsp, wsb, None, None)

    assert call(B=0) == G.GDN_ERR_DIMS
    assert call(N=0) == G.GDN_ERR_DIMS
    assert call(N=66) == G.GDN_ERR_DIMS
    assert call(V=0) == G.GDN_ERR_DIMS
    assert call(logits=None) == G.GDN_ERR_NULL
    assert call(kn=None) == G.GDN_ERR_NULL
    assert call(logits=FAKE + 4) == G.GDN_ERR_ALIGN
    assert call(wsp=None) == G.GDN_ERR_WORKSPACE
    assert call(wsb=ws - 1) == G.GDN_ERR_WORKSPACE
    assert call(wsp=FAKE + 16) == G.GDN_ERR_WORKSPACE


def test_restore_validation(lib):
    d = _dims()

    def call(dims=d, n=4, node=FAKE, ck=FAKE, cc=FAKE, st=FAKE, cs=FAKE):
        return lib.gdn_rollback_restore(ctypes.byref(dims) if dims is not None else None, n, node, ck, cc,
                                        st, cs, None, None)

    assert call(dims=None) == G.GDN_ERR_NULL
    assert call(n=0) == G.GDN_ERR_DIMS
    assert call(node=None) == G.GDN_ERR_NULL
    assert call(ck=None) == G.GDN_ERR_NULL
    assert call(st=FAKE + 8) == G.GDN_ERR_ALIGN
    assert call(cc=FAKE + 8) == G.GDN_ERR_ALIGN


def test_replay_entry_points_validate_before_launch(lib):
    d = _dims()
    f = lib.gdn_verify_span_nockpt
    assert f(ctypes.byref(d), 0, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None) == G.GDN_ERR_DIMS
    assert f(ctypes.byref(d), 4, FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, None, None) == G.GDN_ERR_NULL
    assert f(ctypes.byref(d), 4, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE + 4, None, None) == G.GDN_ERR_ALIGN
    assert f(ctypes.byref(d), 4, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE + 2, None) == G.GDN_ERR_ALIGN
    g = lib.gdn_commit_replay
    assert g(None, 4, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None) == G.GDN_ERR_NULL
    assert g(ctypes.byref(d), 65, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None) == G.GDN_ERR_DIMS
    assert g(ctypes.byref(d), 4, None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None) == G.GDN_ERR_NULL
    assert g(ctypes.byref(d), 4, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE + 8, FAKE, None, None) == G.GDN_ERR_ALIGN
    assert g(ctypes.byref(d), 4, FAKE + 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None) == G.GDN_ERR_ALIGN


def test_wy_entry_points_validate_before_launch(lib):
    d = _dims()
    f = lib.gdn_verify_span_wy
    assert f(ctypes.byref(d), 0, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None) == G.GDN_ERR_DIMS
    assert f(ctypes.byref(d), G.GDN_WY_MAX_TOKENS + 1, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None,
             None) == G.GDN_ERR_DIMS
    assert f(ctypes.byref(d), G.GDN_WY_MAX_TOKENS, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None,
             None) == G.GDN_ERR_NULL
    assert f(ctypes.byref(d), 4, FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, None, None) == G.GDN_ERR_NULL
    assert f(ctypes.byref(d), 4, FAKE + 4, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None) == G.GDN_ERR_ALIGN
    assert f(ctypes.byref(d), 4, FAKE, FAKE, FAKE, FAKE + 8, FAKE, FAKE, FAKE, None, None) == G.GDN_ERR_ALIGN
    assert f(ctypes.byref(d), 4, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE + 4, None, None) == G.GDN_ERR_ALIGN
    assert f(ctypes.byref(d), 4, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE + 2, None) == G.GDN_ERR_ALIGN
    g = lib.gdn_commit_wy
    assert g(None, 4, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None) == G.GDN_ERR_NULL
    assert g(ctypes.byref(d), G.GDN_WY_MAX_TOKENS + 1, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None,
             None) == G.GDN_ERR_DIMS
    assert g(ctypes.byref(d), 4, None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None) == G.GDN_ERR_NULL
    assert g(ctypes.byref(d), 4, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE + 8, FAKE, None, None) == G.GDN_ERR_ALIGN
    assert g(ctypes.byref(d), 4, FAKE + 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None) == G.GDN_ERR_ALIGN


def test_topk_validation(lib):
    ws = G.spec_topk_workspace_bytes(4, 8)
    assert ws > 0 and G.spec_topk_workspace_bytes(4, 33) == 0 and G.spec_topk_workspace_bytes(0, 8) == 0
    f = lib.spec_topk
    assert f(4, 100, 0, FAKE, FAKE, FAKE, FAKE, ws, None, None) == G.GDN_ERR_DIMS
    assert f(4, 100, 33, FAKE, FAKE, FAKE, FAKE, ws, None, None) == G.GDN_ERR_DIMS
    assert f(4, 7, 8, FAKE, FAKE, FAKE, FAKE, ws, None, None) == G.GDN_ERR_DIMS
    assert f(4, 100, 8, None, FAKE, FAKE, FAKE, ws, None, None) == G.GDN_ERR_NULL
    assert f(4, 100, 8, FAKE + 4, FAKE, FAKE, FAKE, ws, None, None) == G.GDN_ERR_ALIGN
    assert f(4, 100, 8, FAKE, FAKE, FAKE, FAKE, ws - 8, None, None) == G.GDN_ERR_WORKSPACE


def test_verify_ex_validates_flags_before_launch(lib):
    """The flagged entry points check everything gdn_verify_span /
    gdn_tree_verify check, and reject flag bits the library does not define
    (GDN_ERR_FLAGS) before anything is queued."""
    d = _dims()
    args = [FAKE] * 9
    assert lib.gdn_verify_span_ex(ctypes.byref(d), 4, *args, None, 0x2, None) == G.GDN_ERR_FLAGS
    assert lib.gdn_verify_span_ex(ctypes.byref(d), 4, *args, None, 0x80000000, None) == G.GDN_ERR_FLAGS
    assert lib.gdn_verify_span_ex(ctypes.byref(d), 0, *args, None, G.GDN_VERIFY_STATE_READY, None) == \
        G.GDN_ERR_DIMS
    assert lib.gdn_verify_span_ex(None, 4, *args, None, 0, None) == G.GDN_ERR_NULL
    par = np.array([-1, 0, 1, 1], dtype=np.int32)
    assert lib.gdn_tree_verify_ex(ctypes.byref(d), 4, par.ctypes.data, *args, FAKE, None, 0x4, None) == \
        G.GDN_ERR_FLAGS
    bad = np.array([-1, 0, 3, 1], dtype=np.int32)
    assert lib.gdn_tree_verify_ex(ctypes.byref(d), 4, bad.ctypes.data, *args, FAKE, None,
                                  G.GDN_VERIFY_STATE_READY, None) == G.GDN_ERR_TREE_PARENT


def test_pipelined_verify_validates_before_launch(lib):
    """The _pipelined calls check what the _ex calls check, plus the input-flag
    array's alignment (GDN_ERR_ALIGN), before anything is queued; with a null
    x_ready they are the _ex calls."""
    d = _dims()
    args = [FAKE] * 9
    odd = ctypes.c_void_p(FAKE + 2)  # not 4-byte aligned
    assert lib.gdn_verify_span_pipelined(ctypes.byref(d), 4, *args, None, 0, odd, None) == G.GDN_ERR_ALIGN
    assert lib.gdn_verify_span_pipelined(ctypes.byref(d), 4, *args, None, 0x2, FAKE, None) == G.GDN_ERR_FLAGS
    assert lib.gdn_verify_span_pipelined(ctypes.byref(d), 0, *args, None, 0, FAKE, None) == G.GDN_ERR_DIMS
    assert lib.gdn_verify_span_pipelined(None, 4, *args, None, 0, FAKE, None) == G.GDN_ERR_NULL
    bad_x = [None] + [FAKE] * 8  # x missing
    assert lib.gdn_verify_span_pipelined(ctypes.byref(d), 4, *bad_x, None, 0, FAKE, None) == G.GDN_ERR_NULL
    par = np.array([-1, 0, 1, 1], dtype=np.int32)
    assert lib.gdn_tree_verify_pipelined(ctypes.byref(d), 4, par.ctypes.data, *args, FAKE, None, 0, odd,
                                         None) == G.GDN_ERR_ALIGN
    assert lib.gdn_tree_verify_pipelined(ctypes.byref(d), 4, par.ctypes.data, *args, FAKE, None, 0x4, FAKE,
                                         None) == G.GDN_ERR_FLAGS
    bad = np.array([-1, 0, 3, 1], dtype=np.int32)
    assert lib.gdn_tree_verify_pipelined(ctypes.byref(d), 4, bad.ctypes.data, *args, FAKE, None, 0, FAKE,
                                         None) == G.GDN_ERR_TREE_PARENT
