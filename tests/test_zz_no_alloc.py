"""spec_accept_greedy_static: greedy acceptance for callers that cannot
allocate device memory (it uses the library's fixed device scratch instead
of a caller workspace). Its results must equal spec_accept_greedy's, call
after call, since every call reuses the same scratch.

This file is collected last on purpose: a run that stops at the first
failure has run every other test before it."""
import ctypes

import numpy as np
import pytest
import torch

from speculative_decode_hybrid_gb300 import build as B
from speculative_decode_hybrid_gb300 import gdnspec as G
from speculative_decode_hybrid_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    B.build()
    G.load()


def _both(logits, tokens, parent=None):
    """Run the workspace entry point and the static one on the same inputs
    through the C ABI; return both sets of outputs."""
    Bn, N, V = logits.shape
    dev = torch.device("cuda")
    lg = torch.from_numpy(np.ascontiguousarray(logits, dtype=np.float32)).to(dev)
    tk = torch.from_numpy(np.ascontiguousarray(tokens, dtype=np.int32)).to(dev)
    pr = None if parent is None else torch.from_numpy(np.ascontiguousarray(parent, dtype=np.int32)).to(dev)
    outs = []
    for static in (False, True):
        am = torch.full((Bn, N), -5, dtype=torch.int32, device=dev)
        kl = torch.full((Bn,), -5, dtype=torch.int32, device=dev)
        kn = torch.full((Bn,), -5, dtype=torch.int32, device=dev)
        ds = torch.zeros((1,), dtype=torch.int32, device=dev)
        if static:
            G.spec_accept_greedy_static(Bn, N, V, lg, tk, pr, am, kl, kn, ds)
        else:
            wsb = G.spec_accept_workspace_bytes(Bn, N)
            ws = torch.zeros((wsb,), dtype=torch.uint8, device=dev)
            G.spec_accept_greedy(Bn, N, V, lg, tk, pr, am, kl, kn, ws, wsb, ds)
        torch.cuda.synchronize()
        outs.append(tuple(t.cpu().numpy() for t in (am, kl, kn, ds)))
    return outs


def _same(a, b):
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


def test_static_matches_workspace_entry_two_calls_in_a_row():
    # call 1: a 48-layer-style chain step (17 rows of the Qwen vocabulary)
    wl = W.make_workload(2, seed=9, layers=1)
    ref, got = _both(wl.logits, wl.tokens)
    _same(ref, got)
    assert int(got[1][0]) == 2
    # call 2, straight after, with a different shape: 16 requests, ties and
    # an out-of-range token, so stale scratch from call 1 would show
    g = np.random.default_rng(77)
    logits = g.integers(-2, 3, (16, 17, 50000)).astype(np.float32)
    tokens = g.integers(0, 50000, (16, 17)).astype(np.int32)
    am_ref = logits.argmax(axis=2)
    tokens[:, 1:6] = am_ref[:, 0:5]
    tokens[3, 2] = 70000
    ref, got = _both(logits, tokens)
    _same(ref, got)
    assert int(got[3][0]) & G.GDN_DEV_TOKEN_RANGE


def test_static_matches_workspace_entry_on_trees():
    for seed in (3, 4):
        wl = W.make_workload(3, seed=seed, layers=1)
        ref, got = _both(wl.logits, wl.tokens, wl.parent)
        _same(ref, got)


def test_static_rejects_sizes_beyond_its_scratch():
    lib = G.load()
    dev = torch.device("cuda")
    n = 65
    batch = 1  # the smallest batch whose scratch no longer fits
    while G.spec_accept_workspace_bytes(batch, n) <= G.GDN_STATIC_SCRATCH_BYTES:
        batch += 1
    assert G.spec_accept_workspace_bytes(batch, n) > G.GDN_STATIC_SCRATCH_BYTES
    dummy = torch.zeros((16,), dtype=torch.float32, device=dev)
    with pytest.raises(G.GdnError) as e:
        G.spec_accept_greedy_static(batch, n, 4, dummy, dummy, None, dummy, dummy, dummy)
    assert e.value.status == G.GDN_ERR_WORKSPACE
    assert hasattr(lib, "spec_accept_greedy_static")
    assert isinstance(lib.spec_accept_greedy_static, ctypes._CFuncPtr)
