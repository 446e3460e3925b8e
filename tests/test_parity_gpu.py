"""GPU parity: the CUDA path (called through the C ABI) against the CPU oracle
on the same seeded inputs.

Bit-exact: accepted lengths and nodes, argmax indices, conv checkpoints
(shifted copies of the inputs) and restored bytes (against the GPU's own
checkpoint slot). Within 2e-3 normwise per (request, layer, slot, head)
slice: SSM checkpoints, outputs, restored state against the oracle.
"""
import dataclasses
import zlib

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import (TOL, check_accept_vs_oracle, check_layer_vs_oracle, check_restore,
                         ensure_built, run, slice_rel_err)
from speculative_decode_hybrid_gb300 import gdnspec as G
from speculative_decode_hybrid_gb300 import workloads as W
from speculative_decode_hybrid_gb300.pipeline import SpecStep

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    ensure_built()


def full_check(wl, layers=None, requests=None):
    st = run(wl)
    s = wl.shape
    layers = list(range(s.layers)) if layers is None else layers
    requests = list(range(s.batch)) if requests is None else requests
    refs = {}
    for r in requests:
        res = oracle.verify_request(wl, r, layers=layers)
        for y, ref in zip(layers, res):
            check_layer_vs_oracle(st, wl, r, y, ref)
            refs[(r, y)] = ref
    kl, kn = check_accept_vs_oracle(st, wl)
    check_restore(st, wl, kn, layers=layers, ref_layers=refs)
    assert int(st.dev_status.item()) == 0
    return st, kl, kn


# ------------------------------------------------------------ the five workloads

def test_workload0_tiny_chain():
    full_check(W.make_workload(0, seed=0))


def test_workload1_single_layer():
    full_check(W.make_workload(1, seed=1))


def test_workload2_full_size_all_layers():
    """48 layers, span 16, batch 1 at full size; every layer against the oracle."""
    wl = W.make_workload(2, seed=2)
    st, kl, kn = full_check(wl)
    assert 0 <= int(kl[0]) <= 16


def test_workload3_tree_full_size_all_layers():
    wl = W.make_workload(3, seed=3)
    depth = oracle.tree_depths(wl.parent[0])[1]
    assert depth.max() <= 16
    st, kl, kn = full_check(wl)
    assert int(kl[0]) == int(depth[int(kn[0])])


def test_workload4_batched_full_size_every_request():
    """16 requests x 48 layers (25 GiB of checkpoints): acceptance of every
    request; checkpoints, outputs and restored state of every request against
    the oracle on two layers each (different layers for different requests,
    so the 32 pairs cover the first, middle and last layers); restored bytes
    of every request against its own slot on three layers."""
    wl = W.make_workload(4, seed=4)
    st = run(wl)
    kl, kn = check_accept_vs_oracle(st, wl)
    s = wl.shape
    pairs = [(r, y) for r in range(s.batch) for y in sorted({(3 * r) % s.layers, (s.layers - 1 - 3 * r) % s.layers})]
    assert len(pairs) == 2 * s.batch
    assert {y for _, y in pairs} >= {0, s.layers - 1}
    refs = {}
    for r, y in pairs:
        refs[(r, y)] = oracle.verify_request(wl, r, layers=[y])[0]
        check_layer_vs_oracle(st, wl, r, y, refs[(r, y)])
    for r in range(s.batch):
        node = int(kn[r])
        for y in (0, 29, 47):
            g = st.ssm_state[r, y].cpu().numpy()
            want = wl.ssm0[r, y] if node == 0 else st.ssm_ckpt[r, y, node - 1].cpu().numpy()
            np.testing.assert_array_equal(g, want)
    for (r, y), (ck, cc, _) in refs.items():
        want = oracle.restore(ck, int(kn[r]), wl.ssm0[r, y])
        assert slice_rel_err(st.ssm_state[r, y].cpu().numpy(), want, s.d_v * s.d_k) <= TOL
        want_c = oracle.restore(cc, int(kn[r]), wl.conv0[r, y])
        np.testing.assert_array_equal(st.conv_state[r, y].cpu().numpy(), want_c.astype(np.float32))
    assert int(st.dev_status.item()) == 0
    assert len(set(int(k) for k in kl)) > 1  # independent acceptance per request


# ------------------------------------------------------------ shapes and edges

def shape(**kw):
    base = dict(batch=1, layers=2, h_k=2, h_v=4, d_k=128, d_v=128, conv_k=4, n_nodes=6,
                vocab=3000, dtype=W.GDN_BF16)
    base.update(kw)
    return W.Shape(**base)


EDGE_SHAPES = {
    "two_row_blocks_ragged": shape(h_k=1, h_v=3, d_v=192, n_nodes=6),
    "min_rows_f32_one_token": shape(h_k=2, h_v=2, d_k=64, d_v=16, n_nodes=2, dtype=W.GDN_F32),
    "max_tokens": shape(d_k=64, d_v=32, n_nodes=65),
    "conv_k1": shape(conv_k=1, d_k=64, d_v=64),
    "conv_k2": shape(conv_k=2),
    "conv_k8": shape(conv_k=8, n_nodes=12),
    "ratio1_batch3": shape(batch=3, h_k=4, h_v=4, d_v=48, layers=3),
    "gqa4_dk64_bf16": shape(h_k=1, h_v=4, d_k=64, d_v=128),
    "vocab_odd": shape(vocab=1001),
    "vocab_tiny": shape(vocab=3, n_nodes=9),
    "wide_dv_four_row_blocks": shape(h_k=1, h_v=2, d_v=512, n_nodes=5, layers=1),
}


@pytest.mark.parametrize("name", sorted(EDGE_SHAPES))
def test_edge_shapes_chain(name):
    full_check(W.draw(EDGE_SHAPES[name], seed=zlib.crc32(name.encode()) % 1000))


@pytest.mark.parametrize("name", ["two_row_blocks_ragged", "max_tokens", "conv_k8", "ratio1_batch3",
                                  "vocab_tiny"])
def test_edge_shapes_tree(name):
    s = dataclasses.replace(EDGE_SHAPES[name], tree=True)
    full_check(W.draw(s, seed=7 + len(name)))


def test_q_scale():
    wl = W.draw(shape(), seed=11)
    st = SpecStep(wl, q_scale=0.08838834764831845)
    st.verify()
    torch.cuda.synchronize()
    for y in range(2):
        ref = oracle.verify_request(wl, 0, layers=[y], q_scale=0.08838834764831845)[0]
        check_layer_vs_oracle(st, wl, 0, y, ref)


def test_star_and_deep_trees():
    for par in (np.array([-1] + [0] * 9, dtype=np.int32), W.chain_parent(10),
                np.array([-1, 0, 1, 1, 3, 0, 5, 6, 2, 8], dtype=np.int32)):
        s = shape(n_nodes=10, tree=True)
        wl = W.draw(s, seed=21)
        wl.parent[0] = par
        full_check(wl)


# ------------------------------------------------------------ invariants on the GPU

def test_gpu_restore_at_k_equals_replay_of_first_k():
    """Verifying only the first k tokens gives, bit for bit, checkpoint k-1
    of the full span (and restore copies exactly that slot)."""
    wl = W.make_workload(1, seed=5)
    full = run(wl, restore=False)
    full_ck = full.ssm_ckpt.cpu()
    full_cc = full.conv_ckpt.cpu()
    full_out = full.out.cpu()
    for k in (1, 2, 7, 16):
        sub = dataclasses.replace(wl, shape=dataclasses.replace(wl.shape, n_nodes=k + 1),
                                  x=wl.x[:, :, :k], a=wl.a[:, :, :k], b=wl.b[:, :, :k],
                                  x_f=wl.x_f[:, :, :k], a_f=wl.a_f[:, :, :k], b_f=wl.b_f[:, :, :k],
                                  logits=wl.logits[:, :k + 1], tokens=wl.tokens[:, :k + 1])
        st = run(sub, restore=False)
        assert torch.equal(st.ssm_ckpt.cpu()[:, :, k - 1], full_ck[:, :, k - 1])
        assert torch.equal(st.conv_ckpt.cpu()[:, :, k - 1], full_cc[:, :, k - 1])
        assert torch.equal(st.out.cpu()[:, :, :k], full_out[:, :, :k])


def test_gpu_tree_that_is_a_chain_equals_chain():
    wl = W.make_workload(1, seed=6)
    chain = run(wl)
    twl = dataclasses.replace(wl, shape=dataclasses.replace(wl.shape, tree=True),
                              parent=W.chain_parent(wl.shape.n_nodes)[None, :].copy())
    tree = run(twl)
    assert torch.equal(chain.ssm_ckpt, tree.ssm_ckpt)
    assert torch.equal(chain.conv_ckpt, tree.conv_ckpt)
    assert torch.equal(chain.out, tree.out)
    assert torch.equal(chain.accept_node, tree.accept_node)
    assert torch.equal(chain.ssm_state, tree.ssm_state)


def test_gpu_tree_many_root_children_d64_big_launch():
    """A launch big enough for 128-row items (10 layers x 32 heads): the tree
    instantiation that parks the root's rows in tensor memory, at d_k = 64,
    with a root of five children (four restarts from the parked rows), and
    every layer checked against the oracle."""
    s = shape(h_k=16, h_v=32, d_k=64, d_v=64, layers=10, n_nodes=12, tree=True)
    wl = W.draw(s, seed=61)
    par = np.array([[-1, 0, 0, 0, 1, 1, 2, 0, 4, 0, 9, 3]], dtype=np.int32)
    wl = dataclasses.replace(wl, parent=par)
    st = run(wl)
    for y, ref in enumerate(oracle.verify_request(wl, 0)):
        check_layer_vs_oracle(st, wl, 0, y, ref)
    assert int(st.dev_status.item()) == 0


def test_gpu_deterministic():
    wl = W.make_workload(3, seed=8, layers=4)
    a = run(wl)
    b = run(wl)
    for name in ("ssm_ckpt", "conv_ckpt", "out", "argmax", "accept_len", "accept_node", "ssm_state",
                 "conv_state"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name


def test_gpu_writes_stay_in_bounds():
    """Guard regions around every output keep their canary pattern."""
    wl = W.draw(shape(h_k=1, h_v=3, d_v=192, n_nodes=7, batch=2), seed=9)
    st = SpecStep(wl)
    pad = 4096
    canary = -12345.678

    def guarded(t):
        buf = torch.full((t.numel() + 2 * pad,), canary, dtype=t.dtype, device=t.device)
        return buf, buf[pad:pad + t.numel()].view(t.shape)

    gck, st.ssm_ckpt = guarded(st.ssm_ckpt)
    gcc, st.conv_ckpt = guarded(st.conv_ckpt)
    go, st.out = guarded(st.out)
    gs, view = guarded(st.ssm_state)
    view.copy_(st.ssm_state)
    st.ssm_state = view
    st.step()
    torch.cuda.synchronize()
    for buf in (gck, gcc, go, gs):
        assert bool((buf[:pad] == canary).all()) and bool((buf[-pad:] == canary).all())
    assert not bool((st.ssm_ckpt == canary).any())


# ------------------------------------------------------------ acceptance edges

def accept_only(logits, tokens, parent=None, dev_status=True):
    B, N, V = logits.shape
    dev = torch.device("cuda")
    lg = torch.from_numpy(np.ascontiguousarray(logits, dtype=np.float32)).to(dev)
    tk = torch.from_numpy(np.ascontiguousarray(tokens, dtype=np.int32)).to(dev)
    pr = None if parent is None else torch.from_numpy(np.ascontiguousarray(parent, dtype=np.int32)).to(dev)
    am = torch.full((B, N), -7, dtype=torch.int32, device=dev)
    kl = torch.full((B,), -7, dtype=torch.int32, device=dev)
    kn = torch.full((B,), -7, dtype=torch.int32, device=dev)
    wsb = G.spec_accept_workspace_bytes(B, N)
    ws = torch.zeros((wsb,), dtype=torch.uint8, device=dev)
    ds = torch.zeros((1,), dtype=torch.int32, device=dev)
    G.spec_accept_greedy(B, N, V, lg, tk, pr, am, kl, kn, ws, wsb, ds if dev_status else None)
    torch.cuda.synchronize()
    return am.cpu().numpy(), kl.cpu().numpy(), kn.cpu().numpy(), int(ds.item()), ws


def expect_oracle(logits, tokens, parent, am, kl, kn):
    for r in range(logits.shape[0]):
        o = oracle.accept_greedy(logits[r], tokens[r], None if parent is None else parent[r])
        np.testing.assert_array_equal(am[r], o[0])
        assert (int(kl[r]), int(kn[r])) == o[1:], r


def test_accept_ties_signed_zero_and_split_boundaries():
    g = np.random.default_rng(30)
    V = 151936
    logits = g.standard_normal((3, 5, V)).astype(np.float32)
    # row 0: equal maxima far apart (different CTAs); row 1: all zeros with mixed signs
    logits[0, 0, [70000, 5, 151935, 123456]] = 9.0
    logits[0, 1] = 0.0
    logits[0, 1, ::3] = -0.0
    logits[0, 2, [151935, 151934]] = 10.0
    logits[1, :, :] = -np.inf
    logits[1, 3, 42] = -1e30
    tokens = g.integers(0, V, (3, 5)).astype(np.int32)
    am, kl, kn, ds, _ = accept_only(logits, tokens)
    assert am[0, 0] == 5 and am[0, 1] == 0 and am[0, 2] == 151934 and am[1, 0] == 0 and am[1, 3] == 42
    expect_oracle(logits, tokens, None, am, kl, kn)
    assert ds == 0


def test_accept_nan_flag_and_first_nan():
    g = np.random.default_rng(31)
    logits = g.standard_normal((1, 3, 4096)).astype(np.float32)
    logits[0, 1, [3000, 17, 4000]] = np.nan
    tokens = np.array([[0, 1, 2]], dtype=np.int32)
    am, kl, kn, ds, _ = accept_only(logits, tokens)
    assert am[0, 1] == 17
    expect_oracle(logits, tokens, None, am, kl, kn)
    assert ds & G.GDN_DEV_NAN_LOGIT


def test_accept_all_match_and_token_range():
    g = np.random.default_rng(32)
    V, L = 151936, 16
    logits = g.standard_normal((2, L + 1, V)).astype(np.float32)
    am_ref = logits.argmax(axis=2)
    tokens = np.zeros((2, L + 1), dtype=np.int32)
    tokens[:, 1:] = am_ref[:, :-1]
    tokens[1, 9] = V + 3            # out of range: a mismatch, flagged
    am, kl, kn, ds, ws = accept_only(logits, tokens)
    assert list(kl) == [L, 8] and list(kn) == [L, 8]
    assert ds & G.GDN_DEV_TOKEN_RANGE
    assert int(ws.count_nonzero().item()) == 0  # keys and counters are back to zero
    expect_oracle(logits, tokens, None, am, kl, kn)


@pytest.mark.parametrize("V", [1, 5, 1001, 4096, 151936])
def test_accept_vocab_sizes_and_root_only(V):
    g = np.random.default_rng(V)
    for N in (1, 2, 17, 65):
        logits = g.integers(-2, 3, (2, N, V)).astype(np.float32)   # many ties
        am_ref = logits.argmax(axis=2)
        tokens = g.integers(0, V, (2, N)).astype(np.int32)
        mask = g.random((2, N)) < 0.7
        for r in range(2):
            for i in range(1, N):
                if mask[r, i]:
                    tokens[r, i] = am_ref[r, i - 1]
        am, kl, kn, _, _ = accept_only(logits, tokens)
        expect_oracle(logits, tokens, None, am, kl, kn)


def test_accept_trees_with_duplicate_siblings_vs_oracle():
    """Tiny vocabularies force duplicate sibling tokens: the deepest matching
    node wins, then the lower index at the first divergence."""
    g = np.random.default_rng(33)
    for trial in range(20):
        B, N, V = 16, int(g.integers(2, 24)), int(g.integers(1, 4))
        logits = g.integers(0, 3, (B, N, V)).astype(np.float32)
        tokens = g.integers(0, V, (B, N)).astype(np.int32)
        parent = np.stack([W.random_tree(g, N, 16) for _ in range(B)])
        am, kl, kn, ds, _ = accept_only(logits, tokens, parent)
        expect_oracle(logits, tokens, parent, am, kl, kn)
        assert ds == 0


def test_accept_workspace_reuse_many_calls():
    """The same workspace across calls of different shapes stays consistent."""
    g = np.random.default_rng(34)
    dev = torch.device("cuda")
    wsb = G.spec_accept_workspace_bytes(16, 65)
    ws = torch.zeros((wsb,), dtype=torch.uint8, device=dev)
    for trial in range(12):
        B, N, V = int(g.integers(1, 17)), int(g.integers(1, 66)), int(g.integers(1, 70000))
        logits = g.standard_normal((B, N, V)).astype(np.float32)
        tokens = g.integers(0, V, (B, N)).astype(np.int32)
        lg = torch.from_numpy(logits).to(dev)
        tk = torch.from_numpy(tokens).to(dev)
        am = torch.empty((B, N), dtype=torch.int32, device=dev)
        kl = torch.empty((B,), dtype=torch.int32, device=dev)
        kn = torch.empty((B,), dtype=torch.int32, device=dev)
        G.spec_accept_greedy(B, N, V, lg, tk, None, am, kl, kn, ws, wsb)
        torch.cuda.synchronize()
        expect_oracle(logits, tokens, None, am.cpu().numpy(), kl.cpu().numpy(), kn.cpu().numpy())


# ------------------------------------------------------------ restore edges

def test_restore_out_of_range_node_is_flagged_not_copied():
    wl = W.draw(shape(batch=2), seed=40)
    st = run(wl, restore=False)
    before_s = st.ssm_state.clone()
    before_c = st.conv_state.clone()
    st.accept_node.copy_(torch.tensor([wl.shape.n_tok + 1, -1], dtype=torch.int32))
    st.dev_status.zero_()
    st.restore()
    torch.cuda.synchronize()
    assert torch.equal(st.ssm_state, before_s) and torch.equal(st.conv_state, before_c)
    assert int(st.dev_status.item()) & G.GDN_DEV_NODE_RANGE
    st.accept_node.copy_(torch.tensor([wl.shape.n_tok, 0], dtype=torch.int32))
    st.restore()
    torch.cuda.synchronize()
    assert torch.equal(st.ssm_state[0], st.ssm_ckpt[0, :, -1])
    assert torch.equal(st.conv_state[0], st.conv_ckpt[0, :, -1])
    assert torch.equal(st.ssm_state[1], before_s[1])


def test_tree_device_parent_mismatch_is_flagged():
    """A device parent array that breaks parent[i] < i (host copy valid) is
    caught by the kernel: flagged, and no out-of-bounds access."""
    wl = W.draw(shape(n_nodes=6, tree=True), seed=41)
    st = SpecStep(wl)
    bad = wl.parent.copy()
    bad[0, 3] = 50
    st.parent.copy_(torch.from_numpy(bad))
    st.verify()
    torch.cuda.synchronize()
    assert int(st.dev_status.item()) & G.GDN_DEV_TREE


def test_accept_bad_device_parent_excludes_its_subtree():
    """A device parent outside [0, i) (the host copy valid) makes that node
    and everything below it unmatched and flags GDN_DEV_TREE; the rest of the
    acceptance is the oracle's on the same tree without that subtree. Every
    drafted token matches its parent's argmax, so the deepest path would run
    through the corrupted node."""
    wl = W.draw(shape(n_nodes=23, tree=True, vocab=3000), seed=43)
    par = wl.parent[0].copy()
    am = np.array([oracle.argmax_f32(wl.logits[0, n]) for n in range(23)], dtype=np.int32)
    tokens = wl.tokens.copy()
    tokens[0, 1:] = am[par[1:]]
    depth = oracle.tree_depths(par)[1]
    deepest = int(np.argmax(depth))
    node = deepest  # the child of the root on the way to the deepest node
    while par[node] != 0:
        node = int(par[node])
    below = [i for i in range(1, 23) if node in _root_path(par, i)]
    st = SpecStep(dataclasses.replace(wl, tokens=tokens))
    bad = par.copy()
    bad[node] = 50
    st.parent.copy_(torch.from_numpy(bad[None, :]))
    st.accept()
    torch.cuda.synchronize()
    want_tokens = tokens[0].copy()
    for i in below:
        want_tokens[i] = (am[par[i]] + 1) % wl.shape.vocab  # never the parent's argmax
    o_am, o_kl, o_kn = oracle.accept_greedy(wl.logits[0], want_tokens, par)
    np.testing.assert_array_equal(st.argmax[0].cpu().numpy(), o_am)
    assert (int(st.accept_len[0]), int(st.accept_node[0])) == (o_kl, o_kn)
    assert int(st.accept_node[0]) not in below
    assert int(st.dev_status.item()) & G.GDN_DEV_TREE


def _root_path(par, i):
    path = []
    while i > 0:
        path.append(i)
        i = int(par[i])
    return path


# ------------------------------------------------------------ both verify kernels

def test_fallback_kernel_long_f32_span():
    """A 64-token f32 span at d_k = 128 does not fit the persistent kernel's
    staging; the one-item-per-CTA kernel runs it."""
    s = shape(h_k=1, h_v=2, d_k=128, d_v=128, n_nodes=65, dtype=W.GDN_F32, layers=2)
    full_check(W.draw(s, seed=50))
    full_check(W.draw(dataclasses.replace(s, tree=True), seed=51))


@pytest.mark.parametrize("tree", [False, True])
def test_persistent_and_fallback_kernels_agree_bitwise(tree):
    """An x tensor that is not 16-byte aligned cannot be staged with cp.async
    and takes the fallback kernel; both kernels must give the same bytes."""
    s = shape(h_k=2, h_v=6, d_v=128, n_nodes=9, layers=3, batch=2, tree=tree)
    wl = W.draw(s, seed=52)
    a = run(wl)
    b = SpecStep(wl)
    shifted = torch.empty(b.x.numel() + 8, dtype=b.x.dtype, device=b.x.device)
    view = shifted[1:1 + b.x.numel()].view(b.x.shape)   # 2-byte offset
    view.copy_(b.x)
    b.x = view
    assert b.x.data_ptr() % 16 != 0
    b.step()
    torch.cuda.synchronize()
    for name in ("ssm_ckpt", "conv_ckpt", "out", "ssm_state", "conv_state", "accept_node"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name


# ------------------------------------------------------------ CUDA graph and host path

@pytest.mark.parametrize("wid", [2, 3])
def test_graph_replay_equals_eager_steps(wid):
    """verify -> accept -> restore captured as one CUDA graph gives the same
    bytes as the eager calls, step after step (the state evolves)."""
    wl = W.make_workload(wid, seed=60, layers=4)
    eager = SpecStep(wl)
    graph = SpecStep(wl)
    graph.capture()                    # runs one eager step first
    eager.step()                       # keep both at the same step count
    for _ in range(3):
        eager.step()
        graph.replay()
    torch.cuda.synchronize()
    for name in ("ssm_ckpt", "conv_ckpt", "out", "argmax", "accept_len", "accept_node", "ssm_state",
                 "conv_state"):
        assert torch.equal(getattr(eager, name), getattr(graph, name)), name


def test_host_buffer_step_matches_device_step():
    """The end-to-end path (pinned host inputs copied in, results copied back)
    gives the device path's acceptance."""
    from speculative_decode_hybrid_gb300.pipeline import pinned_host_inputs, run_host_step
    wl = W.make_workload(2, seed=9, layers=2)
    st = SpecStep(wl)
    host = pinned_host_inputs(wl)
    out = {"accept_len": torch.empty(1, dtype=torch.int32).pin_memory(),
           "accept_node": torch.empty(1, dtype=torch.int32).pin_memory(),
           "argmax": torch.empty((1, 17), dtype=torch.int32).pin_memory()}
    h2d, d2h = run_host_step(st, host, out)
    torch.cuda.synchronize()
    assert h2d == wl.x.nbytes + wl.a.nbytes + wl.b.nbytes + wl.logits.nbytes + wl.tokens.nbytes
    assert d2h == 4 + 4 + 17 * 4
    am, kl, kn = oracle.accept_greedy(wl.logits[0], wl.tokens[0])
    assert int(out["accept_len"][0]) == kl == 2 and int(out["accept_node"][0]) == kn
    np.testing.assert_array_equal(out["argmax"][0].numpy(), am)
    # the packed result buffer comes back in one copy with the same values
    packed = st.host_result_buffers()
    packed["_packed"].fill_(-1)
    _, d2h_p = run_host_step(st, host, packed)
    torch.cuda.synchronize()
    assert d2h_p == d2h
    assert int(packed["accept_len"][0]) == kl and int(packed["accept_node"][0]) == kn
    np.testing.assert_array_equal(packed["argmax"][0].numpy(), am)


@pytest.mark.parametrize("wid,commit", [(2, "checkpoint"), (3, "checkpoint"), (4, "checkpoint"), (2, "replay"),
                                        (2, "wy")])
def test_host_step_graph_equals_eager_host_steps(wid, commit):
    """The whole host step as one graph (copies on two branches, the step,
    the read-back) gives the eager host step's bytes, step after step."""
    from speculative_decode_hybrid_gb300.pipeline import pinned_host_inputs, run_host_step
    wl = W.make_workload(wid, seed=9, layers=2)
    N, B = wl.shape.n_nodes, wl.shape.batch
    host = pinned_host_inputs(wl)

    def outs():
        return {"accept_len": torch.empty(B, dtype=torch.int32).pin_memory(),
                "accept_node": torch.empty(B, dtype=torch.int32).pin_memory(),
                "argmax": torch.empty((B, N), dtype=torch.int32).pin_memory()}

    eager, graph = SpecStep(wl), SpecStep(wl)
    eager.commit = commit
    # the eager side copies each result tensor back, the graph side the one
    # packed result buffer (host_result_buffers)
    out_e, out_g = outs(), graph.host_result_buffers()
    for _ in range(3):  # the capture runs one eager host step first
        run_host_step(eager, host, out_e)
    graph.capture_host_step(host, out_g, commit)
    graph.x.zero_()  # the graph must copy the inputs in itself
    graph.logits.zero_()
    for _ in range(2):
        run_host_step(graph, host, out_g, graph=True)
    torch.cuda.synchronize()
    for name in ("accept_len", "accept_node", "argmax"):
        assert torch.equal(out_e[name], out_g[name]), name
    for name in ("out", "ssm_state", "conv_state"):
        assert torch.equal(getattr(eager, name), getattr(graph, name)), name
    am, kl, kn = oracle.accept_greedy(wl.logits[0], wl.tokens[0], wl.parent[0] if wl.parent is not None else None)
    assert (int(out_g["accept_len"][0]), int(out_g["accept_node"][0])) == (kl, kn)


# ------------------------------------------------------------ replay-commit variant

def test_verify_without_checkpoints_matches_and_writes_none():
    wl = W.make_workload(1, seed=70)
    a = run(wl, restore=False)
    b = SpecStep(wl)
    b.ssm_ckpt.fill_(-7.0)
    b.conv_ckpt.fill_(-7.0)
    b.verify_nockpt()
    torch.cuda.synchronize()
    assert torch.equal(a.out, b.out)
    assert bool((b.ssm_ckpt == -7.0).all()) and bool((b.conv_ckpt == -7.0).all())


@pytest.mark.parametrize("wid,layers", [(1, None), (2, 3), (0, None)])
def test_replay_commit_equals_checkpoint_restore(wid, layers):
    """Replaying the first k tokens from the live state gives, bit for bit,
    the state that restoring checkpoint k gives (k = 0 leaves it alone)."""
    wl = W.make_workload(wid, seed=71, **({} if layers is None else {"layers": layers}))
    ref = run(wl, restore=False)
    T = wl.shape.n_tok
    for k in sorted({0, 1, min(2, T), T // 2, T}):
        st = SpecStep(wl)
        st.accept_len.fill_(k)
        st.commit_replay()
        torch.cuda.synchronize()
        if k == 0:
            want_s = torch.from_numpy(wl.ssm0).cuda()
            want_c = torch.from_numpy(wl.conv0).cuda()
        else:
            want_s = ref.ssm_ckpt[:, :, k - 1]
            want_c = ref.conv_ckpt[:, :, k - 1]
        assert torch.equal(st.ssm_state, want_s), k
        assert torch.equal(st.conv_state, want_c), k
        assert int(st.dev_status.item()) == 0


def test_replay_variant_step_vs_oracle_and_range_flag():
    wl = W.make_workload(2, seed=9, layers=2)
    st = SpecStep(wl)
    st.step_replay()
    torch.cuda.synchronize()
    am, kl, kn = oracle.accept_greedy(wl.logits[0], wl.tokens[0])
    assert int(st.accept_len[0]) == kl == 2
    for y in range(2):
        ck, cc, out = oracle.verify_request(wl, 0, layers=[y])[0]
        assert slice_rel_err(st.ssm_state[0, y].cpu().numpy(), ck[kl - 1], 128 * 128) <= TOL
        np.testing.assert_array_equal(st.conv_state[0, y].cpu().numpy(), cc[kl - 1].astype(np.float32))
        assert slice_rel_err(st.out[0, y].cpu().numpy(), out, 128) <= TOL
    before = st.ssm_state.clone()
    st.accept_len.fill_(wl.shape.n_tok + 3)
    st.dev_status.zero_()
    st.commit_replay()
    torch.cuda.synchronize()
    assert torch.equal(before, st.ssm_state)
    assert int(st.dev_status.item()) & G.GDN_DEV_NODE_RANGE


def test_accept_workspace_shared_across_shapes():
    """One workspace for calls whose counter and key regions overlap (batch
    sizes crossing the 64-request counter block): every call leaves it zero."""
    g = np.random.default_rng(35)
    dev = torch.device("cuda")
    wsb = G.spec_accept_workspace_bytes(300, 17)
    ws = torch.zeros((wsb,), dtype=torch.uint8, device=dev)
    for B in (3, 300, 70, 1, 200):
        N, V = 17, 3000
        logits = g.standard_normal((B, N, V)).astype(np.float32)
        tokens = g.integers(0, V, (B, N)).astype(np.int32)
        lg = torch.from_numpy(logits).to(dev)
        tk = torch.from_numpy(tokens).to(dev)
        am = torch.empty((B, N), dtype=torch.int32, device=dev)
        kl = torch.empty((B,), dtype=torch.int32, device=dev)
        kn = torch.empty((B,), dtype=torch.int32, device=dev)
        G.spec_accept_greedy(B, N, V, lg, tk, None, am, kl, kn, ws, wsb)
        torch.cuda.synchronize()
        assert int(ws.count_nonzero().item()) == 0
        for r in (0, B - 1):
            o = oracle.accept_greedy(logits[r], tokens[r])
            np.testing.assert_array_equal(am[r].cpu().numpy(), o[0])
            assert (int(kl[r]), int(kn[r])) == o[1:]


# ------------------------------------------------------------ chunked (WY) form of the replay variant

WY_NAMES = ["workload0", "workload1", "two_row_blocks_ragged", "min_rows_f32_one_token", "conv_k1",
            "conv_k2", "conv_k8", "ratio1_batch3", "gqa4_dk64_bf16", "wide_dv_four_row_blocks"]


def wy_workload(name, seed):
    if name == "workload0":
        return W.make_workload(0, seed=seed)
    if name == "workload1":
        return W.make_workload(1, seed=seed)
    return W.draw(EDGE_SHAPES[name], seed=seed + zlib.crc32(name.encode()) % 1000)


@pytest.mark.parametrize("name", WY_NAMES)
def test_wy_verify_vs_oracle(name):
    """o of the chunked form against the oracle's token-by-token recurrence,
    and next to the rank-1 kernel's; the live state is left untouched."""
    wl = wy_workload(name, 80)
    s = wl.shape
    st = SpecStep(wl)
    st.verify_wy()
    torch.cuda.synchronize()
    out_wy = st.out.clone()
    assert torch.equal(st.ssm_state.cpu(), torch.from_numpy(wl.ssm0))
    st.verify_nockpt()
    torch.cuda.synchronize()
    for r in range(s.batch):
        refs = oracle.verify_request(wl, r)
        for y, (ck, cc, out) in enumerate(refs):
            e = slice_rel_err(out_wy[r, y].cpu().numpy(), out, s.d_v)
            assert e <= TOL, (name, r, y, e)
            # f32 accuracy in both forms (the tensor-core product runs as 3 x TF32:
            # a single TF32 pass would be off by ~1e-3 relative)
            e2 = slice_rel_err(out_wy[r, y].cpu().numpy(), st.out[r, y].cpu().numpy(), s.d_v)
            assert e2 <= 1e-4, (name, r, y, e2)
    assert int(st.dev_status.item()) == 0


@pytest.mark.parametrize("name", WY_NAMES)
def test_wy_commit_vs_oracle(name):
    """The live state after the chunked commit of k tokens is the oracle's
    checkpoint k-1 (within TOL; the conv state bit for bit); k = 0 leaves
    the request untouched. Requests take different k."""
    wl = wy_workload(name, 81)
    s = wl.shape
    T = s.n_tok
    refs = {r: oracle.verify_request(wl, r) for r in range(s.batch)}
    for k0 in sorted({0, 1, min(2, T), T // 2, T}):
        ks = [(k0 + r) % (T + 1) for r in range(s.batch)]
        st = SpecStep(wl)
        st.accept_len.copy_(torch.tensor(ks, dtype=torch.int32))
        st.commit_wy()
        torch.cuda.synchronize()
        for r, k in enumerate(ks):
            for y in range(s.layers):
                g_s = st.ssm_state[r, y].cpu().numpy()
                g_c = st.conv_state[r, y].cpu().numpy()
                if k == 0:
                    np.testing.assert_array_equal(g_s, wl.ssm0[r, y])
                    np.testing.assert_array_equal(g_c, wl.conv0[r, y])
                    continue
                ck, cc, _ = refs[r][y]
                e = slice_rel_err(g_s, ck[k - 1], s.d_v * s.d_k)
                assert e <= TOL, (name, k, r, y, e)
                if s.conv_k > 1:
                    np.testing.assert_array_equal(g_c, cc[k - 1].astype(np.float32))
        assert int(st.dev_status.item()) == 0


def test_wy_step_vs_oracle_graph_and_range_flag():
    wl = W.make_workload(2, seed=9, layers=2)
    st = SpecStep(wl)
    st.step_wy()
    torch.cuda.synchronize()
    am, kl, kn = oracle.accept_greedy(wl.logits[0], wl.tokens[0])
    assert int(st.accept_len[0]) == kl == 2
    for y in range(2):
        ck, cc, out = oracle.verify_request(wl, 0, layers=[y])[0]
        assert slice_rel_err(st.ssm_state[0, y].cpu().numpy(), ck[kl - 1], 128 * 128) <= TOL
        np.testing.assert_array_equal(st.conv_state[0, y].cpu().numpy(), cc[kl - 1].astype(np.float32))
        assert slice_rel_err(st.out[0, y].cpu().numpy(), out, 128) <= TOL
    # the captured step gives the eager step's bytes
    a, b = SpecStep(wl), SpecStep(wl)
    a.step_wy()
    a.step_wy()
    b.capture("wy")  # one eager step, then the capture
    b.replay()
    torch.cuda.synchronize()
    assert torch.equal(a.ssm_state, b.ssm_state) and torch.equal(a.conv_state, b.conv_state)
    assert torch.equal(a.out, b.out)
    # k out of range: nothing changes, the flag is set
    before = st.ssm_state.clone()
    st.accept_len.fill_(wl.shape.n_tok + 3)
    st.dev_status.zero_()
    st.commit_wy()
    torch.cuda.synchronize()
    assert torch.equal(before, st.ssm_state)
    assert int(st.dev_status.item()) & G.GDN_DEV_NODE_RANGE


def test_wy_rejects_long_spans():
    wl = W.draw(EDGE_SHAPES["max_tokens"], seed=5)
    st = SpecStep(wl)
    with pytest.raises(G.GdnError) as ei:
        st.verify_wy()
    assert ei.value.status == G.GDN_ERR_DIMS
    with pytest.raises(G.GdnError):
        st.commit_wy()


@pytest.mark.parametrize("tree", [False, True])
def test_per_layer_launches_equal_one_launch(tree):
    """One verify launch per layer gives, bit for bit, the all-layers launch.
    12 layers: the all-layers launch has whole 128-row items (16 rows per
    warp); a one-layer launch has 32-row items (4 rows per warp)."""
    wl = W.make_workload(3 if tree else 2, seed=12, layers=12)
    a, b = SpecStep(wl), SpecStep(wl)
    a.verify()
    b.verify_per_layer()
    torch.cuda.synchronize()
    assert torch.equal(a.out, b.out)
    assert torch.equal(a.ssm_ckpt, b.ssm_ckpt) and torch.equal(a.conv_ckpt, b.conv_ckpt)
    assert int(b.dev_status.item()) == 0


@pytest.mark.parametrize("tree", [False, True])
def test_state_ready_flag_per_layer(tree):
    """GDN_VERIFY_STATE_READY (the state, conv taps, conv state and parents
    read before the wait for the previous launch): per-layer launches with
    the flag give the bytes of the same launches without it and match the
    oracle; and three graph replays of the whole step (flagged per-layer
    verify -> accept -> restore, where each restore rewrites the state the
    next replay reads) leave the state of three eager unflagged steps."""
    wl = W.make_workload(3 if tree else 2, seed=21, layers=6)
    a, b = SpecStep(wl), SpecStep(wl)
    a.verify_per_layer(state_ready=False)
    b.verify_per_layer()
    torch.cuda.synchronize()
    assert torch.equal(a.out, b.out)
    assert torch.equal(a.ssm_ckpt, b.ssm_ckpt) and torch.equal(a.conv_ckpt, b.conv_ckpt)
    for y in (0, 3, 5):
        check_layer_vs_oracle(b, wl, 0, y)
    assert int(b.dev_status.item()) == 0

    a2, b2 = SpecStep(wl), SpecStep(wl)
    b2.capture("checkpoint-per-layer")  # runs one eager step first
    for _ in range(2):
        b2.replay()
    for _ in range(3):
        a2.verify_per_layer(state_ready=False)
        a2.accept()
        a2.restore()
    torch.cuda.synchronize()
    if int(a2.accept_node[0]) > 0:  # the state moved: the later steps read restored state
        assert not torch.equal(a2.ssm_state, SpecStep(wl).ssm_state)
    assert torch.equal(a2.ssm_state, b2.ssm_state) and torch.equal(a2.conv_state, b2.conv_state)
    assert torch.equal(a2.ssm_ckpt, b2.ssm_ckpt) and torch.equal(a2.out, b2.out)
    assert int(b2.dev_status.item()) == 0
