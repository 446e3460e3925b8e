"""Cases run against the bounds-checking build of the library.

test_debug_bounds_gpu.py runs this file in a process of its own, with
GDNSPEC_LIB pointing at _lib/libgdnspec_debug.so, whose kernels check every
global access against the extent of its buffer and OR GDN_DEV_BOUNDS into
the call's dev_status word (skipping the access) instead of reading or
writing outside it. Every case below must leave no flag but the ones it
expects, and the results must still match the CPU oracle. Prints
"debug-bounds ok" at the end.
"""
import dataclasses
import os
import sys
import zlib

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)
sys.path.insert(0, os.path.dirname(HERE))

import oracle  # noqa: E402
from gpu_helpers import check_accept_vs_oracle, check_layer_vs_oracle, check_restore  # noqa: E402
from speculative_decode_hybrid_gb300 import gdnspec as G  # noqa: E402
from speculative_decode_hybrid_gb300 import workloads as W  # noqa: E402
from speculative_decode_hybrid_gb300.pipeline import SpecStep  # noqa: E402
from test_parity_gpu import EDGE_SHAPES  # noqa: E402


def status(st):
    return int(st.dev_status.item())


def check_step(wl, what, per_layer=False):
    """verify -> accept -> restore against the oracle on every layer; no flag."""
    st = SpecStep(wl)
    if per_layer:
        st.verify_per_layer()
    else:
        st.verify()
    st.accept()
    st.restore()
    torch.cuda.synchronize()
    s = wl.shape
    refs = {}
    for r in range(s.batch):
        for y, ref in zip(range(s.layers), oracle.verify_request(wl, r)):
            check_layer_vs_oracle(st, wl, r, y, ref)
            refs[(r, y)] = ref
    kl, kn = check_accept_vs_oracle(st, wl)
    check_restore(st, wl, kn, ref_layers=refs)
    assert status(st) == 0, (what, status(st))


def main():
    lib = os.environ.get("GDNSPEC_LIB", "")
    assert lib.endswith("libgdnspec_debug.so") and os.path.exists(lib), lib
    G.load()
    assert torch.cuda.is_available()

    check_step(W.make_workload(0, seed=0), "workload 0")
    check_step(W.make_workload(1, seed=1), "workload 1")
    check_step(W.make_workload(3, seed=3, layers=4), "workload 3, 4 layers")
    check_step(W.make_workload(2, seed=5, layers=4), "per-layer chain", per_layer=True)
    check_step(W.make_workload(3, seed=6, layers=4), "per-layer tree", per_layer=True)
    for name, s in sorted(EDGE_SHAPES.items()):
        check_step(W.draw(s, seed=zlib.crc32(name.encode()) % 1000), "edge " + name)
    for name in ("two_row_blocks_ragged", "max_tokens", "conv_k8", "ratio1_batch3", "vocab_tiny"):
        check_step(W.draw(dataclasses.replace(EDGE_SHAPES[name], tree=True), seed=7 + len(name)), "edge tree " + name)

    # replay commit (rank-1 and chunked) against checkpoint + restore
    wl = W.make_workload(2, seed=7, layers=4)
    a, b, c = SpecStep(wl), SpecStep(wl), SpecStep(wl)
    a.step()
    b.verify_nockpt()
    b.accept()
    b.commit_replay()
    c.verify_wy()
    c.accept()
    c.commit_wy()
    torch.cuda.synchronize()
    assert torch.equal(a.ssm_state, b.ssm_state) and torch.equal(a.conv_state, b.conv_state)
    assert torch.equal(a.conv_state, c.conv_state)
    for st, what in ((a, "step"), (b, "replay"), (c, "wy")):
        assert status(st) == 0, (what, status(st))

    # the pipelined verify calls (flags set up front; batch 16 takes the
    # work-stealing path) and the pipelined end-to-end step graph, whose
    # copies set the flags while the verify runs
    from speculative_decode_hybrid_gb300.pipeline import pinned_host_inputs, run_host_step
    for wid, layers in ((2, 3), (3, 3), (4, 1)):
        wl = W.make_workload(wid, seed=9 + wid, layers=layers)
        a, b = SpecStep(wl), SpecStep(wl)
        a.verify()
        b.x_ready.fill_(1)
        b.verify(x_ready=b.x_ready)
        torch.cuda.synchronize()
        assert torch.equal(a.out, b.out) and torch.equal(a.ssm_ckpt, b.ssm_ckpt), ("pipelined", wid)
        assert status(b) == 0, ("pipelined", wid, status(b))
        if wid == 4:
            continue
        st = SpecStep(wl)
        out = st.host_result_buffers()
        host = pinned_host_inputs(wl)
        st.capture_host_step(host, out, "checkpoint")
        for _ in range(2):
            run_host_step(st, host, out, graph=True)
        torch.cuda.synchronize()
        assert status(st) == 0, ("pipelined host step", wid, status(st))

    # top-k and the no-allocation accept
    g = np.random.default_rng(11)
    for rows, V, k in ((3, 151936, 32), (5, 1001, 7), (1, 64, 1)):
        logits = g.standard_normal((rows, V)).astype(np.float32)
        lg = torch.from_numpy(logits).cuda()
        idx = torch.zeros((rows, k), dtype=torch.int32, device="cuda")
        val = torch.zeros((rows, k), dtype=torch.float32, device="cuda")
        wsb = G.spec_topk_workspace_bytes(rows, k)
        ws = torch.zeros((wsb,), dtype=torch.uint8, device="cuda")
        ds = torch.zeros((1,), dtype=torch.int32, device="cuda")
        G.spec_topk(rows, V, k, lg, idx, val, ws, wsb, ds)
        torch.cuda.synchronize()
        for r in range(rows):
            oi, ov = oracle.topk_f32(logits[r], k)
            np.testing.assert_array_equal(idx[r].cpu().numpy(), oi)
        assert int(ds.item()) == 0, ("topk", int(ds.item()))
    wl = W.make_workload(4, seed=8, layers=1)
    st = SpecStep(wl)
    G.spec_accept_greedy_static(wl.shape.batch, wl.shape.n_nodes, wl.shape.vocab, st.logits, st.tokens, None,
                                st.argmax, st.accept_len, st.accept_node, st.dev_status)
    torch.cuda.synchronize()
    check_accept_vs_oracle(st, wl)
    assert status(st) == 0, ("static accept", status(st))
    print("debug-bounds ok")


if __name__ == "__main__":
    main()
