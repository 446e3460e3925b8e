"""Shared helpers of the GPU parity tests: run a workload through the C ABI,
fetch the results, and compare them with the CPU oracle."""
import numpy as np
import torch

import oracle
from speculative_decode_hybrid_gb300 import build as B
from speculative_decode_hybrid_gb300 import gdnspec as G
from speculative_decode_hybrid_gb300.pipeline import SpecStep

# Max relative error per (request, layer, slot, head) slice, normwise:
# max_i |x_i - r_i| / max_i |r_i|. bf16 inputs, fp32 state and arithmetic.
TOL = 2e-3


def ensure_built():
    B.build()
    G.load()


def slice_rel_err(gpu: np.ndarray, ref: np.ndarray, slice_len: int) -> float:
    g = np.asarray(gpu, dtype=np.float64).reshape(-1, slice_len)
    r = np.asarray(ref, dtype=np.float64).reshape(-1, slice_len)
    num = np.abs(g - r).max(axis=1)
    den = np.abs(r).max(axis=1)
    err = np.where(den > 0, num / np.where(den > 0, den, 1.0), num)
    return float(err.max()) if err.size else 0.0


def run(wl, restore=True, stream=None):
    """Upload, verify -> accept -> restore, synchronise; returns the SpecStep."""
    st = SpecStep(wl)
    st.verify(stream)
    st.accept(stream)
    if restore:
        st.restore(stream)
    torch.cuda.synchronize()
    return st


def check_layer_vs_oracle(st, wl, r, y, ref=None):
    """Compare checkpoints, conv checkpoints and o of (request r, layer y)."""
    s = wl.shape
    if ref is None:
        ref = oracle.verify_request(wl, r, layers=[y])[0]
    ck, cc, out = ref
    g_ck = st.ssm_ckpt[r, y].cpu().numpy()
    g_cc = st.conv_ckpt[r, y].cpu().numpy()
    g_out = st.out[r, y].cpu().numpy()
    e_ck = slice_rel_err(g_ck, ck, s.d_v * s.d_k)
    e_out = slice_rel_err(g_out, out, s.d_v)
    assert e_ck <= TOL, f"ckpt rel err {e_ck:.3e} (r={r}, y={y})"
    assert e_out <= TOL, f"out rel err {e_out:.3e} (r={r}, y={y})"
    if s.conv_k > 1:
        np.testing.assert_array_equal(g_cc, cc.astype(np.float32))
    return e_ck, e_out


def check_accept_vs_oracle(st, wl):
    am = st.argmax.cpu().numpy()
    kl = st.accept_len.cpu().numpy()
    kn = st.accept_node.cpu().numpy()
    for r in range(wl.shape.batch):
        par = wl.parent[r] if wl.parent is not None else None
        o_am, o_kl, o_kn = oracle.accept_greedy(wl.logits[r], wl.tokens[r], par)
        np.testing.assert_array_equal(am[r], o_am)
        assert (int(kl[r]), int(kn[r])) == (o_kl, o_kn), r
    return kl, kn


def check_restore(st, wl, kn, layers=None, ref_layers=None):
    """Restored state == the GPU's own checkpoint slot, bit for bit (or the
    untouched initial state for node 0); and within TOL of the oracle."""
    s = wl.shape
    layers = range(s.layers) if layers is None else layers
    for r in range(s.batch):
        node = int(kn[r])
        for y in layers:
            g_state = st.ssm_state[r, y].cpu().numpy()
            g_conv = st.conv_state[r, y].cpu().numpy()
            if node == 0:
                np.testing.assert_array_equal(g_state, wl.ssm0[r, y])
                np.testing.assert_array_equal(g_conv, wl.conv0[r, y])
            else:
                np.testing.assert_array_equal(g_state, st.ssm_ckpt[r, y, node - 1].cpu().numpy())
                np.testing.assert_array_equal(g_conv, st.conv_ckpt[r, y, node - 1].cpu().numpy())
            if ref_layers is not None and (r, y) in ref_layers:
                ck, cc, _ = ref_layers[(r, y)]
                want = oracle.restore(ck, node, wl.ssm0[r, y])
                assert slice_rel_err(g_state, want, s.d_v * s.d_k) <= TOL
                want_c = oracle.restore(cc, node, wl.conv0[r, y])
                np.testing.assert_array_equal(g_conv, want_c.astype(np.float32))
