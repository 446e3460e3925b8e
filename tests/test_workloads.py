"""The seeded input generator (CPU): determinism, shapes, bf16 rounding,
planted targets, match rates and tree geometry."""
import numpy as np
import torch

import oracle
from speculative_decode_hybrid_gb300 import workloads as W


def test_deterministic_and_shaped():
    a = W.make_workload(1, seed=5)
    b = W.make_workload(1, seed=5)
    for name in ("x", "a", "b", "conv_w", "ssm0", "conv0", "logits", "tokens"):
        np.testing.assert_array_equal(getattr(a, name), getattr(b, name))
    s = a.shape
    assert a.x.shape == (1, 1, 16, 8192) and a.x.dtype == np.uint16
    assert a.ssm0.shape == (1, 1, 32, 128, 128) and a.ssm0.dtype == np.float32
    assert a.conv0.shape == (1, 1, 8192, 3)
    assert a.logits.shape == (1, 17, 151936) and a.logits.dtype == np.float32
    assert s.conv_ch == 8192 and W.WORKLOADS[0].conv_ch == 512
    c = W.make_workload(1, seed=6)
    assert not np.array_equal(a.ssm0, c.ssm0)


def test_bf16_rounding_matches_torch():
    g = np.random.default_rng(0)
    x = (g.standard_normal(100000) * np.exp(g.uniform(-20, 20, 100000))).astype(np.float32)
    x[:4] = [0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8]   # exact ties round to even
    bits, widened = W.bf16_round(x)
    t = torch.from_numpy(x).to(torch.bfloat16)
    np.testing.assert_array_equal(bits, t.view(torch.int16).numpy().view(np.uint16))
    np.testing.assert_array_equal(widened, t.float().numpy())


def test_value_ranges():
    wl = W.make_workload(1, seed=3)
    s = wl.shape
    assert wl.a_f.min() >= 0.89 and wl.a_f.max() <= 1.0
    assert wl.b_f.min() > 0 and wl.b_f.max() < 1
    assert abs(wl.ssm0.std() - 0.1) < 0.01 and abs(wl.conv0.std() - 0.1) < 0.01
    assert abs(wl.conv_w_f.std() - 0.5) < 0.02
    qf = wl.x_f[0, 0, :, : s.h_k * s.d_k].reshape(16, s.h_k, s.d_k)
    np.testing.assert_allclose(np.linalg.norm(qf, axis=-1), 1.0, rtol=1e-2)


def test_planted_targets_and_match_rate_chain():
    hits = total = 0
    for seed in range(40):
        wl = W.make_workload(1, seed=seed)
        am, _, _ = oracle.accept_greedy(wl.logits[0], wl.tokens[0])
        assert np.all(wl.logits[0, np.arange(17), am] == W.PLANTED_LOGIT)
        hits += int(np.sum(wl.tokens[0, 1:] == am[:-1]))
        total += 16
    assert 0.5 < hits / total < 0.7


def test_tree_geometry_and_distinct_siblings():
    for seed in range(10):
        wl = W.make_workload(3, seed=seed, layers=1)
        par = wl.parent[0]
        rc, depth = oracle.tree_depths(par)
        assert rc == 0 and depth.max() <= 16 and par[0] == -1
        for p in np.unique(par[1:]):
            kids = np.nonzero(par == p)[0]
            assert len(set(wl.tokens[0, kids].tolist())) == len(kids)


def test_acceptance_independent_of_layer_count():
    a = W.make_workload(2, seed=9, layers=1)
    b = W.make_workload(2, seed=9, layers=3)
    np.testing.assert_array_equal(a.logits, b.logits)
    np.testing.assert_array_equal(a.tokens, b.tokens)
    np.testing.assert_array_equal(a.x[:, 0], b.x[:, 0])


def test_batched_requests_independent():
    wl = W.make_workload(4, seed=4, layers=1)
    assert wl.x.shape[0] == 16
    assert np.all((wl.match_p >= 0.3) & (wl.match_p <= 0.7)) and wl.match_p.std() > 0.01
    assert not np.array_equal(wl.ssm0[0], wl.ssm0[1])
    assert wl.conv_w.shape[0] == 1   # weights are per layer, shared by the requests


def test_tiny_workload_uniform_drafts():
    wl = W.make_workload(0, seed=0)
    assert wl.logits.shape == (1, 5, 1024) and wl.x.dtype == np.float32
    assert wl.tokens.min() >= 0 and wl.tokens.max() < 1024
