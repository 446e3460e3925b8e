"""Pins of the CPU oracle to facts outside itself.

The pages print no worked example, state or logit value, so every pin here is
a closed form, an invariant, a library routine on a special case, or brute
force on tiny inputs. Each is chosen so that a plausible slip in the oracle
(a dropped term, a wrong sign, a transposed operand, a wrong window index,
a wrong tie rule) fails at least one of them.
"""
import itertools

import numpy as np
import pytest
import scipy.signal
import scipy.special

import oracle
from speculative_decode_hybrid_gb300 import workloads as W


def rng(seed):
    return np.random.default_rng(seed)


def unit_rows(g, shape):
    x = g.standard_normal(shape)
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def silu_ref(x):
    return x * scipy.special.expit(x)


# ---------------------------------------------------------------- recurrence

@pytest.mark.parametrize("d_k,d_v,T", [(8, 5, 6), (64, 64, 4), (16, 24, 9)])
def test_b_zero_is_pure_decay(d_k, d_v, T):
    """b = 0: S_t = (prod_{s<=t} a_s) S_0 and o_t = (prod_{s<=t} a_s) S_0 q_t."""
    g = rng(1)
    q, k = unit_rows(g, (T, d_k)), unit_rows(g, (T, d_k))
    v = g.standard_normal((T, d_v))
    a = g.uniform(0.5, 1.0, T)
    S0 = g.standard_normal((d_v, d_k))
    S, o = oracle.delta_rule(q, k, v, a, np.zeros(T), S0)
    decay = np.cumprod(a)
    for t in range(T):
        np.testing.assert_allclose(S[t], decay[t] * S0, rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(o[t], decay[t] * (S0 @ q[t]), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("d_k,d_v,m", [(8, 3, 8), (16, 16, 5), (64, 32, 12)])
def test_unit_gates_orthonormal_keys_store_v(d_k, d_v, m):
    """a = b = 1 with orthonormal keys: S_T k_i = v_i for every i, for any S_0;
    with S_0 = 0, S_T = sum_i v_i k_i^T."""
    g = rng(2)
    Q, _ = np.linalg.qr(g.standard_normal((d_k, d_k)))
    keys = Q[:, :m].T.copy()
    v = g.standard_normal((m, d_v))
    q = unit_rows(g, (m, d_k))
    ones = np.ones(m)
    S0 = g.standard_normal((d_v, d_k))
    S, _ = oracle.delta_rule(q, keys, v, ones, ones, S0)
    for i in range(m):
        np.testing.assert_allclose(S[-1] @ keys[i], v[i], atol=1e-12)
    S, _ = oracle.delta_rule(q, keys, v, ones, ones, np.zeros((d_v, d_k)))
    np.testing.assert_allclose(S[-1], v.T @ keys, atol=1e-12)


def test_orthonormal_keys_general_gates_closed_form():
    """General a, b with orthonormal keys k_1..k_m (m < d_k):
    S_T k_i = (prod_{s>i} a_s) [ (1-b_i) a_i (prod_{s<i} a_s) S_0 k_i + b_i v_i ]
    and S_T x = (prod_s a_s) S_0 x for x orthogonal to every key."""
    d_k, d_v, m = 12, 7, 6
    g = rng(3)
    Q, _ = np.linalg.qr(g.standard_normal((d_k, d_k)))
    keys = Q[:, :m].T.copy()
    x_perp = Q[:, m]
    v = g.standard_normal((m, d_v))
    q = unit_rows(g, (m, d_k))
    a = g.uniform(0.8, 1.0, m)
    b = g.uniform(0.1, 0.9, m)
    S0 = g.standard_normal((d_v, d_k))
    S, _ = oracle.delta_rule(q, keys, v, a, b, S0)
    for i in range(m):
        before = np.prod(a[:i])
        after = np.prod(a[i + 1:])
        want = after * ((1 - b[i]) * a[i] * before * (S0 @ keys[i]) + b[i] * v[i])
        np.testing.assert_allclose(S[-1] @ keys[i], want, atol=1e-12)
    np.testing.assert_allclose(S[-1] @ x_perp, np.prod(a) * (S0 @ x_perp), atol=1e-12)


@pytest.mark.parametrize("d_k,d_v,T", [(5, 3, 6), (4, 7, 3), (9, 9, 5)])
def test_rank1_form_equals_explicit_matrix_form(d_k, d_v, T):
    """The rank-1 update equals S_{t-1} (I - b k k^T) a + b v k^T written with
    explicit d x d matrices (brute force)."""
    g = rng(4)
    q, k = g.standard_normal((T, d_k)), g.standard_normal((T, d_k))
    v = g.standard_normal((T, d_v))
    a, b = g.uniform(0.5, 1.0, T), g.uniform(0.0, 1.0, T)
    S0 = g.standard_normal((d_v, d_k))
    S1, o1 = oracle.delta_rule(q, k, v, a, b, S0)
    S2, o2 = oracle.delta_rule(q, k, v, a, b, S0, explicit=True)
    np.testing.assert_allclose(S1, S2, atol=1e-12)
    np.testing.assert_allclose(o1, o2, atol=1e-12)
    # and the explicit form against numpy matrix products (library routine)
    S = S0.copy()
    for t in range(T):
        M = np.eye(d_k) - b[t] * np.outer(k[t], k[t])
        S = a[t] * (S @ M) + b[t] * np.outer(v[t], k[t])
        np.testing.assert_allclose(S2[t], S, atol=1e-12)
        np.testing.assert_allclose(o2[t], S @ q[t], atol=1e-12)


def test_value_rows_are_independent():
    """Permuting the value rows (v entries and the rows of S_0) permutes S and o."""
    d_k, d_v, T = 6, 9, 5
    g = rng(5)
    q, k = unit_rows(g, (T, d_k)), unit_rows(g, (T, d_k))
    v = g.standard_normal((T, d_v))
    a, b = g.uniform(0.9, 1.0, T), g.uniform(0.0, 1.0, T)
    S0 = g.standard_normal((d_v, d_k))
    perm = g.permutation(d_v)
    S, o = oracle.delta_rule(q, k, v, a, b, S0)
    Sp, op = oracle.delta_rule(q, k, v[:, perm], a, b, S0[perm])
    np.testing.assert_array_equal(Sp, S[:, perm])
    np.testing.assert_array_equal(op, o[:, perm])


# ---------------------------------------------------------------- conv, norm

@pytest.mark.parametrize("K,T", [(4, 10), (2, 3), (1, 4), (5, 7)])
def test_conv_matches_causal_fir(K, T):
    """Pre-activation = causal FIR (scipy.signal.lfilter with the taps reversed)
    over [state, x]; conv state after token t = the last K-1 inputs."""
    g = rng(6)
    w = g.standard_normal(K)
    st = g.standard_normal(K - 1)
    x = g.standard_normal(T)
    y, s_after = oracle.conv1d_silu(w, st, x)
    seq = np.concatenate([st, x])
    pre = scipy.signal.lfilter(w[::-1], [1.0], seq)[K - 1:]
    np.testing.assert_allclose(y, silu_ref(pre), rtol=1e-13, atol=1e-14)
    for t in range(T):
        np.testing.assert_array_equal(s_after[t], seq[t + 1:t + K])


def test_conv_identity_tap_and_delay():
    """w = e_{K-1}: y = SiLU(x). A unit impulse through zero state gives the
    taps back in reverse order, delayed to the impulse (a pure delay line)."""
    K, T = 4, 9
    g = rng(7)
    x = g.standard_normal(T)
    y, _ = oracle.conv1d_silu(np.eye(K)[K - 1], g.standard_normal(K - 1), x)
    np.testing.assert_allclose(y, silu_ref(x), rtol=1e-14)
    w = g.standard_normal(K)
    t0 = 3
    imp = np.zeros(T)
    imp[t0] = 1.0
    y, _ = oracle.conv1d_silu(w, np.zeros(K - 1), imp)
    pre = np.zeros(T)
    for lag in range(K):
        if t0 + lag < T:
            pre[t0 + lag] = w[K - 1 - lag]
    np.testing.assert_allclose(y, silu_ref(pre), rtol=1e-14, atol=1e-15)


def test_l2norm_unit_length():
    g = rng(8)
    for n in (1, 7, 128):
        v = g.standard_normal(n) * 10
        u = oracle.l2norm(v)
        np.testing.assert_allclose(np.linalg.norm(u), 1.0, rtol=1e-7)
        np.testing.assert_allclose(u, v / np.linalg.norm(v), rtol=1e-7)
    np.testing.assert_array_equal(oracle.l2norm(np.zeros(5)), np.zeros(5))


# ---------------------------------------------------------------- layer verify

def _layer_inputs(seed, h_k=2, h_v=4, d_k=8, d_v=6, K=4, T=5):
    g = rng(seed)
    C = 2 * h_k * d_k + h_v * d_v
    return dict(h_k=h_k, h_v=h_v, d_k=d_k, d_v=d_v, K=K,
                x=g.standard_normal((T, C)), a=g.uniform(0.9, 0.999, (T, h_v)),
                b=scipy.special.expit(g.standard_normal((T, h_v))),
                w=g.normal(0, 0.5, (C, K)), ssm_in=g.normal(0, 0.1, (h_v, d_v, d_k)),
                conv_in=g.normal(0, 0.1, (C, K - 1)))


def _run(inp, parent=None, q_scale=1.0, T=None):
    x, a, b = inp["x"], inp["a"], inp["b"]
    if T is not None:
        x, a, b = x[:T], a[:T], b[:T]
    return oracle.verify_layer(inp["h_k"], inp["h_v"], inp["d_k"], inp["d_v"], inp["K"],
                               x, a, b, inp["w"], inp["ssm_in"], inp["conv_in"],
                               parent=parent, q_scale=q_scale)


@pytest.mark.parametrize("q_scale", [1.0, 0.125])
def test_layer_is_fir_norm_and_delta_rule_composed(q_scale):
    """verify_layer == per-channel causal FIR (scipy) -> SiLU -> split
    [q | k | v] -> per-head unit norm (numpy) -> q *= scale -> delta rule per
    value head with key head floor(h H_k / H_v)."""
    inp = _layer_inputs(9)
    h_k, h_v, d_k, d_v, K = (inp[n] for n in ("h_k", "h_v", "d_k", "d_v", "K"))
    T, C = inp["x"].shape
    ck, cc, out = _run(inp, q_scale=q_scale)
    y = np.zeros((T, C))
    for c in range(C):
        seq = np.concatenate([inp["conv_in"][c], inp["x"][:, c]])
        y[:, c] = silu_ref(scipy.signal.lfilter(inp["w"][c][::-1], [1.0], seq)[K - 1:])
        for t in range(T):
            np.testing.assert_array_equal(cc[t, c], seq[t + 1:t + K])
    q = y[:, :h_k * d_k].reshape(T, h_k, d_k)
    k = y[:, h_k * d_k:2 * h_k * d_k].reshape(T, h_k, d_k)
    v = y[:, 2 * h_k * d_k:].reshape(T, h_v, d_v)
    q = q / np.sqrt((q ** 2).sum(-1, keepdims=True) + 1e-6) * q_scale
    k = k / np.sqrt((k ** 2).sum(-1, keepdims=True) + 1e-6)
    for h in range(h_v):
        gk = h * h_k // h_v
        S = inp["ssm_in"][h]
        for t in range(T):
            M = np.eye(d_k) - inp["b"][t, h] * np.outer(k[t, gk], k[t, gk])
            S = inp["a"][t, h] * (S @ M) + inp["b"][t, h] * np.outer(v[t, h], k[t, gk])
            np.testing.assert_allclose(ck[t, h], S, atol=1e-12)
            np.testing.assert_allclose(out[t, h], S @ q[t, gk], atol=1e-12)


def test_restore_at_k_equals_replay_of_first_k():
    """Restoring checkpoint k equals replaying only the first k tokens from the
    initial state (bit-exact within the oracle); k = 0 keeps the initial state."""
    inp = _layer_inputs(10, T=6)
    ck, cc, _ = _run(inp)
    for kk in range(0, 7):
        st = oracle.restore(ck, kk, inp["ssm_in"])
        cst = oracle.restore(cc, kk, inp["conv_in"])
        if kk == 0:
            np.testing.assert_array_equal(st, inp["ssm_in"])
            np.testing.assert_array_equal(cst, inp["conv_in"])
            continue
        ck2, cc2, _ = _run(inp, T=kk)
        np.testing.assert_array_equal(st, ck2[-1])
        np.testing.assert_array_equal(cst, cc2[-1])


def test_tree_that_is_a_chain_equals_chain():
    inp = _layer_inputs(11, T=6)
    a1 = _run(inp)
    a2 = _run(inp, parent=W.chain_parent(7))
    for u, v in zip(a1, a2):
        np.testing.assert_array_equal(u, v)


def test_star_tree_is_independent_single_steps():
    """All nodes children of the root: each node equals a one-token verify of
    its own inputs from the initial state."""
    inp = _layer_inputs(12, T=5)
    par = np.array([-1, 0, 0, 0, 0, 0], dtype=np.int32)
    ck, cc, out = _run(inp, parent=par)
    for i in range(5):
        one = dict(inp, x=inp["x"][i:i + 1], a=inp["a"][i:i + 1], b=inp["b"][i:i + 1])
        c1, cc1, o1 = _run(one)
        np.testing.assert_array_equal(ck[i], c1[0])
        np.testing.assert_array_equal(cc[i], cc1[0])
        np.testing.assert_array_equal(out[i], o1[0])


def test_tree_node_equals_chain_over_its_root_path():
    """Every tree node's checkpoint equals a chain verify over the tokens of
    its root path (bit-exact): state and conv window follow the parents."""
    g = rng(13)
    T = 9
    inp = _layer_inputs(13, T=T)
    par = W.random_tree(g, T + 1, max_depth=16)
    ck, cc, out = _run(inp, parent=par)
    for i in range(1, T + 1):
        path = []
        n = i
        while n > 0:
            path.append(n)
            n = int(par[n])
        path = path[::-1]
        rows = [p - 1 for p in path]
        sub = dict(inp, x=inp["x"][rows], a=inp["a"][rows], b=inp["b"][rows])
        c1, cc1, o1 = _run(sub)
        np.testing.assert_array_equal(ck[i - 1], c1[-1])
        np.testing.assert_array_equal(cc[i - 1], cc1[-1])
        np.testing.assert_array_equal(out[i - 1], o1[-1])


def test_bad_tree_rejected():
    inp = _layer_inputs(14, T=3)
    for par in ([0, 0, 1, 2], [-1, 1, 1, 2], [-1, 0, 3, 1], [-1, 0, -1, 2]):
        with pytest.raises(oracle.OracleError):
            _run(inp, parent=np.array(par, dtype=np.int32))


# ---------------------------------------------------------------- acceptance

def test_argmax_matches_numpy_first_occurrence():
    g = rng(15)
    for _ in range(50):
        V = int(g.integers(1, 40))
        row = g.integers(-3, 4, V).astype(np.float32)   # many ties
        assert oracle.argmax_f32(row) == int(np.argmax(row))
    row = np.array([1.0, np.nan, 3.0, np.nan], dtype=np.float32)
    assert oracle.argmax_f32(row) == int(np.argmax(row)) == 1
    row = np.array([-0.0, 0.0, -1.0], dtype=np.float32)
    assert oracle.argmax_f32(row) == int(np.argmax(row)) == 0
    row = np.array([-np.inf, -np.inf], dtype=np.float32)
    assert oracle.argmax_f32(row) == 0
    big = g.standard_normal(151936).astype(np.float32)
    assert oracle.argmax_f32(big) == int(np.argmax(big))


def _brute_accept(am, tokens, par):
    """Enumerate every node's root path; keep those whose tokens all match the
    argmax of their parent row; longest wins, then the lexicographically
    smallest path of node indices."""
    N = len(tokens)
    best = None
    for n in range(N):
        path = []
        m = n
        while m > 0:
            path.append(m)
            m = int(par[m])
        path = path[::-1]
        prev = 0
        good = True
        for p in path:
            if tokens[p] != am[prev]:
                good = False
                break
            prev = p
        if not good:
            continue
        key = (-len(path), path)
        if best is None or key < best[0]:
            best = (key, n)
    return len(_path_of(best[1], par)), best[1]


def _path_of(n, par):
    out = []
    while n > 0:
        out.append(n)
        n = int(par[n])
    return out


def test_accept_tree_brute_force():
    g = rng(16)
    for trial in range(300):
        N = int(g.integers(1, 9))
        V = int(g.integers(1, 4))        # tiny vocab: many matches and duplicate siblings
        logits = g.integers(0, 3, (N, V)).astype(np.float32)
        tokens = g.integers(0, V, N).astype(np.int32)
        par = W.random_tree(g, N, max_depth=16)
        am, kl, kn = oracle.accept_greedy(logits, tokens, par)
        np.testing.assert_array_equal(am, np.argmax(logits, axis=1))
        assert (kl, kn) == _brute_accept(am, tokens, par), trial


def test_accept_chain_cases():
    g = rng(17)
    L, V = 16, 1000
    logits = g.standard_normal((L + 1, V)).astype(np.float32)
    am = np.argmax(logits, axis=1)
    tokens = np.zeros(L + 1, dtype=np.int32)
    tokens[1:] = am[:-1]
    _, kl, kn = oracle.accept_greedy(logits, tokens)
    assert (kl, kn) == (L, L)
    bad = tokens.copy()
    bad[1] = (am[0] + 1) % V
    _, kl, kn = oracle.accept_greedy(logits, bad)
    assert (kl, kn) == (0, 0)
    for j in range(1, L + 1):
        bad = tokens.copy()
        bad[j] = (am[j - 1] + 1) % V
        _, kl, kn = oracle.accept_greedy(logits, bad)
        assert (kl, kn) == (j - 1, j - 1)
    # out-of-range token ids never match
    bad = tokens.copy()
    bad[3] = V + 5
    assert oracle.accept_greedy(logits, bad)[1] == 2
    # chain given as an explicit parent array gives the same answer
    assert oracle.accept_greedy(logits, tokens, W.chain_parent(L + 1))[1:] == (L, L)


def test_accept_brute_force_all_match_patterns_chain():
    """Every one of the 2^L match patterns of a short chain: k = index of the
    first mismatch."""
    L, V = 6, 50
    g = rng(18)
    logits = g.standard_normal((L + 1, V)).astype(np.float32)
    am = np.argmax(logits, axis=1)
    for bits in itertools.product([0, 1], repeat=L):
        tokens = np.zeros(L + 1, dtype=np.int32)
        for j in range(1, L + 1):
            tokens[j] = am[j - 1] if bits[j - 1] else (am[j - 1] + 1) % V
        k = next((j for j in range(L) if not bits[j]), L)
        assert oracle.accept_greedy(logits, tokens)[1:] == (k, k)


# ---------------------------------------------------------------- golden geometry

from golden_cases import tree_geometry_cases  # noqa: E402


@pytest.mark.parametrize("case", tree_geometry_cases(), ids=lambda c: c[0])
def test_oracle_tree_geometry_golden(case):
    """The oracle accepts exactly the well-formed parent arrays of the fixture
    (tree mode; the chain-only classes are checked on the library side)."""
    name, mode, parent, want = case
    if parent is None or len(parent) == 0:
        return
    rc, _ = oracle.tree_depths(np.array(parent, dtype=np.int32))
    if want in ("ok", "not_chain"):
        assert rc == oracle.ORA_OK, name
    elif want == "truncated":
        # a root alone is a valid tree with nothing to verify
        assert rc == oracle.ORA_OK, name
    else:
        assert rc == oracle.ORA_ERR_TREE, name


# ---------------------------------------------------------------- top-k

def test_topk_matches_stable_argsort():
    """Finite rows: the order of numpy's stable argsort of -x (larger first,
    lower index first among equals)."""
    g = rng(19)
    for trial in range(40):
        V = int(g.integers(1, 300))
        k = int(g.integers(1, min(V, 32) + 1))
        row = g.integers(-4, 5, V).astype(np.float32) if trial % 2 else g.standard_normal(V).astype(np.float32)
        idx, val = oracle.topk_f32(row, k)
        want = np.argsort(-row.astype(np.float64), kind="stable")[:k]
        np.testing.assert_array_equal(idx, want)
        np.testing.assert_array_equal(val, row[want])
    assert oracle.topk_f32(np.array([3.0], dtype=np.float32), 1)[0][0] == 0


def test_topk_nan_and_signed_zero():
    row = np.array([0.0, np.nan, -0.0, 5.0, np.nan, -1.0], dtype=np.float32)
    idx, _ = oracle.topk_f32(row, 6)
    assert list(idx) == [1, 4, 3, 0, 2, 5]
    assert oracle.topk_f32(row, 1)[0][0] == oracle.argmax_f32(row) == 1
