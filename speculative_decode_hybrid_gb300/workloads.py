"""Seeded synthetic inputs for GDN span verify + greedy acceptance + rollback.

This module only draws random inputs. It holds none of the method's
arithmetic (no conv, no normalisation of the method's q/k, no recurrence,
no argmax): both the CUDA path and the CPU oracle consume the arrays it
returns, byte for byte.

Workloads (no dataset, prompt or trained weight is used; these stand in for
the DFlash/DDTree target verify workloads of the lucebox and openinfer pull
requests, "Sustained performance" and "Benchmark" sections):

  0  tiny chain: 1 layer, 1 request, H_k=2, H_v=4, d=64, 512 channels,
     conv kernel 4, span 4, fp32 inputs, logits [5, 1024], drafts uniform
  1  one Qwen-shaped GDN layer: H_k=16, H_v=32, d=128, 8192 channels,
     span 16, bf16 inputs, fp32 state, logits [17, 151936]
  2  48 layers of workload 1, chain span 16 (the headline)
  3  48 layers, DDTree of 23 nodes (root + 22), depth <= 16, logits [23, V]
  4  16 requests x 48 layers, span 16, per-request match probability

Input recipe (per request, per layer, in draw order; request r of base seed
s draws its layers from the stream [s + r, 1] and its acceptance inputs from
[s + r, 2], so the accepted length does not depend on the layer count; model
weights come from [s, 0x5EED]):
  * pre-conv channels x = [q | k | v]: q, k ~ N(0,1) drawn per key head and
    scaled to unit length per head and token; v ~ N(0,1)
  * b = logistic(N(0,1)), a ~ U(0.9, 0.999), one per value head and token
  * conv weights ~ N(0, 0.25) (variance; std 0.5), per layer, shared by all
    requests (they are model weights)
  * initial S ~ N(0, 0.01) and initial conv state ~ N(0, 0.01) (variances)
  * bf16 workloads round x, a, b and the conv weights to bf16 once, here,
    with round-to-nearest-even; states stay fp32
  * logits ~ N(0,1) fp32. For workloads 1-4 each row n gets a planted target
    id tau_n whose logit is set to 6.0, above any N(0,1) draw with
    overwhelming probability; draft token n+1 (chain) or each child of node n
    (tree) equals tau_n with the match probability, else a uniform id other
    than tau_n. Siblings in a tree get distinct tokens (redrawn).
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

GDN_F32 = 0
GDN_BF16 = 1

QWEN_VOCAB = 151936
PLANTED_LOGIT = 6.0


@dataclasses.dataclass(frozen=True)
class Shape:
    batch: int
    layers: int
    h_k: int
    h_v: int
    d_k: int
    d_v: int
    conv_k: int
    n_nodes: int          # N = processed tokens + 1 (node 0 is the committed root)
    vocab: int
    dtype: int            # GDN_F32 | GDN_BF16 for x, a, b, conv weights
    tree: bool = False
    max_depth: int = 16

    @property
    def conv_ch(self) -> int:
        return 2 * self.h_k * self.d_k + self.h_v * self.d_v

    @property
    def n_tok(self) -> int:
        return self.n_nodes - 1


WORKLOADS = {
    0: Shape(batch=1, layers=1, h_k=2, h_v=4, d_k=64, d_v=64, conv_k=4,
             n_nodes=5, vocab=1024, dtype=GDN_F32),
    1: Shape(batch=1, layers=1, h_k=16, h_v=32, d_k=128, d_v=128, conv_k=4,
             n_nodes=17, vocab=QWEN_VOCAB, dtype=GDN_BF16),
    2: Shape(batch=1, layers=48, h_k=16, h_v=32, d_k=128, d_v=128, conv_k=4,
             n_nodes=17, vocab=QWEN_VOCAB, dtype=GDN_BF16),
    3: Shape(batch=1, layers=48, h_k=16, h_v=32, d_k=128, d_v=128, conv_k=4,
             n_nodes=23, vocab=QWEN_VOCAB, dtype=GDN_BF16, tree=True),
    4: Shape(batch=16, layers=48, h_k=16, h_v=32, d_k=128, d_v=128, conv_k=4,
             n_nodes=17, vocab=QWEN_VOCAB, dtype=GDN_BF16),
}

WORKLOAD_NAMES = {
    0: "tiny chain (1 layer, H_k=2, H_v=4, d=64, span 4, fp32)",
    1: "1 GDN layer, H_k=16, H_v=32, d=128, span 16, bf16 in / fp32 state",
    2: "48 GDN layers, H_k=16, H_v=32, d=128, chain span 16, batch 1",
    3: "48 GDN layers, DDTree 23 nodes (depth<=16), batch 1",
    4: "16 requests x 48 GDN layers, chain span 16",
}


def bf16_round(x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Round fp32 values to bf16 (round to nearest, ties to even).

    Returns (bits as uint16, the exact bf16 values widened to fp32)."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    rounded = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    widened = (rounded.astype(np.uint32) << 16).view(np.float32)
    return rounded, widened


def _unit_rows(rng: np.random.Generator, shape) -> np.ndarray:
    g = rng.standard_normal(shape)
    return g / np.linalg.norm(g, axis=-1, keepdims=True)


def random_tree(rng: np.random.Generator, n_nodes: int, max_depth: int) -> np.ndarray:
    """Parent array: node 0 is the root (parent -1); parent[i] ~ U[0, i),
    redrawn until depth(i) <= max_depth."""
    parent = np.full(n_nodes, -1, dtype=np.int32)
    depth = np.zeros(n_nodes, dtype=np.int64)
    for i in range(1, n_nodes):
        while True:
            p = int(rng.integers(0, i))
            if depth[p] + 1 <= max_depth:
                break
        parent[i] = p
        depth[i] = depth[p] + 1
    return parent


def _other_id(rng: np.random.Generator, vocab: int, avoid) -> int:
    avoid = set(int(t) for t in avoid)
    if len(avoid) >= vocab:          # tiny vocabularies: nothing left to avoid
        return int(rng.integers(0, vocab))
    while True:
        t = int(rng.integers(0, vocab))
        if t not in avoid:
            return t


@dataclasses.dataclass
class Workload:
    shape: Shape
    seed: int
    # device-ready arrays (dtype per shape.dtype for x/a/b/conv_w)
    x: np.ndarray          # [B][Y][T][C]   uint16 (bf16 bits) or float32
    a: np.ndarray          # [B][Y][T][H_v]
    b: np.ndarray          # [B][Y][T][H_v]
    conv_w: np.ndarray     # [Y][C][K]
    # the same values as float32 (exact)
    x_f: np.ndarray
    a_f: np.ndarray
    b_f: np.ndarray
    conv_w_f: np.ndarray
    ssm0: np.ndarray       # [B][Y][H_v][d_v][d_k] float32
    conv0: np.ndarray      # [B][Y][C][K-1]        float32
    logits: np.ndarray     # [B][N][V] float32
    tokens: np.ndarray     # [B][N] int32 (tokens[:, 0] is the committed root token)
    parent: Optional[np.ndarray]  # [B][N] int32 for trees, else None
    match_p: np.ndarray    # [B] per-request match probability used


def _draw_request(rng: np.random.Generator, s: Shape):
    T, Y = s.n_tok, s.layers
    xs, as_, bs, ss, cs = [], [], [], [], []
    for _ in range(Y):
        q = _unit_rows(rng, (T, s.h_k, s.d_k)).reshape(T, -1)
        k = _unit_rows(rng, (T, s.h_k, s.d_k)).reshape(T, -1)
        v = rng.standard_normal((T, s.h_v * s.d_v))
        xs.append(np.concatenate([q, k, v], axis=1))
        bs.append(1.0 / (1.0 + np.exp(-rng.standard_normal((T, s.h_v)))))
        as_.append(rng.uniform(0.9, 0.999, size=(T, s.h_v)))
        ss.append(rng.normal(0.0, 0.1, size=(s.h_v, s.d_v, s.d_k)))
        cs.append(rng.normal(0.0, 0.1, size=(s.conv_ch, s.conv_k - 1)))
    return (np.stack(xs), np.stack(as_), np.stack(bs),
            np.stack(ss).astype(np.float32), np.stack(cs).astype(np.float32))


def _draw_acceptance(rng: np.random.Generator, s: Shape, p: float, planted: bool):
    N, V = s.n_nodes, s.vocab
    logits = rng.standard_normal((N, V), dtype=np.float32)
    if not planted:
        tokens = rng.integers(0, V, size=N).astype(np.int32)
        parent = random_tree(rng, N, s.max_depth) if s.tree else None
        return logits, tokens, parent
    tau = rng.integers(0, V, size=N)
    logits[np.arange(N), tau] = PLANTED_LOGIT
    tokens = np.zeros(N, dtype=np.int32)
    tokens[0] = int(rng.integers(0, V))
    if s.tree:
        parent = random_tree(rng, N, s.max_depth)
        children: dict[int, list[int]] = {}
        for i in range(1, N):
            pi = int(parent[i])
            used = [tokens[c] for c in children.get(pi, [])]
            want = int(tau[pi])
            if rng.random() < p and want not in used:
                t = want
            else:
                t = _other_id(rng, V, used + [want])
            tokens[i] = t
            children.setdefault(pi, []).append(i)
    else:
        parent = None
        for i in range(1, N):
            want = int(tau[i - 1])
            tokens[i] = want if rng.random() < p else _other_id(rng, V, [want])
    return logits, tokens, parent


def make_workload(wid: int, seed: int = 0, *, layers: Optional[int] = None,
                  batch: Optional[int] = None, n_nodes: Optional[int] = None,
                  vocab: Optional[int] = None) -> Workload:
    """Draw workload `wid` (0-4) with the given base seed.

    `layers`, `batch`, `n_nodes` and `vocab` override the workload's sizes
    (used for reduced parity cases); the distributions stay the same."""
    s = WORKLOADS[wid]
    repl = {}
    if layers is not None:
        repl["layers"] = layers
    if batch is not None:
        repl["batch"] = batch
    if n_nodes is not None:
        repl["n_nodes"] = n_nodes
    if vocab is not None:
        repl["vocab"] = vocab
    if repl:
        s = dataclasses.replace(s, **repl)
    return draw(s, seed, planted=(wid != 0), per_request_p=(wid == 4))


def draw(s: Shape, seed: int, *, planted: bool = True,
         per_request_p: bool = False, p: float = 0.6) -> Workload:
    wrng = np.random.default_rng([seed, 0x5EED])
    conv_w = wrng.normal(0.0, 0.5, size=(s.layers, s.conv_ch, s.conv_k))
    X, A, Bg, S0, C0, L, TK, P, MP = [], [], [], [], [], [], [], [], []
    for r in range(s.batch):
        # separate streams: the acceptance draw does not depend on the layer count
        rng = np.random.default_rng([seed + r, 1])
        arng = np.random.default_rng([seed + r, 2])
        pr = float(arng.uniform(0.3, 0.7)) if per_request_p else p
        x, a, b, s0, c0 = _draw_request(rng, s)
        lg, tk, par = _draw_acceptance(arng, s, pr, planted)
        X.append(x); A.append(a); Bg.append(b); S0.append(s0); C0.append(c0)
        L.append(lg); TK.append(tk); P.append(par); MP.append(pr)
    x = np.stack(X).astype(np.float32)
    a = np.stack(A).astype(np.float32)
    b = np.stack(Bg).astype(np.float32)
    w = conv_w.astype(np.float32)
    if s.dtype == GDN_BF16:
        xd, x = bf16_round(x)
        ad, a = bf16_round(a)
        bd, b = bf16_round(b)
        wd, w = bf16_round(w)
    else:
        xd, ad, bd, wd = x, a, b, w
    parent = np.stack(P).astype(np.int32) if s.tree else None
    return Workload(shape=s, seed=seed, x=xd, a=ad, b=bd, conv_w=wd,
                    x_f=x, a_f=a, b_f=b, conv_w_f=w,
                    ssm0=np.stack(S0), conv0=np.stack(C0),
                    logits=np.stack(L), tokens=np.stack(TK), parent=parent,
                    match_p=np.asarray(MP))


def chain_parent(n_nodes: int) -> np.ndarray:
    """The parent array of a chain: parent[0] = -1, parent[i] = i - 1."""
    p = np.arange(-1, n_nodes - 1, dtype=np.int32)
    return p
