"""One speculative step on the device: verify -> greedy accept -> restore.

`SpecStep` owns the device buffers of a workload (all in HBM, allocated once
through PyTorch) and queues the three C-ABI calls on one stream with no host
synchronisation in between: the accepted node travels from
spec_accept_greedy to gdn_rollback_restore in device memory.
`run_host_step` is the end-to-end form of the same step: inputs come from
pinned host memory and the accepted length / node / bonus token go back to
the host.
"""
from __future__ import annotations

import numpy as np
import torch

from . import gdnspec as G
from .workloads import GDN_BF16, Workload


def _dev(a: np.ndarray, device, dtype=None) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.to(device)


class SpecStep:
    """Device-resident buffers and launches for one workload."""

    def __init__(self, wl: Workload, device="cuda", q_scale: float = 1.0):
        s = wl.shape
        self.wl = wl
        self.shape = s
        self.device = torch.device(device)
        self.tree = wl.parent is not None
        self.dims = G.make_dims(s.batch, s.layers, s.h_k, s.h_v, s.d_k, s.d_v, s.conv_k,
                                s.dtype, q_scale=q_scale)
        self.n_nodes = s.n_nodes
        self.n_tok = s.n_tok
        in_dt = torch.bfloat16 if s.dtype == GDN_BF16 else torch.float32
        dev = self.device
        self.x = _dev(wl.x, dev, in_dt if s.dtype == GDN_BF16 else None)
        self.a = _dev(wl.a, dev, in_dt if s.dtype == GDN_BF16 else None)
        self.b = _dev(wl.b, dev, in_dt if s.dtype == GDN_BF16 else None)
        self.conv_w = _dev(wl.conv_w, dev, in_dt if s.dtype == GDN_BF16 else None)
        self.ssm_state = _dev(wl.ssm0, dev)
        self.conv_state = _dev(wl.conv0, dev)
        B, Y, T = s.batch, s.layers, s.n_tok
        self.ssm_ckpt = torch.empty((B, Y, T, s.h_v, s.d_v, s.d_k), dtype=torch.float32, device=dev)
        self.conv_ckpt = torch.empty((B, Y, T, s.conv_ch, s.conv_k - 1), dtype=torch.float32, device=dev)
        self.out = torch.empty((B, Y, T, s.h_v, s.d_v), dtype=torch.float32, device=dev)
        self.logits = _dev(wl.logits, dev)
        self.tokens = _dev(wl.tokens, dev)
        self.parent_host = wl.parent
        self.parent = _dev(wl.parent, dev) if self.tree else None
        # the step's result, one buffer [accept_len (B) | accept_node (B) |
        # argmax (B x nodes)] so that it goes back to the host in one copy
        self.result = torch.zeros((2 * B + B * s.n_nodes,), dtype=torch.int32, device=dev)
        self.accept_len = self.result[:B]
        self.accept_node = self.result[B:2 * B]
        self.argmax = self.result[2 * B:].view(B, s.n_nodes)
        # inputs landing during the verify (the pipelined host step): x_ready[b][y]
        # != 0 once the x, a, b rows of (b, y) are on the device, set from the
        # pinned ones by the copy that follows those rows
        self.x_ready = torch.zeros((B, Y), dtype=torch.int32, device=dev)
        self._ones = torch.ones((B * Y,), dtype=torch.int32).pin_memory()
        self.ws_bytes = G.spec_accept_workspace_bytes(B, s.n_nodes)
        self.workspace = torch.zeros((self.ws_bytes,), dtype=torch.uint8, device=dev)
        self.dev_status = torch.zeros((1,), dtype=torch.int32, device=dev)

    # -- the three calls -------------------------------------------------
    def verify(self, stream=None, x_ready=None):
        """The verify of all requests and layers as one launch; x_ready (device
        int32 [B][Y]): inputs that land during it (the _pipelined calls)."""
        if self.tree:
            G.gdn_tree_verify(self.dims, self.n_nodes, self.parent_host, self.parent, self.x, self.a,
                              self.b, self.conv_w, self.ssm_state, self.conv_state, self.ssm_ckpt,
                              self.conv_ckpt, self.out, self.dev_status, stream, x_ready=x_ready)
        else:
            G.gdn_verify_span(self.dims, self.n_tok, self.x, self.a, self.b, self.conv_w,
                              self.ssm_state, self.conv_state, self.ssm_ckpt, self.conv_ckpt,
                              self.out, self.dev_status, stream, x_ready=x_ready)

    def accept(self, stream=None):
        s = self.shape
        G.spec_accept_greedy(s.batch, s.n_nodes, s.vocab, self.logits, self.tokens, self.parent,
                             self.argmax, self.accept_len, self.accept_node, self.workspace,
                             self.ws_bytes, self.dev_status, stream)

    def restore(self, stream=None):
        G.gdn_rollback_restore(self.dims, self.n_tok, self.accept_node, self.ssm_ckpt, self.conv_ckpt,
                               self.ssm_state, self.conv_state, self.dev_status, stream)

    def step(self, stream=None):
        self.verify(stream)
        self.accept(stream)
        self.restore(stream)

    LAUNCHES_PER_STEP = 3

    # -- the replay-commit variant (chains): no checkpoints, re-run k tokens --
    def verify_nockpt(self, stream=None):
        G.gdn_verify_span_nockpt(self.dims, self.n_tok, self.x, self.a, self.b, self.conv_w,
                                 self.ssm_state, self.conv_state, self.out, self.dev_status, stream)

    def commit_replay(self, stream=None):
        G.gdn_commit_replay(self.dims, self.n_tok, self.accept_len, self.x, self.a, self.b, self.conv_w,
                            self.ssm_state, self.conv_state, self.dev_status, stream)

    def verify_nockpt_fastest(self, stream=None):
        """The faster of the two checkpoint-free verifies: the chunked form
        (tensor-core product) for spans it takes, else the rank-1 kernel.
        Their o agree to f32 rounding, and the state they leave is the same
        (neither writes it)."""
        if self.n_tok <= G.GDN_WY_MAX_TOKENS:
            self.verify_wy(stream)
        else:
            self.verify_nockpt(stream)

    def step_replay(self, stream=None):
        """verify (no checkpoints) -> accept -> replay the accepted tokens
        (rank-1, from the live state)."""
        self.verify_nockpt_fastest(stream)
        self.accept(stream)
        self.commit_replay(stream)

    LAUNCHES_PER_STEP_REPLAY = 4

    # -- the same variant in chunked (WY) form --------------------------------
    def verify_wy(self, stream=None):
        G.gdn_verify_span_wy(self.dims, self.n_tok, self.x, self.a, self.b, self.conv_w,
                             self.ssm_state, self.conv_state, self.out, self.dev_status, stream)

    def commit_wy(self, stream=None):
        G.gdn_commit_wy(self.dims, self.n_tok, self.accept_len, self.x, self.a, self.b, self.conv_w,
                        self.ssm_state, self.conv_state, self.dev_status, stream)

    def step_wy(self, stream=None):
        """verify (chunked form, no checkpoints) -> accept -> commit the
        accepted prefix in closed form."""
        self.verify_wy(stream)
        self.accept(stream)
        self.commit_wy(stream)

    LAUNCHES_PER_STEP_WY = 4

    # -- verify over a block of requests x layers (contiguous slices) ------
    def _dims_of(self, nb: int, ny: int):
        cache = self.__dict__.setdefault("_sub_dims", {})
        if (nb, ny) not in cache:
            s = self.shape
            cache[(nb, ny)] = G.make_dims(nb, ny, s.h_k, s.h_v, s.d_k, s.d_v, s.conv_k, s.dtype,
                                          q_scale=self.dims.q_scale)
        return cache[(nb, ny)]

    def verify_block(self, b0: int, b1: int, y0: int, y1: int, kind: str = "checkpoint", stream=None,
                     flags: int = 0):
        """The verify of requests [b0, b1) x layers [y0, y1) as one launch.
        The slices of the [B][Y] layouts must be contiguous: all layers, or
        one request. kind: "checkpoint", "replay" (no checkpoints: the
        faster form, as verify_nockpt_fastest) or "wy" (no checkpoints,
        chunked form). flags: GDN_VERIFY_* of the checkpoint verify."""
        s = self.shape
        if not (y0 == 0 and y1 == s.layers) and b1 - b0 != 1:
            raise ValueError("a layer range is contiguous for one request only")
        d = self._dims_of(b1 - b0, y1 - y0)
        bs, ys = slice(b0, b1), slice(y0, y1)
        x, a, b = self.x[bs, ys], self.a[bs, ys], self.b[bs, ys]
        w, S, Cs = self.conv_w[ys], self.ssm_state[bs, ys], self.conv_state[bs, ys]
        if not all(t.is_contiguous() for t in (x, a, b, w, S, Cs)):
            raise ValueError("verify_block needs contiguous slices")
        if kind == "checkpoint":
            if self.tree:
                G.gdn_tree_verify(d, self.n_nodes, self.parent_host[bs], self.parent[bs], x, a, b, w, S, Cs,
                                  self.ssm_ckpt[bs, ys], self.conv_ckpt[bs, ys], self.out[bs, ys],
                                  self.dev_status, stream, flags=flags)
            else:
                G.gdn_verify_span(d, self.n_tok, x, a, b, w, S, Cs, self.ssm_ckpt[bs, ys],
                                  self.conv_ckpt[bs, ys], self.out[bs, ys], self.dev_status, stream,
                                  flags=flags)
        elif kind == "replay" and self.n_tok > G.GDN_WY_MAX_TOKENS:
            G.gdn_verify_span_nockpt(d, self.n_tok, x, a, b, w, S, Cs, self.out[bs, ys], self.dev_status, stream)
        else:
            G.gdn_verify_span_wy(d, self.n_tok, x, a, b, w, S, Cs, self.out[bs, ys], self.dev_status, stream)

    def blocks(self, n=4):
        """Contiguous (b0, b1, y0, y1) blocks covering every request and
        layer, in item order: layer ranges for one request, request ranges
        otherwise. n: a number of (nearly) equal blocks, or a list of
        relative block sizes (e.g. [1, 3, 8]: small first, growing)."""
        B, Y = self.shape.batch, self.shape.layers
        total = Y if B == 1 else B
        if isinstance(n, int):
            n = max(1, min(n, total))
            cuts = [k * total // n for k in range(n + 1)]
        else:
            w = [float(v) for v in n]
            acc, cuts = 0.0, [0]
            for v in w:
                acc += v
                cuts.append(int(round(acc / sum(w) * total)))
            cuts = sorted(set(min(total, max(0, c)) for c in cuts) | {0, total})
        spans = [(a, b) for a, b in zip(cuts[:-1], cuts[1:]) if b > a]
        if B == 1:
            return [(0, 1, a, b) for a, b in spans]
        return [(a, b, 0, Y) for a, b in spans]

    # -- per-layer launches: how a model whose layers run in sequence calls it
    def verify_per_layer(self, stream=None, state_ready: bool = True):
        """The verify of each layer as its own launch (batch 1, where a
        layer's slices of the [B][Y] layouts are contiguous). Every launch
        after the first follows the previous layer's verify, which writes
        none of its state, conv taps or parents, so it carries
        GDN_VERIFY_STATE_READY (state_ready=False: no flags). The first one
        follows whatever came before (a restore writes the live state)."""
        if self.shape.batch != 1:
            raise ValueError("per-layer launches are laid out for batch 1")
        for y in range(self.shape.layers):
            fl = G.GDN_VERIFY_STATE_READY if state_ready and y > 0 else 0
            self.verify_block(0, 1, y, y + 1, "checkpoint", stream, flags=fl)

    def step_per_layer(self, stream=None):
        """verify (one launch per layer) -> accept -> restore (all layers)."""
        self.verify_per_layer(stream)
        self.accept(stream)
        self.restore(stream)

    COMMITS = ("checkpoint", "replay", "wy")

    def step_fn(self, commit: str = "checkpoint"):
        """The step of a commit variant: "checkpoint" (verify with per-token
        checkpoints -> accept -> restore), "replay" (rank-1 verify without
        checkpoints -> accept -> replay of the accepted tokens) or "wy" (the
        replay variant in chunked form)."""
        return {"checkpoint": self.step, "replay": self.step_replay, "wy": self.step_wy,
                "checkpoint-per-layer": self.step_per_layer}[commit]

    def replay_bytes(self, accept_len: np.ndarray) -> int:
        """Algorithmic bytes of one replay-variant step (either form): the
        verify reads the state and inputs and writes o; the commit reads and
        writes the state of every request with k > 0 and reads its k tokens'
        inputs."""
        s = self.shape
        el = 2 if s.dtype == GDN_BF16 else 4
        T, C, K = s.n_tok, s.conv_ch, s.conv_k
        state = s.h_v * s.d_v * s.d_k * 4 + C * (K - 1) * 4
        verify = s.batch * s.layers * (state + T * C * el + 2 * T * s.h_v * el + T * s.h_v * s.d_v * 4) \
            + s.layers * C * K * el
        rep = 0
        for k in np.asarray(accept_len).tolist():
            if k > 0:
                rep += s.layers * (2 * state + k * C * el + 2 * k * s.h_v * el + C * K * el)
        return verify + self.accept_bytes() + rep

    # -- the same step as one CUDA graph ------------------------------------
    def capture(self, commit: str = "checkpoint"):
        """Capture the step of a commit variant (see step_fn) into a CUDA
        graph over this object's fixed buffers and shapes, so that a step is
        one graph launch (no per-kernel launch gaps). One eager step runs
        first, outside the capture, so that every kernel attribute is already
        set."""
        fn = self.step_fn(commit)
        fn()
        torch.cuda.synchronize(self.device)
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream(device=self.device)
        s.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.graph(g, stream=s):
            fn(stream=s)
        torch.cuda.current_stream(self.device).wait_stream(s)
        self._graph = g
        return g

    def replay(self):
        """One captured step on the current stream (capture() first)."""
        self._graph.replay()

    def host_result_buffers(self) -> dict:
        """Pinned host buffers for the step's result, laid out like the device
        result buffer: "accept_len", "accept_node" and "argmax" are views of
        "_packed", which run_host_step and capture_host_step copy back in one
        piece (a dict without "_packed" gets one copy per tensor)."""
        packed = torch.empty(self.result.shape, dtype=torch.int32).pin_memory()
        B = self.accept_len.numel()
        return {"_packed": packed, "accept_len": packed[:B], "accept_node": packed[B:2 * B],
                "argmax": packed[2 * B:].view(self.argmax.shape)}

    def _copy_result(self, out_host: dict):
        if "_packed" in out_host:
            out_host["_packed"].copy_(self.result, non_blocking=True)
        else:
            for name in ("accept_len", "accept_node", "argmax"):
                out_host[name].copy_(getattr(self, name), non_blocking=True)

    def capture_host_step(self, host: dict, out_host: dict, commit: str = "checkpoint", chunks=None,
                          pipelined=None):
        """Capture the end-to-end step for fixed pinned host buffers (see
        run_host_step) into one CUDA graph that pipelines the host link with
        the verify. A copy branch DMAs x, a, b in contiguous blocks in item
        order (blocks(chunks): layer ranges for one request, request ranges
        otherwise), then logits and tokens. Then:
        - pipelined (the checkpoint commit; the default there): one verify
          launch starts at once on the main branch (gdn_*_verify_pipelined);
          after each block the copy branch sets that block's flags in x_ready
          (a host-to-device copy of ones, queued behind the block's rows), and
          the kernel waits for an item's flag before it reads the item's x,
          a, b. A tree's parent array is copied first and the verify waits for
          it. Default blocks 1 : 1 : 2 : 4 : 8 : 8 (48 layers: 2, 2, 4, 8, 16,
          16): small first blocks for the verify's first items, larger ones
          once the copies run ahead of it. x_ready is zeroed after the step;
        - otherwise (the replay commits, whose kernels take no flags): the
          verify of each block is its own launch on its own branch, which
          starts when its block has landed (the blocks' layers and requests
          are independent); default blocks 1 : 3 : 8 (48 layers: 4, 12, 32;
          this beat 4 equal blocks by 2-4 %, 2 and 5 blocks too).
        All branches join before the acceptance; then come the commit
        (restore or replay) and the D2H copy of the result. One eager host
        step runs first, outside the capture."""
        finish = {"checkpoint": self.restore, "replay": self.commit_replay, "wy": self.commit_wy}[commit]
        if pipelined is None:
            pipelined = commit == "checkpoint"
        if pipelined and commit != "checkpoint":
            raise ValueError("the pipelined host step is for the checkpoint commit")
        if chunks is None:
            chunks = (1, 1, 2, 4, 8, 8) if pipelined else (1, 3, 8)
        saved = getattr(self, "commit", "checkpoint")
        self.commit = commit
        run_host_step(self, host, out_host)
        self.commit = saved
        torch.cuda.synchronize(self.device)
        blocks = self.blocks(chunks)
        g = torch.cuda.CUDAGraph()
        main = torch.cuda.Stream(device=self.device)
        copy = torch.cuda.Stream(device=self.device)
        main.wait_stream(torch.cuda.current_stream(self.device))
        if pipelined:
            Y = self.shape.layers
            flat = self.x_ready.view(-1)
            with torch.cuda.graph(g, stream=main):
                fork = torch.cuda.Event()
                fork.record(main)
                copy.wait_event(fork)
                parent_done = None
                with torch.cuda.stream(copy):
                    if self.tree and "parent" in host:
                        self.parent.copy_(host["parent"], non_blocking=True)
                        parent_done = torch.cuda.Event()
                        parent_done.record(copy)
                    for b0, b1, y0, y1 in blocks:
                        for name in ("x", "a", "b"):
                            getattr(self, name)[b0:b1, y0:y1].copy_(host[name][b0:b1, y0:y1], non_blocking=True)
                        i0, i1 = b0 * Y + y0, (b1 - 1) * Y + y1  # the block's (request, layer) items
                        flat[i0:i1].copy_(self._ones[i0:i1], non_blocking=True)
                    for name in ("logits", "tokens"):
                        if name in host:
                            getattr(self, name).copy_(host[name], non_blocking=True)
                copied = torch.cuda.Event()
                copied.record(copy)
                if parent_done is not None:
                    main.wait_event(parent_done)
                self.verify(stream=main, x_ready=self.x_ready)
                main.wait_event(copied)
                self.accept(stream=main)
                finish(stream=main)
                self.x_ready.zero_()  # for the next step's copies
                self._copy_result(out_host)
            torch.cuda.current_stream(self.device).wait_stream(main)
            self._graph_host = g
            self._graph_host_bufs = (host, out_host)
            return g
        branches = [torch.cuda.Stream(device=self.device) for _ in blocks]
        with torch.cuda.graph(g, stream=main):
            fork = torch.cuda.Event()
            fork.record(main)
            copy.wait_event(fork)
            landed = []
            with torch.cuda.stream(copy):
                if "parent" in host:  # first: every block's tree verify reads it
                    self.parent.copy_(host["parent"], non_blocking=True)
                for b0, b1, y0, y1 in blocks:
                    for name in ("x", "a", "b"):
                        getattr(self, name)[b0:b1, y0:y1].copy_(host[name][b0:b1, y0:y1], non_blocking=True)
                    e = torch.cuda.Event()
                    e.record(copy)
                    landed.append(e)
                for name in ("logits", "tokens"):
                    if name in host:
                        getattr(self, name).copy_(host[name], non_blocking=True)
            copied = torch.cuda.Event()
            copied.record(copy)
            done = []
            for (b0, b1, y0, y1), e, br in zip(blocks, landed, branches):
                br.wait_event(e)
                self.verify_block(b0, b1, y0, y1, commit, stream=br)
                d = torch.cuda.Event()
                d.record(br)
                done.append(d)
            for d in done:
                main.wait_event(d)
            main.wait_event(copied)
            self.accept(stream=main)
            finish(stream=main)
            self._copy_result(out_host)
        torch.cuda.current_stream(self.device).wait_stream(main)
        self._graph_host = g
        self._graph_host_bufs = (host, out_host)
        return g

    # -- algorithmic bytes -------------------------------------------------
    def verify_bytes(self) -> int:
        """Bytes the verify must move: S and conv state read once, every
        checkpoint written once, inputs read once, o written once."""
        s = self.shape
        T, C, K = s.n_tok, s.conv_ch, s.conv_k
        el = 2 if s.dtype == GDN_BF16 else 4
        per = (s.h_v * s.d_v * s.d_k * 4 + C * (K - 1) * 4            # state read
               + T * (s.h_v * s.d_v * s.d_k * 4 + C * (K - 1) * 4)    # checkpoints
               + T * C * el + 2 * T * s.h_v * el                      # x, a, b
               + T * s.h_v * s.d_v * 4)                               # o
        weights = s.layers * C * K * el
        return s.batch * s.layers * per + weights

    def slot_bytes(self) -> int:
        s = self.shape
        return s.h_v * s.d_v * s.d_k * 4 + s.conv_ch * (s.conv_k - 1) * 4

    def restore_bytes(self, accept_node: np.ndarray) -> int:
        """Read + write of one slot per (request, layer) whose node > 0."""
        moved = int(np.count_nonzero(np.asarray(accept_node) > 0))
        return 2 * self.slot_bytes() * self.shape.layers * moved

    def accept_bytes(self) -> int:
        s = self.shape
        return s.batch * s.n_nodes * (s.vocab * 4 + 4 + 4) + 8 * s.batch

    def units(self) -> int:
        """Verified tokens x layers (nodes x layers for trees) per step."""
        s = self.shape
        return s.batch * s.n_tok * s.layers


def pinned_host_inputs(wl: Workload):
    """The per-step inputs (x, a, b, logits, tokens[, parent]) in pinned host memory."""
    s = wl.shape
    in_dt = torch.bfloat16 if s.dtype == GDN_BF16 else None

    def pin(a, dt=None):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if dt is not None:
            t = t.view(dt)
        return t.pin_memory()

    d = dict(x=pin(wl.x, in_dt), a=pin(wl.a, in_dt), b=pin(wl.b, in_dt),
             logits=pin(wl.logits), tokens=pin(wl.tokens))
    if wl.parent is not None:
        d["parent"] = pin(wl.parent)
    return d


def run_host_step(st: SpecStep, host: dict, out_host: dict, stream=None, graph: bool = False):
    """End-to-end step through the public API: H2D copy of the step's inputs
    from pinned memory, verify -> accept -> commit, D2H copy of the result
    (accept_len, accept_node, argmax: one copy when out_host comes from
    SpecStep.host_result_buffers). With graph=True the step is one graph
    launch: the whole host step captured by capture_host_step for these
    buffers, else the captured device step between eager copies. Returns
    (h2d_bytes, d2h_bytes)."""
    h2d = sum(host[n].numel() * host[n].element_size()
              for n in ("x", "a", "b", "logits", "tokens", "parent") if n in host)
    d2h = sum(out_host[n].numel() * out_host[n].element_size()
              for n in ("accept_len", "accept_node", "argmax"))
    bufs = getattr(st, "_graph_host_bufs", None)
    if graph and bufs is not None and bufs[0] is host and bufs[1] is out_host:
        st._graph_host.replay()
        return h2d, d2h
    for name in ("x", "a", "b", "logits", "tokens", "parent"):
        if name in host:
            getattr(st, name).copy_(host[name], non_blocking=True)
    if graph:
        st.replay()
    else:
        st.step_fn(getattr(st, "commit", "checkpoint"))(stream)
    st._copy_result(out_host)
    return h2d, d2h
