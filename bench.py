#!/usr/bin/env python3
"""Benchmark: GDN verify + greedy accept + on-device restore, one GPU.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one pass of the whole path over one batch: gdn_verify_span over
every layer (with per-token F32 checkpoints), spec_accept_greedy over the
logits, gdn_rollback_restore of the accepted slot. Default workload: 48 GDN
layers (H_k=16, H_v=32, d=128, 8192 channels, conv 4), chain span 16,
batch 1, logits [17, 151936] (synthetic, seeded). Metric: verified
tokens x layers per second.

Timing: W untimed warm-up steps, then exactly K timed steps between a barrier
+ synchronize on both sides. Each step is bracketed by CUDA events on the
launching stream; a 256 MiB buffer (larger than the 129 MB L2) is written
between steps, outside the events. The verify kernel's own events give the
roofline line. For N > 1 (torchrun) every rank runs its own requests
(replicas, no data-path collective); the step time is the max over ranks and
the value sums the units of all ranks.

--impl reference times the CPU oracle (plain C, double precision, one
thread) on the same workload, each step a bounded sample of it (a few
layers); it is a deliberately slow correctness program, not a target.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GDN verify+rollback tokens·layers/s (span 16, 48 layers); % of HBM roofline"
UNIT = "tokens*layers/s"
FLUSH_BYTES = 256 << 20
FALLBACK_HBM_GBS = 6800.0
CSRC = os.path.join(ROOT, "speculative_decode_hybrid_gb300", "csrc")
# the verify kernel's sources, hashed together (in this order) to tie the
# recorded ncu traffic to the code it was taken with
VERIFY_SRCS = [os.path.join(CSRC, f) for f in ("gdn_verify.cu", "gdn_verify_parts.cuh", "gdn_device.cuh")]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "gdn_verify_kernel_traffic.txt")
# one full-size ncu capture each: (workload, layers, verify kind) -> DRAM bytes
# of one verify launch, with the kernel sources it was taken at
TRAFFIC_FILES = [TRAFFIC_FILE,
                 os.path.join(ROOT, "profiles", "gdn_tree_verify_traffic.txt"),
                 os.path.join(ROOT, "profiles", "gdn_wy_kernel_traffic.txt")]


def parse():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=2, choices=[0, 1, 2, 3, 4])
    ap.add_argument("--seed", type=int, default=9,
                    help="base seed (9: the chain accepts k=2 of 16, near the mean for p=0.6)")
    ap.add_argument("--layers", type=int, default=None,
                    help="override the layer count (smaller profiling cases)")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--commit", choices=["checkpoint", "replay", "wy"], default="checkpoint",
                    help="checkpoint: per-token checkpoints + restore (the method); replay: "
                         "verify without checkpoints, then re-run the accepted tokens; wy: the "
                         "replay variant with the span solved in chunked (WY) form")
    ap.add_argument("--per-layer-steps", type=int, default=200,
                    help="steps of the per-layer launch measurement (batch 1, checkpoint commit)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle baseline sample")
    return ap.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def read_traffic_file(path):
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    return vals


def sources_sha(names):
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def recorded_traffic(workload=2, layers=48, kind="checkpoint"):
    """DRAM bytes per verify launch from the committed ncu summary of this
    workload, layer count and verify kind ("checkpoint" or "chunked"), or
    None when there is none or the kernel source changed since the counters
    were taken."""
    for path in TRAFFIC_FILES:
        try:
            vals = read_traffic_file(path)
            if (int(vals["workload"]), int(vals["layers"]), vals["verify"]) != (workload, layers, kind):
                continue
            if vals.get("source_sha256") != sources_sha(vals["sources"].split()):
                return None
            return int(vals["dram_bytes_per_launch"])
        except (OSError, KeyError, ValueError):
            continue
    return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed loop runs."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.lines = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        t0 = time.time()
        while not self.lines and time.time() - t0 < 5:
            time.sleep(0.02)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, t_begin: float, t_end: float):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            rows.append((ts, parts))
        inside = [r for r in rows if t_begin - 0.05 <= r[0] <= t_end + 0.15] or rows[-2:]
        sm = []
        reasons = set()
        pw = []
        smax = None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, p in inside:
            try:
                sm.append(float(p[2]))
                smax = float(p[3])
                pw.append(float(p[4]))
            except ValueError:
                pass
            for n, v in zip(names, p[6:10]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(inside),
                "power_w_max": max(pw) if pw else None}


def aggregate(local_time, local_units, ws, device):
    """Whole-job figures over the ranks of a replica run: the slowest rank's
    time (max) and the units of all ranks (sum). With one rank, unchanged."""
    if ws <= 1:
        return float(local_time), float(local_units)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(local_time)], dtype=torch.float64, device=device)
    u = torch.tensor([float(local_units)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def verify_footprint_bytes(s):
    """Bytes one verify of shape s moves (state and conv state read, every
    checkpoint written, inputs read, o written, conv weights read)."""
    T, C, K = s.n_tok, s.conv_ch, s.conv_k
    el = 2 if s.dtype == 1 else 4
    per = ((T + 1) * (s.h_v * s.d_v * s.d_k * 4 + C * (K - 1) * 4)
           + T * C * el + 2 * T * s.h_v * el + T * s.h_v * s.d_v * 4)
    return s.batch * s.layers * per + s.layers * C * K * el


def config_of(wl, kl, commit="checkpoint", l2=None):
    """The workload's config dict; both arms print it, so that the two lines
    can be matched key by key (only `l2`, how the GPU arm keeps the L2 cold,
    is the arm's own)."""
    s = wl.shape
    from speculative_decode_hybrid_gb300.workloads import WORKLOAD_NAMES
    if l2 is None:
        l2 = ("256 MiB buffer written between timed steps (outside the events); "
              "step footprint %.2f GiB" % (verify_footprint_bytes(s) / 2 ** 30))
    return {"workload": WORKLOAD_NAMES.get(BENCH_WID, "custom"), "batch": s.batch, "layers": s.layers,
            "span": s.n_tok, "tree_nodes": s.n_nodes if s.tree else None,
            "h_k": s.h_k, "h_v": s.h_v, "d_k": s.d_k, "d_v": s.d_v, "conv_channels": s.conv_ch,
            "conv_k": s.conv_k, "vocab": s.vocab, "input_dtype": "bf16" if s.dtype == 1 else "f32",
            "state_dtype": "f32", "accepted_len": [int(k) for k in kl], "seed": wl.seed,
            "l2": l2,
            "parallelism": "replicas (independent requests per rank, no collective)",
            "commit": commit}


def med_ms(xs):
    return statistics.median(xs) if xs else None


BENCH_WID = 2


def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    from speculative_decode_hybrid_gb300 import build as B
    from speculative_decode_hybrid_gb300 import gdnspec as G
    from speculative_decode_hybrid_gb300 import workloads as W
    from speculative_decode_hybrid_gb300.pipeline import SpecStep

    ws, rank, local = dist_env()
    if ws > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    B.build()
    G.load()

    wl = W.make_workload(BENCH_WID, seed=args.seed + 1000 * rank, layers=args.layers)
    st = SpecStep(wl, device=dev)
    replay = args.commit != "checkpoint"
    if replay and st.tree:
        raise SystemExit("the replay commit is defined for chains only")
    st.commit = args.commit
    f_verify = {"checkpoint": st.verify, "replay": st.verify_nockpt_fastest, "wy": st.verify_wy}[args.commit]
    f_commit = {"checkpoint": st.restore, "replay": st.commit_replay, "wy": st.commit_wy}[args.commit]
    step_fn = st.step_fn(args.commit)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    ssm0 = st.ssm_state.clone()
    conv0 = st.conv_state.clone()

    def barrier():
        if ws > 1:
            dist.barrier()

    for i in range(max(3, args.warmup)):
        step_fn()
    torch.cuda.synchronize(dev)
    kl = st.accept_len.cpu().numpy()
    kn = st.accept_node.cpu().numpy()

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    sampler = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                           else int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[0]))
    sampler.start()
    barrier()
    torch.cuda.synchronize(dev)
    t_begin = time.time()
    for i in range(K):
        flush.fill_(i & 0xFF)
        e = ev[i]
        e[0].record(stream)
        f_verify()
        e[1].record(stream)
        st.accept()
        e[2].record(stream)
        f_commit()
        e[3].record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    t_end = time.time()
    clocks = sampler.stop(t_begin, t_end)

    step_ms = [e[0].elapsed_time(e[3]) for e in ev]
    ver_ms = [e[0].elapsed_time(e[1]) for e in ev]
    acc_ms = [e[1].elapsed_time(e[2]) for e in ev]
    res_ms = [e[2].elapsed_time(e[3]) for e in ev]
    units = st.units()
    eager_max_ms, units_all = aggregate(sum(step_ms), units * K, ws, dev)
    eager_value = units_all / (eager_max_ms / 1e3)

    # ---- the same K steps as one CUDA graph launch each (the headline):
    #      events around every replay, L2 flushed between replays
    graph_ok = True
    try:
        st.capture(args.commit)
        for _ in range(3):
            st.replay()
        torch.cuda.synchronize(dev)
    except Exception as exc:  # capture unsupported: report the eager steps
        graph_ok = False
        print("graph capture failed: %r" % (exc,), file=sys.stderr)
    if graph_ok:
        gev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
        sampler2 = ClockSampler(sampler.index)
        sampler2.start()
        barrier()
        torch.cuda.synchronize(dev)
        tg0 = time.time()
        for i in range(K):
            flush.fill_(i & 0xFF)
            gev[i][0].record(stream)
            st.replay()
            gev[i][1].record(stream)
        torch.cuda.synchronize(dev)
        barrier()
        tg1 = time.time()
        gstep_ms = [e[0].elapsed_time(e[1]) for e in gev]
        total_max_ms, units_all = aggregate(sum(gstep_ms), units * K, ws, dev)
    else:
        gstep_ms = step_ms
        total_max_ms = eager_max_ms
    value = units_all / (total_max_ms / 1e3)

    hbm, peak_kind = peaks()
    vbytes = st.verify_bytes() if not replay else st.replay_bytes(np.zeros(st.shape.batch, dtype=int)) - st.accept_bytes()
    # the kernel timed: checkpointing, or the chunked checkpoint-free one (chain spans <= 16)
    verify_kind = "checkpoint" if not replay else ("chunked" if st.n_tok <= 16 and not st.tree else "other")
    ver_mean_s = statistics.mean(ver_ms) / 1e3
    achieved = vbytes / ver_mean_s / 1e9
    step_bytes = (vbytes + st.accept_bytes() + st.restore_bytes(kn)) if not replay else st.replay_bytes(kl)
    step_gbs = step_bytes / (statistics.mean(gstep_ms) / 1e3) / 1e9

    # ---- each kernel's cost inside the step graph (the eager per-kernel
    #      events above include launch gaps that programmatic dependent
    #      launch hides in the graph): graphs of the verify alone and of
    #      verify -> accept, beside the whole step
    parts = None
    if graph_ok and rank == 0:
        parts = graph_part_costs(st, args.commit, f_verify, flush, dev, stream, min(K, 200))

    # ---- end to end through the public API, host buffers, copies timed
    e2e = None
    if args.e2e_steps > 0:
        e2e = run_e2e(args, st, wl, flush, dev, stream, K, units, ws, kl)

    # ---- the same step with one verify launch per layer (how a model whose
    #      layers run in sequence calls it), as a CUDA graph; batch 1 only
    per_layer = None
    if args.commit == "checkpoint" and st.shape.batch == 1 and graph_ok and args.per_layer_steps > 0:
        per_layer = run_per_layer(st, flush, dev, stream, min(K, args.per_layer_steps), units, ws)

    # clocks: sampled from the graph loop to the end of the last timed loop
    # (graph step, in-graph parts, end to end, per-layer), all under load
    if graph_ok:
        clocks_graph = sampler2.stop(tg0, time.time())
        if clocks_graph.get("samples"):
            clocks = clocks_graph

    # the state moved every step; put the initial one back (not timed)
    st.ssm_state.copy_(ssm0)
    st.conv_state.copy_(conv0)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": K,
        "warmup": max(3, args.warmup), "ms_per_step": total_max_ms / K,
        "ms_per_step_median": statistics.median(gstep_ms), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": config_of(wl, kl, getattr(st, "commit", "checkpoint")),
        "roofline": {"bound": "hbm",
                     "kernel": {"checkpoint": "gdn_verify_persistent (%s)" % (
                                    "gdn_tree_verify" if st.tree else "gdn_verify_span"),
                                "replay": ("gdn_wy_kernel (gdn_verify_span_wy)" if st.n_tok <= 16
                                           else "gdn_verify_persistent (gdn_verify_span_nockpt)"),
                                "wy": "gdn_wy_kernel (gdn_verify_span_wy)"}[args.commit],
                     "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "peak_source": peak_kind, "traffic": recorded_traffic(BENCH_WID, st.shape.layers, verify_kind),
                     "algorithmic_bytes_per_launch": vbytes,
                     "verify_us_mean": ver_mean_s * 1e6,
                     "verify_us_median": statistics.median(ver_ms) * 1e3,
                     "accept_us_mean": statistics.mean(acc_ms) * 1e3,
                     "accept_us_median": statistics.median(acc_ms) * 1e3,
                     "restore_us_mean": statistics.mean(res_ms) * 1e3,
                     "restore_us_median": statistics.median(res_ms) * 1e3,
                     "eager_step_us_median": statistics.median(step_ms) * 1e3,
                     "step_bytes": step_bytes, "step_gbs": step_gbs, "step_frac": step_gbs / hbm,
                     "in_graph_us": parts},
        "e2e": e2e,
        "per_layer": per_layer,
        "mode": "cuda_graph" if graph_ok else "eager",
        "eager": {"value": eager_value, "ms_per_step": eager_max_ms / K},
        "clocks": clocks,
        "gpu_launches": {"checkpoint": SpecStep.LAUNCHES_PER_STEP, "replay": SpecStep.LAUNCHES_PER_STEP_REPLAY,
                         "wy": SpecStep.LAUNCHES_PER_STEP_WY}[args.commit] * K,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, args.cpu_seconds)
    if ws > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_e2e(args, st, wl, flush, dev, stream, K, units, ws, kl):
    """The same metric end to end through the public API: each step copies
    its inputs from pinned host memory, runs verify -> accept -> restore and
    reads the accepted length / node / argmax back; wall clock per step."""
    import torch
    from speculative_decode_hybrid_gb300.pipeline import pinned_host_inputs, run_host_step
    host = pinned_host_inputs(wl)
    out_host = st.host_result_buffers()  # the result comes back in one copy
    E = max(1, min(args.e2e_steps, K))
    e2e_s = []
    h2d = d2h = 0
    mode = "eager copies + device graph"
    try:
        st.capture_host_step(host, out_host, args.commit)
        if args.commit == "checkpoint":
            mode = "one graph per step: one verify launch at once (gdn_*_verify_pipelined) while x/a/b land " \
                   "in blocks (sizes 1:1:2:4:8:8), each block's flags set by a copy behind it; " \
                   "logits/tokens copied during the verify, then accept, commit, one D2H of the result"
        else:
            mode = "one graph per step: x/a/b copied in 3 blocks (sizes 1:3:8), the verify of each block " \
                   "launched as its block lands, logits/tokens copied during the verify, then accept, " \
                   "commit, one D2H of the result"
    except Exception as exc:  # capture unsupported: copies stay eager around the device graph
        print("host-step capture failed: %r" % (exc,), file=sys.stderr)
    for i in range(E + 3):
        flush.fill_(i & 0xFF)
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        h2d, d2h = run_host_step(st, host, out_host, graph=getattr(st, "_graph", None) is not None)
        stream.synchronize()
        t1 = time.perf_counter()
        if i >= 3:
            e2e_s.append(t1 - t0)
    e2e_max_s, e2e_units = aggregate(sum(e2e_s), units * E, ws, dev)
    assert int(out_host["accept_len"][0]) == int(kl[0])
    return {"value": e2e_units / e2e_max_s, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": E, "ms_per_step": 1e3 * statistics.mean(e2e_s),
            "ms_per_step_median": 1e3 * statistics.median(e2e_s),
            "mode": mode}


def graph_part_costs(st, commit, f_verify, flush, dev, stream, n):
    """Median µs of graph replays of the verify alone, of the verify with
    either of the other two kernels and of the whole step, L2 flushed
    between replays; the accept's and the commit's costs inside the step
    are what each adds to the other two."""
    import torch
    main_graph = getattr(st, "_graph", None)
    f_commit = {"checkpoint": st.restore, "replay": st.commit_replay, "wy": st.commit_wy}[commit]
    ssm0, conv0 = st.ssm_state.clone(), st.conv_state.clone()
    fns = {"verify": lambda stream=None: f_verify(stream),
           "verify_accept": lambda stream=None: (f_verify(stream), st.accept(stream)),
           "verify_commit": lambda stream=None: (f_verify(stream), f_commit(stream)),
           "step": lambda stream=None: (f_verify(stream), st.accept(stream), f_commit(stream))}
    out = {}
    try:
        graphs = {}
        for name, fn in fns.items():
            st.step_fn = lambda c, fn=fn: fn
            graphs[name] = st.capture(name)
            for _ in range(3):
                graphs[name].replay()
        torch.cuda.synchronize(dev)
        # the four graphs replayed in turn, so that a drift of the box's
        # speed during the loop weighs on all of them alike
        ev = {name: [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)] for name in graphs}
        for i in range(n):
            for name, g in graphs.items():
                flush.fill_(i & 0xFF)
                ev[name][i][0].record(stream)
                g.replay()
                ev[name][i][1].record(stream)
        torch.cuda.synchronize(dev)
        for name in graphs:
            out[name] = statistics.median([a.elapsed_time(b) for a, b in ev[name]]) * 1e3
        st.ssm_state.copy_(ssm0)
        st.conv_state.copy_(conv0)
    finally:
        st.__dict__.pop("step_fn", None)  # the class's step_fn again
        st._graph = main_graph
    # the cost a kernel adds to the other two (its tail overlaps the next
    # kernel's launch, so it is less than its own graph's end-to-end time)
    out["accept"] = out["step"] - out["verify_commit"]
    out["commit"] = out["step"] - out["verify_accept"]
    return {k: round(v, 2) for k, v in out.items()}


def run_per_layer(st, flush, dev, stream, K, units, ws):
    """Graph-replayed steps whose verify is one launch per layer, with the L2
    flushed between replays; plus the per-layer verify launches alone
    (eager, events around the whole loop)."""
    import torch
    main_graph = getattr(st, "_graph", None)
    st.capture("checkpoint-per-layer")
    for _ in range(3):
        st.replay()
    torch.cuda.synchronize(dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    for i in range(K):
        flush.fill_(i & 0xFF)
        ev[i][0].record(stream)
        st.replay()
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    vev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(min(K, 50))]
    for i in range(len(vev)):
        flush.fill_(i & 0xFF)
        vev[i][0].record(stream)
        st.verify_per_layer()
        vev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    ver_ms = [a.elapsed_time(b) for a, b in vev]
    st._graph = main_graph
    total_max_ms, units_all = aggregate(sum(step_ms), units * K, ws, dev)
    return {"value": units_all / (total_max_ms / 1e3), "unit": UNIT, "steps": K,
            "ms_per_step": total_max_ms / K, "ms_per_step_median": statistics.median(step_ms),
            "launches_per_step": st.shape.layers + 2,
            "verify_us_mean": statistics.mean(ver_ms) * 1e3,
            "verify_us_median": statistics.median(ver_ms) * 1e3,
            "verify_us_per_layer": statistics.mean(ver_ms) * 1e3 / st.shape.layers,
            "mode": "cuda_graph (step), eager (verify alone)"}


def oracle_full_step(wl, layers, accept=True, pool=None):
    """One oracle step over `layers`: verify + restore of each, plus acceptance.
    With a thread pool the layers' verifies run concurrently (the oracle is C
    called through ctypes, which releases the GIL; the layers are independent)."""
    import oracle
    if pool is None:
        res = oracle.verify_request(wl, 0, layers=layers)
    else:
        res = list(pool.map(lambda y: oracle.verify_request(wl, 0, layers=[y])[0], layers))
    par = wl.parent[0] if wl.parent is not None else None
    kl, kn = 0, 0
    if accept:
        _, kl, kn = oracle.accept_greedy(wl.logits[0], wl.tokens[0], par)
    for y, (ck, cc, _) in zip(layers, res):
        oracle.restore(ck, kn, wl.ssm0[0, y])
        oracle.restore(cc, kn, wl.conv0[0, y])
    return kl


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def cpu_baseline(wl, target_s):
    """The oracle as it stands on full steps of request 0: on all host cores
    (one thread per layer in flight), and on one thread (`single_thread`).
    Each leg runs for about half of `target_s`."""
    from concurrent.futures import ThreadPoolExecutor
    s = wl.shape
    layers = list(range(s.layers))

    def leg(pool, budget):
        times = []
        t_all = time.perf_counter()
        while True:
            t0 = time.perf_counter()
            oracle_full_step(wl, layers, pool=pool)
            times.append(time.perf_counter() - t0)
            if time.perf_counter() - t_all >= budget or len(times) >= 30:
                return times

    t1 = leg(None, target_s / 2)
    cores = max(1, min(host_cores(), s.layers))
    with ThreadPoolExecutor(max_workers=cores) as pool:
        tn = leg(pool, target_s / 2)
    v1 = s.n_tok * s.layers / statistics.mean(t1)
    vn = s.n_tok * s.layers / statistics.mean(tn)
    return {"value": vn, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": "%d full steps of request 0 (%d layers verify + accept + restore), plain C "
                      "double precision, the layers on %d threads, %.1f s total"
                      % (len(tn), s.layers, cores, sum(tn)),
            "single_thread": {"value": v1, "cores": 1, "steps": len(t1), "seconds": sum(t1)}}


def run_reference(args):
    """The oracle on the host cores, K steps of a bounded sample each."""
    ws, rank, local = dist_env()
    if rank != 0:
        return
    import oracle
    from speculative_decode_hybrid_gb300 import workloads as W
    oracle.build()
    wl = W.make_workload(BENCH_WID, seed=args.seed, layers=args.layers)
    s = wl.shape
    from concurrent.futures import ThreadPoolExecutor
    cores = max(1, min(host_cores(), s.layers))
    pool = ThreadPoolExecutor(max_workers=cores)
    # calibrate: one layer + acceptance; the layers of a step run on `cores` threads
    t0 = time.perf_counter()
    oracle_full_step(wl, [0])
    t1 = time.perf_counter() - t0
    budget = 150.0 / max(1, args.steps + args.warmup)
    nl = int(max(1, min(s.layers, cores * (budget // max(t1, 1e-3)))))
    # the acceptance runs once per s.layers layers of verify work, as in a full step
    def sample(i):
        layers = [(i * nl + j) % s.layers for j in range(nl)]
        return layers, (i * nl) % s.layers < nl

    for i in range(args.warmup):
        oracle_full_step(wl, *sample(i), pool=pool)
    times = []
    for i in range(args.steps):
        layers, acc = sample(i)
        t0 = time.perf_counter()
        oracle_full_step(wl, layers, acc, pool=pool)
        times.append(time.perf_counter() - t0)
    pool.shutdown()
    par = wl.parent[0] if wl.parent is not None else None
    k_ref = int(oracle.accept_greedy(wl.logits[0], wl.tokens[0], par)[1])
    total = sum(times)
    value = s.n_tok * nl * args.steps / total
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": config_of(wl, [k_ref], "checkpoint",
                                l2="CPU arm: host caches, no GPU L2 to flush"),
            "ms_per_step_median": 1e3 * statistics.median(times),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": "each step: %d of %d layers (verify + restore); the acceptance "
                                       "once per %d layers of work; plain C double precision, the "
                                       "layers on %d threads" % (nl, s.layers, s.layers, cores),
                             "layers_per_step_sample": nl},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    global BENCH_WID
    args = parse()
    BENCH_WID = args.workload
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
