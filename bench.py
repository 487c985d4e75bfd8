"""Benchmark of the verify-and-accept step on GB300.

One step = one speculative round over a batch: the tree attention mask
(sv_tree_build_mask), the tree verify (sv_verify_tree: best-child path, row
statistics, accept walk, residual / bonus sampling) and the KV compaction of
the accepted paths (sv_kv_compact, in place).  The mask and the compaction run
on a second stream: the mask needs only the tree, and the compaction starts
at the verify call's accept event, overlapping the residual / bonus sampling.  Default workload: the dynamic
EAGLE-2 tree (B=128, 60-node budget, depth 6, top-k 10, V=128256, bf16 logits,
KV shaped like a 70B model: 80 layers x 8 KV heads x 128).  `--config 3` runs
the large-vocabulary chain (B=256, N=7) instead (verify + chain rollback).

Prints one JSON line.  `value` = verified logit rows per second (B*T per tree
round, B*(N+1) per chain round) with inputs resident in HBM; `e2e` = the same
with the inputs in page-locked host memory, which the kernels read in place
over NVLink-C2C (only the rows a round touches cross the link), and the
device -> host read of the results inside the timed region (`e2e.copy_all`:
the same with a full host -> device copy of every input first); `roofline` = the row-statistics
kernel's algorithmic bytes over its CUDA-event time against the measured HBM
copy bandwidth; `cpu_baseline` = the CPU oracle on a bounded sample.

The timed region runs K steps with no event between launches (the library
chains its kernels by programmatic dependent launch).  Per-kernel durations
come from a second pass over the same K steps with an event pair around every
launch; those events serialise the launches, so that pass reports its own
`traced_ms_per_step` and is not the step time.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config 5|3]
    python bench.py --impl reference ...      # the CPU oracle alone
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified rows/s and accepted tokens/s at 1 GB300; achieved HBM GB/s vs ~8 TB/s"
L2_BYTES = 129 * 2 ** 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default 1000; 20 for --impl reference, the CPU oracle)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=5, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--pool", type=int, default=4, help="distinct rounds rotated in the timed loop")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample", type=int, default=16, help="sequences the oracle times")
    ap.add_argument("--tree-build", action="store_true",
                    help="time the GPU dynamic-tree builder instead of the verify step")
    ap.add_argument("--attention", action="store_true",
                    help="time the tree-masked verifier attention (one layer) instead")
    ap.add_argument("--greedy", action="store_true",
                    help="temperature 0: greedy verification (verifier rows only, no sampling)")
    ap.add_argument("--graph", action="store_true",
                    help="capture each pooled round's step in a CUDA graph and replay it in "
                         "the timed loop (the latency-bound small configurations)")
    ap.add_argument("--early-exit", action="store_true",
                    help="chain configs: sv_verify_chain_early_exit (rows after a sequence's "
                         "first rejection are not read once it is known)")
    ap.add_argument("--no-secondary", action="store_true",
                    help="config 5 only: leave out the large-vocabulary chain lines")
    ap.add_argument("--batch", type=int, default=0,
                    help="per-GPU batch override (smaller cases for profiler captures)")
    return ap.parse_args()


# ------------------------------------------------------------------ helpers
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def shard_batch(B, rank, world):
    """Weak scaling: every rank verifies its own batch of B sequences (the
    per-GPU batch of the workload), so the job covers world * B sequences.
    Returns (first global sequence index of this rank, B)."""
    return rank * B, B


def rank_seed(base, rank):
    """Philox key of a rank: ranks draw independent uniforms (the kernel's
    counter carries the in-batch sequence index, the key the rank)."""
    return base + rank


def _reduce(x, op):
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=op)
    return float(t.item())


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    return _reduce(x, dist.ReduceOp.MAX)


def sum_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    return _reduce(x, dist.ReduceOp.SUM)


def aggregate(units, ms, world):
    """Whole-job throughput: the units all ranks processed over the slowest
    rank's time.  Returns (total units, max ms, units per second)."""
    ms_max = max_over_ranks(ms, world)
    total = sum_over_ranks(units, world)
    return total, ms_max, total / (ms_max / 1e3)


def best_path_depth(parent, score, max_depth):
    """Depth of the best-child walk per sequence (host, numpy), used only to
    count the rows the verify step reads."""
    B, T = parent.shape
    out = np.zeros(B, np.int64)
    for b in range(B):
        cur, D = 0, 0
        while D < max_depth:
            kids = np.nonzero(parent[b] == cur)[0]
            if kids.size == 0:
                break
            s = score[b, kids]
            cur = int(kids[np.flatnonzero(s == s.max())[0]])
            D += 1
        out[b] = D
    return out


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons; `region()` marks
    the timed region on the host clock, and the summary keeps the samples
    stamped inside it (all samples if none fell inside)."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.t0 = self.t1 = None

    def region(self, start):
        import datetime
        now = datetime.datetime.now()
        if start:
            self.t0 = now
        else:
            self.t1 = now

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        import datetime
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = []
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f")
                rows.append((ts, float(f[2]), float(f[3]), f[6:10]))
            except ValueError:
                continue
        inside = [r for r in rows if self.t0 and self.t1 and self.t0 <= r[0] <= self.t1]
        use = inside or rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        reasons = sorted({n for r in use for n, v in zip(names, r[3])
                          if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[1] for r in use),
                "sm_max_mhz": max(r[2] for r in use), "reasons": reasons,
                "samples": len(use), "samples_in_timed_region": len(inside)}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# the sources each profiled kernel is built from (its counters stay valid while
# these files are unchanged)
KERNEL_SOURCES = {
    "row_stats": ("common.cuh", "rowstat.cuh", "verify.cu"),
    "row_stats_ee": ("common.cuh", "rowstat.cuh", "verify.cu"),
    "sampler_kv": ("common.cuh", "rowstat.cuh", "tree_kv.cu", "verify.cu"),
    "launches": ("common.cuh", "rowstat.cuh", "tree_kv.cu", "verify.cu"),
    "tree_attention": ("common.cuh", "tree_attn.cu"),
    "tree_expand": ("common.cuh", "rowstat.cuh", "tree_build.cu"),
}


def source_hash(kernel):
    src = os.path.join(ROOT, "speculative_decoding_verification_vocab_gb300", "csrc")
    return hashlib.sha256(b"".join(open(os.path.join(src, f), "rb").read()
                                   for f in KERNEL_SOURCES[kernel])).hexdigest()[:16]


def recorded_traffic(kernel, cfg_name):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, if it
    was taken on the current sources of the kernel (source hash recorded)."""
    p = os.path.join(ROOT, "profiles", f"{kernel}_{cfg_name}.txt")
    if not os.path.exists(p):
        return None
    txt = open(p).read()
    m = re.search(r"dram_bytes_per_launch_full_size:\s*([0-9.eE+]+)", txt)
    h = re.search(r"source_sha256:\s*([0-9a-f]+)", txt)
    if not m or not h:
        return None
    return float(m.group(1)) if source_hash(kernel) == h.group(1) else None


# ------------------------------------------------------------------ workload
class Workload:
    def __init__(self, cfg, pool, device, seq_offset):
        import torch
        from speculative_decoding_verification_vocab_gb300 import synth
        self.cfg = cfg
        self.greedy = False
        self.early = False
        self.rounds = []
        self.tree = cfg.kind.startswith("tree")
        for r in range(pool):
            if self.tree:
                vq, dp, parent, token, score = synth.tree_inputs(cfg, seed=r + 1000 * seq_offset,
                                                                 device=device)
                depth = best_path_depth(parent.cpu().numpy(), score.cpu().numpy(), cfg.depth)
                self.rounds.append(dict(vq=vq, dp=dp, parent=parent, token=token, score=score,
                                        depth=depth))
            else:
                vq, dp, d = synth.chain_inputs(cfg, seed=r + 1000 * seq_offset, device=device)
                self.rounds.append(dict(vq=vq, dp=dp, d=d,
                                        depth=np.full(cfg.B, cfg.N, np.int64)))
        torch.cuda.synchronize()
        self.B = cfg.B
        self.T = self.rounds[0]["vq"].shape[1]
        self.V = cfg.V
        self.esize = self.rounds[0]["vq"].element_size()
        kv = cfg.kv
        # KV window: the slots the round writes and compacts, for every sequence
        # (the prefix of `kv.base` rows is never touched by the step)
        self.S = self.T + 4
        self.kv = synth.kv_cache(kv.L, cfg.B, self.S, kv.H, kv.D, device=device, seed=7)
        self.kv_base = torch.zeros(cfg.B, dtype=torch.int32, device=device)
        self.row_bytes = kv.H * kv.D * self.kv.element_size()

    def rows_per_step(self):
        return self.B * self.T

    def stats_bytes(self, r, acc=None):
        """Logit bytes the row pass must read: verifier and draft rows along
        the path (2D+1 per sequence), the verifier rows alone when greedy, or
        with early exit the rows the walk reaches given the accept lengths
        `acc`: 2(a+1) after a rejection at a < D, 2D+1 on full acceptance."""
        d = self.rounds[r]["depth"]
        if self.early and acc is not None:
            a = np.asarray(acc, np.int64)
            rows = np.where(a < d, 2 * (a + 1), 2 * d + 1)
        else:
            rows = d + 1 if self.greedy else 2 * d + 1
        return int((rows * self.V * self.esize).sum())


def run_round(sv, wl, cfg, maxd, src, out, i, seed, step_no, ws, stream, side, ev_fork, ev_acc):
    """One speculative round, the way a serving loop would issue it: the main
    stream verifies; a side stream builds the tree mask (it needs only the
    tree) and, once the accept walk's event fires, compacts the KV cache while
    the main stream still samples the correction / bonus tokens.  The main
    stream joins the side stream at the end, so the round is complete there.
    `out` holds per-round output views: path, tok, acc, st, kv, mask, depth."""
    ev_fork.record(stream)
    side.wait_event(ev_fork)
    if wl.tree:
        sv.sv_tree_build_mask(src["parent"], out["mask"], out["depth"], side)
        sv.sv_verify_tree(src["vq"], src["dp"], src["parent"], src["token"], src["score"], maxd,
                          cfg.temperature, seed, step_no, out["path"][i], out["tok"][i],
                          out["acc"][i], None, None, None, out["st"][i], ws, stream,
                          accept_event=ev_acc)
        side.wait_event(ev_acc)
        sv.sv_kv_compact(wl.kv, wl.kv, wl.kv_base, wl.kv_base, out["path"][i], out["acc"][i], 1,
                         out["kv"][i], side)
    else:
        verify = sv.sv_verify_chain_early_exit if wl.early else sv.sv_verify_chain
        verify(src["vq"], src["dp"], src["d"], cfg.temperature, seed, step_no,
               out["tok"][i], out["acc"][i], None, None, None, out["st"][i], ws,
               stream, accept_event=ev_acc)
        side.wait_event(ev_acc)
        # chain rollback: the accepted drafts' rows are already in place;
        # only the logical length moves (rows NULL = identity)
        sv.sv_kv_compact(wl.kv, wl.kv, wl.kv_base, wl.kv_base, None, out["acc"][i], 1,
                         out["kv"][i], side)
    stream.wait_stream(side)


def run_ours(args):
    import torch

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    line = measure(args, rank, world, local)
    if args.config == 5 and not (args.greedy or args.early_exit or args.graph or args.batch or
                                 args.no_secondary):
        line["secondary"] = secondary(args, rank, world, local)
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


SECONDARY_STEPS = 50


def secondary(args, rank, world, local):
    """The large-vocabulary chain (B=256, N=7, V=128256), the workload the
    bandwidth target names, measured in the same run as the headline line:
    the full reading and the early-exit reading, each over SECONDARY_STEPS
    timed steps (at least K) with its own row-pass roofline.  Device-resident
    inputs only (no end-to-end or CPU legs)."""
    import argparse as ap
    out = {}
    for name, early in (("config 3: large_vocab_chain", False),
                        ("config 3: large_vocab_chain (early exit)", True)):
        a = ap.Namespace(**vars(args))
        a.config, a.early_exit, a.greedy, a.graph, a.batch = 3, early, False, False, 0
        a.steps = max(args.steps, SECONDARY_STEPS)
        a.no_e2e = a.no_cpu_baseline = True
        m = measure(a, rank, world, local)
        out[name] = {k: m[k] for k in ("value", "unit", "steps", "ms_per_step",
                                       "accepted_tokens_per_s", "mean_accept_len",
                                       "rows_read_per_s", "hbm_gbs", "hbm_frac_measured",
                                       "roofline", "kernels", "repeats", "clocks",
                                       "alg_bytes_per_step", "config")}
    return out


def measure(args, rank, world, local):
    """One workload measured as the JSON line reports it (returns the dict)."""
    import torch
    import speculative_decoding_verification_vocab_gb300 as sv
    from speculative_decoding_verification_vocab_gb300 import synth

    dev = torch.device("cuda", local)
    sv.load_library()
    cfg = synth.CONFIGS[args.config]
    import dataclasses
    if args.batch:
        cfg = dataclasses.replace(cfg, B=args.batch)
    _, B = shard_batch(cfg.B, rank, world)
    wl = Workload(cfg, args.pool, dev, rank)  # inputs drawn at the configuration's T
    if args.greedy:  # then verified at T = 0
        cfg = dataclasses.replace(cfg, temperature=0.0)
        wl.greedy = True
    if args.early_exit:
        if wl.tree or wl.greedy:
            raise SystemExit("--early-exit applies to chain configs at T > 0")
        wl.early = True
    K, W = args.steps, args.warmup
    T, V = wl.T, wl.V
    maxd = cfg.depth if wl.tree else cfg.N
    P = maxd + 1
    # per-step outputs land in slices of these buffers (no extra work per step)
    o_path = torch.empty(K + W, B, P, dtype=torch.int32, device=dev)
    o_tok = torch.empty(K + W, B, P, dtype=torch.int32, device=dev)
    o_acc = torch.empty(K + W, B, dtype=torch.int32, device=dev)
    o_st = torch.empty(K + W, B, dtype=torch.int32, device=dev)
    o_kv = torch.empty(K + W, B, dtype=torch.int32, device=dev)
    Wm = (T + 63) // 64
    o_mask = torch.empty(B, T, Wm, dtype=torch.int64, device=dev)
    o_depth = torch.empty(B, T, dtype=torch.int32, device=dev)
    ws_bytes = (sv.sv_verify_tree_workspace(B, T, maxd, V) if wl.tree
                else sv.sv_verify_chain_workspace(B, cfg.N, V))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    side = torch.cuda.Stream(device=dev)
    ev_fork, ev_acc = torch.cuda.Event(), torch.cuda.Event()
    outs = dict(path=o_path, tok=o_tok, acc=o_acc, st=o_st, kv=o_kv, mask=o_mask, depth=o_depth)

    def step(i, rd, seed_step, on=None):
        run_round(sv, wl, cfg, maxd, rd, outs, i, rank_seed(1234, rank), seed_step, ws,
                  stream if on is None else on, side, ev_fork, ev_acc)

    graphs, graph_launches = None, 0
    if args.graph:
        # one graph per pooled round (its step number fixed at capture, its
        # outputs in slice W + round), both streams of the step inside it;
        # every replay re-runs every kernel
        cap = torch.cuda.Stream(device=dev)
        graphs = []
        c0 = sv.sv_launch_count()
        for r in range(args.pool):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                step(W + r, wl.rounds[r], W + r, on=cap)
            graphs.append(g)
        graph_launches = (sv.sv_launch_count() - c0) // args.pool
        torch.cuda.synchronize()

    def timed_step(k):
        if graphs is not None:
            graphs[k % args.pool].replay()
        else:
            step(W + k, wl.rounds[k % args.pool], W + k)

    def out_slice(k):  # where timed step k left its outputs
        return W + (k % args.pool) if graphs is not None else W + k

    # timed region: K steps back to back (kernels chained by programmatic
    # dependent launch; no event between them)
    # a pool of rounds smaller than twice L2 (the tiny chain) would be read
    # from L2: then every step is timed alone, with a 256 MB write between
    # steps outside its events
    pool_bytes = sum(v.numel() * v.element_size() for rd in wl.rounds
                     for v in (rd["vq"], rd["dp"]))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if pool_bytes < 2 * L2_BYTES \
        else None
    def time_loop():
        """K timed steps: back to back under one event pair, or (flush mode)
        each under its own pair with the L2 flush between them.  Returns ms."""
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        step_ms = 0.0
        for k in range(K):
            if flush is not None:
                flush.fill_(k & 255)
                s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                s0.record(stream)
            timed_step(k)
            if flush is not None:
                s1.record(stream)
                s1.synchronize()
                step_ms += s0.elapsed_time(s1)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) if flush is None else step_ms

    # the clock sampler starts first (it idles the host for a moment while
    # nvidia-smi comes up); the W untimed warm-up steps then run right before
    # the timed ones, so the timing starts on warm clocks
    with Clocks(local) as clk:
        for i in range(W):
            step(i, wl.rounds[i % args.pool], i)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        n_launch0 = sv.sv_launch_count()
        clk.region(True)
        ms = time_loop()
        clk.region(False)
    if world > 1:
        torch.distributed.barrier()
    launches = sv.sv_launch_count() - n_launch0 + K * graph_launches
    # the same K steps again with an event pair around every launch: per-kernel
    # durations (the events serialise the launches, so this pass is slower and
    # is not the step time)
    sv.sv_trace_enable(True)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for k in range(K):
        step(W + k, wl.rounds[k % args.pool], W + k)
    t1.record(stream)
    torch.cuda.synchronize()
    sv.sv_trace_enable(False)
    trace = sv.sv_trace_collect()
    traced_ms = t0.elapsed_time(t1)
    # the spread: 5 more repeats of the timed loop, each timed the same way
    # (outside the measurement above)
    rep_ms = [time_loop() / K for _ in range(5)]

    acc = o_acc[W:].cpu().numpy()
    st = o_st[W:].cpu().numpy()
    paths = o_path[W:].cpu().numpy()
    rows = wl.rows_per_step() * K
    tokens = int((acc + 1).sum())
    depth_used = np.stack([wl.rounds[k % args.pool]["depth"] for k in range(K)])
    alpha_hat = float(acc.sum() / max(1, np.minimum(acc + 1, depth_used).sum()))
    # algorithmic bytes
    stats_bytes = sum(wl.stats_bytes(k % args.pool, acc[k]) for k in range(K))
    kv_moved = 0
    if wl.tree:
        for k in range(K):
            for b in range(B):
                a = acc[k, b]
                kv_moved += int(sum(1 for j in range(1, a + 1) if paths[k, b, j] != j))
    kvb = cfg.kv
    kv_bytes = kv_moved * 2 * kvb.L * 2 * wl.row_bytes
    mask_bytes = K * B * T * (4 + 8 * Wm + 4) if wl.tree else 0
    alg_bytes = stats_bytes + kv_bytes + mask_bytes
    total_rows, ms_max, value = aggregate(rows, ms, world)
    total_tokens = sum_over_ranks(tokens, world)

    peak, peak_kind = measured_peaks()
    rs_name = ("row_argmax" if cfg.temperature == 0.0 else
               "row_stats_ee" if wl.early else "row_stats")
    rs_launches, rs_ms = trace.get(rs_name, (0, 0.0))
    rs_bytes_per_launch = stats_bytes / K
    rs_avg_ms = rs_ms / max(rs_launches, 1)
    achieved = rs_bytes_per_launch / (rs_avg_ms / 1e3) / 1e9 if rs_launches else None
    roofline = {"kernel": rs_name, "bound": "hbm", "achieved": achieved, "peak": peak,
                "peak_kind": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
                "unit": "GB/s", "frac": (achieved / peak) if achieved else None,
                "traffic": recorded_traffic(rs_name, cfg.name),
                "alg_bytes_per_launch": rs_bytes_per_launch, "avg_launch_ms": rs_avg_ms}

    line = {
        "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": ms_max / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if cfg.dtype.__repr__().endswith("bfloat16") else "f32",
        "data": "synthetic",
        "config": {"workload": f"config {cfg.index}: {cfg.name}" + (" (greedy, T=0)" if wl.greedy else "")
                   + (" (CUDA graph replay)" if graphs is not None else "")
                   + (" (early exit)" if wl.early else ""), "B_per_gpu": B, "T": T, "V": V,
                   "max_depth": maxd, "logits": str(cfg.dtype).replace("torch.", ""),
                   "kv": f"{kvb.L} layers x {kvb.H} kv heads x {kvb.D}, bf16",
                   "pool_rounds": args.pool,
                   "l2": (f"L2 flushed between steps (a 256 MB write outside each step's events; "
                          f"the pool of rounds is {pool_bytes / 1e6:.2f} MB)") if flush is not None else
                         f"inputs larger than L2: each step reads {stats_bytes / K / 1e6:.0f} MB of "
                         f"logit rows from a pool of {args.pool} distinct rounds "
                         f"({args.pool * wl.rounds[0]['vq'].numel() * wl.esize * 2 / 1e9:.1f} GB)"},
        "accepted_tokens_per_s": total_tokens / (ms_max / 1e3),
        # logit rows the row pass actually reads (verifier and draft rows on
        # the path; `value` counts B*T tree slots, most of which are never read)
        "rows_read_per_s": sum_over_ranks(stats_bytes / (V * wl.esize), world) / (ms_max / 1e3),
        "mean_emitted_per_seq": tokens / (K * B), "mean_accept_len": float(acc.mean()),
        "alpha_hat": alpha_hat,
        "us_per_round": 1e3 * ms_max / K,
        "repeats": {"n": len(rep_ms), "ms_per_step_median": float(np.median(rep_ms)),
                    "p10": float(np.percentile(rep_ms, 10)),
                    "p90": float(np.percentile(rep_ms, 90)),
                    "note": "5 further repeats of the K-step loop after the measurement"},
        "hbm_gbs": alg_bytes / (ms_max / 1e3) / 1e9,
        "hbm_frac_measured": alg_bytes / (ms_max / 1e3) / 1e9 / peak,
        "hbm_frac_nominal_8tbs": alg_bytes / (ms_max / 1e3) / 1e9 / 8000.0,
        "alg_bytes_per_step": {"row_stats": stats_bytes / K, "kv_compact": kv_bytes / K,
                               "tree_mask": mask_bytes / K},
        "kernels": {k: {"launches": v[0], "avg_us": 1e3 * v[1] / max(v[0], 1)} for k, v in trace.items()},
        "traced_ms_per_step": traced_ms / K,
        "status_nonzero": int((st != 0).sum()),
        "gpu_launches": int(launches),
        "roofline": roofline,
        "clocks": clk.summary(),
    }
    kv_launches, kv_ms = trace.get("kv_compact", (0, 0.0))
    if wl.tree and kv_launches:
        # the compaction runs on the side stream beside the sampling: its
        # bandwidth inside the step (event pair on that stream, traced pass)
        kv_gbs = (kv_bytes / K) / (kv_ms / kv_launches / 1e3) / 1e9
        line["kv_compact_in_step"] = {"alg_bytes_per_launch": kv_bytes / K,
                                      "avg_launch_ms": kv_ms / kv_launches, "achieved": kv_gbs,
                                      "unit": "GB/s", "frac": kv_gbs / peak}
    if not args.no_e2e:
        line["e2e"] = e2e_ours(args, wl, cfg, sv, dev, stream, maxd, B, world)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args, wl, cfg)
    del wl
    torch.cuda.empty_cache()
    return line


def e2e_ours(args, wl, cfg, sv, dev, stream, maxd, B, world):
    """The step through host buffers, end to end: the round's inputs sit in
    page-locked host memory, the three calls run on them, and the results are
    read back to page-locked host buffers, all inside the timed region.

    Main figure: the calls take the host buffers themselves; the kernels read
    in place, over NVLink-C2C, only the logit rows the round touches (the best
    path's rows, then the one or two sampled rows twice), so the host->device
    bytes are those reads.  `copy_all` is the plain alternative, timed the
    same way: copy every input to the device first, then run on the copies."""
    import torch
    rd = wl.rounds[0]
    names = ["vq", "dp", "parent", "token", "score"] if wl.tree else ["vq", "dp", "d"]
    host = {n: rd[n].cpu().pin_memory() for n in names}
    P = maxd + 1
    T, V = wl.T, wl.V
    outs = dict(path=torch.empty(B, P, dtype=torch.int32, device=dev),
                tok=torch.empty(B, P, dtype=torch.int32, device=dev),
                acc=torch.empty(B, dtype=torch.int32, device=dev),
                st=torch.empty(B, dtype=torch.int32, device=dev),
                kv=torch.empty(B, dtype=torch.int32, device=dev))
    hout = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in outs.items()}
    # the host-size workspace: each host row read crosses the link once
    ws = torch.empty(sv.sv_verify_tree_workspace_host(B, T, maxd, V, rd["vq"].dtype) if wl.tree
                     else sv.sv_verify_chain_workspace_host(B, cfg.N, V, rd["vq"].dtype),
                     dtype=torch.uint8, device=dev)
    Wm = (T + 63) // 64
    o_mask = torch.empty(B, T, Wm, dtype=torch.int64, device=dev)
    o_depth = torch.empty(B, T, dtype=torch.int32, device=dev)
    d2h = sum(h.numel() * h.element_size() for h in hout.values())

    side = torch.cuda.Stream(device=dev)
    ev_fork, ev_acc = torch.cuda.Event(), torch.cuda.Event()
    o1 = {k: v[None] for k, v in outs.items()}
    o1.update(mask=o_mask, depth=o_depth)

    def calls(src, i):
        run_round(sv, wl, cfg, maxd, src, o1, 0, 99, i, ws, stream, side, ev_fork, ev_acc)
        for k in outs:
            hout[k].copy_(outs[k], non_blocking=True)

    def timed(one, n):
        one(0)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        e0.record(stream)
        for i in range(n):
            one(i + 1)
        e1.record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        ms = max(e0.elapsed_time(e1), wall * 1e3)
        return aggregate(wl.rows_per_step() * n, ms, world)

    n = max(1, args.e2e_steps)
    rows, ms, value = timed(lambda i: calls(host, i), n)
    # host bytes the kernels read: the stats rows (copied to the device as
    # they are read; the accept walk and the sampler use the copies) and the
    # tree arrays
    h2d = (wl.stats_bytes(0, hout["acc"].numpy() if wl.early else None)
           + sum(host[k].numel() * host[k].element_size() for k in names if k not in ("vq", "dp")))
    in_bytes = sum(h.numel() * h.element_size() for h in host.values())

    devb = {k: torch.empty_like(rd[k]) for k in names}

    def copy_all(i):
        for k in names:
            devb[k].copy_(host[k], non_blocking=True)
        calls(devb, i)

    nc = max(1, min(n, 3))
    _, ms_c, value_c = timed(copy_all, nc)
    return {"value": value, "unit": "rows/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": d2h, "steps": n, "ms_per_step": ms / n,
            "inputs": f"page-locked host memory ({in_bytes / 1e9:.2f} GB per round), read in place",
            "copy_all": {"value": value_c, "unit": "rows/s", "h2d_bytes_per_step": in_bytes,
                         "d2h_bytes_per_step": d2h, "steps": nc, "ms_per_step": ms_c / nc}}


# ------------------------------------------------------------------ CPU oracle
def _rows_for_oracle(rd, ids, tree, maxd):
    """Float copies of the logit rows the oracle reads for sequences `ids`:
    every row of a chain; for a tree only the best path's nodes (the other
    rows stay zero and are never read), so marshalling stays cheap."""
    import torch
    tid = torch.as_tensor(ids)
    if not tree:
        return rd["vq"][tid].float().cpu().numpy(), rd["dp"][tid].float().cpu().numpy()
    import oracle
    k, T, V = len(ids), rd["vq"].shape[1], rd["vq"].shape[2]
    vq = np.zeros((k, T, V), np.float32)
    dp = np.zeros((k, T, V), np.float32)
    par = rd["parent"][tid].cpu().numpy()
    sc = rd["score"][tid].cpu().numpy()
    for j, b in enumerate(ids):
        nodes = torch.as_tensor(oracle.tree_best_path(par[j], sc[j], maxd).astype(np.int64))
        vq[j, nodes.numpy()] = rd["vq"][int(b)][nodes].float().cpu().numpy()
        dp[j, nodes.numpy()] = rd["dp"][int(b)][nodes].float().cpu().numpy()
    return vq, dp


def _oracle_job(cfg, rd, ids, step, early=False):
    """The oracle's inputs for the sequences `ids` of a pooled round, marshalled
    up front, and a function that runs the round on them: the tree (or chain)
    verify and, for trees, the in-place KV compaction of the sampled
    sequences' window (a KV buffer is passed in, one per thread).  Returns
    (rows covered, run)."""
    import oracle
    import torch
    tree = "parent" in rd
    vq, dp = _rows_for_oracle(rd, ids, tree, cfg.depth if tree else cfg.N)
    tid = torch.as_tensor(ids)
    if tree:
        par = rd["parent"][tid].cpu().numpy()
        tok = rd["token"][tid].cpu().numpy()
        sc = rd["score"][tid].cpu().numpy()

        def run(kv):
            o = oracle.verify_tree(vq, dp, par, tok, sc, cfg.depth, T=cfg.temperature, seed=1234,
                                   step=step, seq_ids=ids)
            oracle.tree_mask(par)
            if kv is not None:
                L, H, D, S, buf = kv
                nb = len(ids)
                base = np.zeros(nb, np.int32)
                oracle.kv_compact(buf, buf, L, nb, S, S, H, D, 2, base, base, o["path"],
                                  o["accept_len"] + 1)
    else:
        d = rd["d"][tid].cpu().numpy()

        def run(kv):
            oracle.verify_chain(vq, dp, d, T=cfg.temperature, seed=1234, step=step, seq_ids=ids,
                                early_exit=early)
    return len(ids) * vq.shape[1], run


def _oracle_round(cfg, rd, ids, step, kv=None, early=False):
    """One round of the oracle on the sequences `ids` (see _oracle_job).
    Returns (rows covered, seconds in the oracle)."""
    rows, run = _oracle_job(cfg, rd, ids, step, early)
    t0 = time.perf_counter()
    run(kv)
    return rows, time.perf_counter() - t0


def _kv_window(cfg, k, S):
    kvc = cfg.kv
    buf = np.random.default_rng(0).integers(0, 256, (kvc.L, 2, k, S, kvc.H, kvc.D * 2),
                                            dtype=np.uint8)
    return (kvc.L, kvc.H, kvc.D, S, buf)


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def cpu_baseline(args, wl, cfg, budget_s=10.0, cap_s=30.0, all_core_s=5.0):
    """The oracle on the host cores: groups of `--cpu-sample` sequences taken
    in turn from the pooled rounds (a new step number each group) until the
    oracle has run for `budget_s` seconds (at most `cap_s`), single-threaded;
    then the same kind of groups on every host core (one Python thread per
    core; the C oracle keeps no global state and ctypes releases the GIL
    during its calls) for about `all_core_s` seconds of wall time.
    Marshalling is outside both timings."""
    from concurrent.futures import ThreadPoolExecutor
    k = min(args.cpu_sample, wl.B)
    kv = _kv_window(cfg, k, wl.S) if wl.tree else None
    rows, secs, groups = 0, 0.0, 0

    def group(g):
        rd = wl.rounds[g % len(wl.rounds)]
        start = (g // len(wl.rounds)) * k % wl.B
        return rd, np.sort((start + np.arange(k)) % wl.B)

    while secs < budget_s and secs < cap_s:
        rd, ids = group(groups)
        r, t = _oracle_round(cfg, rd, ids, groups, kv, early=wl.early)
        rows += r
        secs += t
        groups += 1
    out = {"value": rows / secs, "unit": "rows/s", "cores": 1, "kind": "oracle",
           "sample": f"{groups} groups of {k} sequences from {len(wl.rounds)} rounds of "
                     f"config {cfg.index} ({cfg.name}); {rows} rows; single-threaded C "
                     f"oracle in double precision, {secs:.1f} s in the oracle"}
    # every core: one marshalled group per thread (its own KV window), run
    # over and over until the wall-clock budget is spent
    n = host_cores()
    jobs = [_oracle_job(cfg, *group(g), g, wl.early) for g in range(n)]
    kvs = [None] * n
    if wl.tree:
        kvc = cfg.kv
        kvs = [(kvc.L, kvc.H, kvc.D, wl.S,
                np.full((kvc.L, 2, k, wl.S, kvc.H, kvc.D * 2), 1, np.uint8)) for _ in range(n)]
    t0 = time.perf_counter()
    deadline = t0 + all_core_s

    def work(i):
        r, run = jobs[i]
        done = 0
        while time.perf_counter() < deadline:
            run(kvs[i])
            done += r
        return done

    with ThreadPoolExecutor(max_workers=n) as ex:
        rows_all = sum(ex.map(work, range(n)))
    wall = time.perf_counter() - t0
    ng = n
    out["all_cores"] = {"value": rows_all / wall, "unit": "rows/s", "cores": n,
                        "sample": f"{ng} groups of {k} sequences, one per thread on {n} "
                                  f"threads, each run repeatedly for {wall:.1f} s wall"}
    return out


def run_reference(args):
    """--impl reference: the CPU oracle as it stands, timed on the host cores,
    each step a bounded sample of the same workload."""
    import torch
    from speculative_decoding_verification_vocab_gb300 import synth
    rank, world, _ = dist_env()
    if rank != 0:
        return
    cfg = synth.CONFIGS[args.config]
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    if cfg.kind.startswith("tree"):
        vq, dp, parent, token, score = synth.tree_inputs(cfg, seed=1, device=dev)
        rd = dict(vq=vq, dp=dp, parent=parent, token=token, score=score)
    else:
        vq, dp, d = synth.chain_inputs(cfg, seed=1, device=dev)
        rd = dict(vq=vq, dp=dp, d=d)
    k = max(1, min(args.cpu_sample * 2, cfg.B))
    T = vq.shape[1]
    kv = _kv_window(cfg, k, T + 4) if cfg.kind.startswith("tree") else None
    for i in range(args.warmup):
        _oracle_round(cfg, rd, np.arange(i * k, (i + 1) * k) % cfg.B, i, kv)
    rows, secs = 0, 0.0
    for i in range(args.steps):
        ids = np.arange((args.warmup + i) * k, (args.warmup + i + 1) * k) % cfg.B
        r, s = _oracle_round(cfg, rd, np.sort(ids), args.warmup + i, kv)
        rows += r
        secs += s
    value = rows / secs
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * secs / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"config {cfg.index}: {cfg.name}", "B_per_gpu": cfg.B, "T": T,
                       "V": cfg.V},
            "cpu_baseline": {"value": value, "unit": "rows/s", "cores": 1, "kind": "oracle",
                             "sample": f"{k} sequences per step of config {cfg.index} "
                                       f"({cfg.name}), single-threaded C oracle"},
            "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def run_tree_build(args):
    """--tree-build: the EAGLE-2 dynamic tree of config 5 (B=128, depth 6,
    top-k 10, budget 60, V=128256 bf16) built on the GPU, one build per step:
    per level sv_tree_expand over the frontier's draft rows and sv_tree_select,
    then sv_tree_finalize.  The draft rows of every level are pre-generated
    (the draft model is out of scope), 4 distinct pools rotated."""
    import torch
    import speculative_decoding_verification_vocab_gb300 as sv
    from speculative_decoding_verification_vocab_gb300 import synth
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    sv.load_library()
    cfg = synth.CONFIGS[5]
    B, V, K, depth, Tn = cfg.B, cfg.V, cfg.topk, cfg.depth, cfg.T
    pools = []
    for r in range(args.pool):
        g = torch.Generator(device=dev).manual_seed(1000 + r)
        pools.append([(torch.randn((B, 1 if lvl == 1 else K, V), generator=g, device=dev) *
                       cfg.sigma_q).to(cfg.dtype) for lvl in range(1, depth + 1)])
    stream = torch.cuda.current_stream()

    def step(i):
        rows = pools[i % args.pool]
        return sv.build_tree(lambda lvl, f: rows[lvl - 1] if lvl <= depth else None, K, Tn,
                             cfg.temperature, stream)

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with Clocks(local) as clk:  # warm-up inside: the timing starts on warm clocks
        for i in range(args.warmup):
            step(i)
        torch.cuda.synchronize()
        n0 = sv.sv_launch_count()
        clk.region(True)
        e0.record(stream)
        for k in range(args.steps):
            step(k)
        e1.record(stream)
        torch.cuda.synchronize()
        clk.region(False)
    ms = e0.elapsed_time(e1)
    launches = sv.sv_launch_count() - n0
    sv.sv_trace_enable(True)
    for k in range(args.steps):
        step(k)
    torch.cuda.synchronize()
    sv.sv_trace_enable(False)
    trace = sv.sv_trace_collect()
    rows_per_build = B * (1 + K * (depth - 1))
    bytes_per_build = rows_per_build * V * 2
    ex_n, ex_ms = trace.get("tree_expand", (0, 0.0))
    per_level_bytes = bytes_per_build / depth
    peak, peak_kind = measured_peaks()
    ach = per_level_bytes / (ex_ms / max(ex_n, 1) / 1e3) / 1e9 if ex_n else None
    line = {
        "metric": "dynamic-tree builds/s (draft rows expanded per second)", "value":
        args.steps / (ms / 1e3), "unit": "builds/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "config 5 tree build: B=128, depth 6, top-k 10, budget 60, "
                               "V=128256 bf16", "draft_rows_per_build": rows_per_build,
                   "l2": f"draft rows rotate over {args.pool} pools of "
                         f"{bytes_per_build / 1e9:.2f} GB"},
        "draft_rows_per_s": rows_per_build * args.steps / (ms / 1e3),
        "kernels": {k: {"launches": v[0], "avg_us": 1e3 * v[1] / max(v[0], 1)}
                    for k, v in trace.items()},
        "gpu_launches": int(launches),
        "roofline": {"kernel": "tree_expand", "bound": "hbm", "achieved": ach, "peak": peak,
                     "unit": "GB/s", "frac": ach / peak if ach else None,
                     "peak_kind": f"{peak_kind} copy bandwidth",
                     "alg_bytes_per_launch": per_level_bytes,
                     "traffic": recorded_traffic("tree_expand", cfg.name)},
        "clocks": clk.summary(),
    }
    print(json.dumps(line))


def run_attention(args):
    """--attention: the tree-masked verifier attention of one layer for the
    dynamic-tree workload (B=128 trees of 60 nodes built over 6 levels, a
    70B-shaped layer: 64 query heads on 8 KV heads of 128, bf16, context 4096),
    one sv_tree_attention launch per step.  Every launch reads the 2.2 GB of
    keys and values (larger than L2)."""
    import torch
    import speculative_decoding_verification_vocab_gb300 as sv
    from speculative_decoding_verification_vocab_gb300 import synth
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    sv.load_library()
    B, T, Hq, Hkv, D, ctx = args.batch or 128, 60, 64, 8, 128, 4096
    S = ctx + 64
    q, kv, base = synth.attention_inputs(B, T, Hq, Hkv, D, S, ctx, seed=rank_seed(3, rank),
                                         device=dev)
    parent = synth.level_tree_parents(B, T, 6, seed=rank_seed(3, rank)).to(dev)
    mask, depth = sv.tree_build_mask(parent)
    out = torch.empty_like(q)
    lse = torch.empty(B, T, Hq, dtype=torch.float32, device=dev)
    status = torch.zeros(B, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    scale = D ** -0.5

    def step():
        sv.sv_tree_attention(q, kv, base, mask, scale, out, lse, status, stream)

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with Clocks(local) as clk:  # warm-up inside: the timing starts on warm clocks
        for _ in range(max(args.warmup, 3)):
            step()
        torch.cuda.synchronize()
        n0 = sv.sv_launch_count()
        clk.region(True)
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        clk.region(False)
    ms = e0.elapsed_time(e1) / args.steps
    launches = sv.sv_launch_count() - n0
    assert int(torch.count_nonzero(status)) == 0
    # algorithmic work: every (node, query head) row against its visible keys
    vis = (base.double()[:, None] + depth.double() + 1.0).sum().item() * Hq
    flops = 4.0 * D * vis
    kv_bytes = 2.0 * (base.double() + T).sum().item() * Hkv * D * 2
    io_bytes = kv_bytes + 2.0 * q.numel() * 2 + lse.numel() * 4
    d = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) \
        if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")) else None
    # a timed region of more than half a second is sustained load: the
    # sustained bf16 figure (the part settles under its power cap), else burst
    sustained = ms * args.steps > 500.0
    if d:
        peak = float(d["bf16_tflops_sustained"] if sustained else d["bf16_tflops"])
        kind = "measured" + (" sustained" if sustained else " burst")
    else:
        peak, kind = (1700.0, "fallback sustained") if sustained else (1900.0, "fallback burst")
    hbm, _ = measured_peaks()
    ach = flops / (ms / 1e3) / 1e12
    line = {
        "metric": "tree-attention verifier rows/s (one layer)", "value":
        B * T * Hq / (ms / 1e3), "unit": "query rows/s", "n_gpus": 1, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "tree attention, dynamic-tree shape: B=%d, T=60 (6 levels), "
                               "Hq=64, Hkv=8, D=128, context 4096, bf16" % B,
                   "l2": "inputs larger than L2: %.2f GB of keys and values per launch"
                         % (kv_bytes / 1e9)},
        "tflops": ach, "hbm_gbs": io_bytes / (ms / 1e3) / 1e9,
        "hbm_frac_measured": io_bytes / (ms / 1e3) / 1e9 / hbm,
        "gpu_launches": int(launches),
        "roofline": {"kernel": "tree_attention", "bound": "tensor", "achieved": ach,
                     "peak": peak, "unit": "TFLOP/s", "frac": ach / peak,
                     "peak_kind": f"{kind} bf16 dense",
                     "alg_flops_per_launch": flops,
                     "traffic": recorded_traffic("tree_attention", "dynamic_eagle2_tree")},
        "clocks": clk.summary(),
    }
    print(json.dumps(line))


def main():
    args = parse()
    if args.steps is None:
        args.steps = 20 if args.impl == "reference" else 1000
    if args.impl == "reference":
        run_reference(args)
    elif args.tree_build:
        run_tree_build(args)
    elif args.attention:
        run_attention(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
