#!/usr/bin/env python
"""Benchmark of split tree attention (verification attention of tree
speculative decoding) on one or more GPUs of one node.

A step is one pass of the whole hot path over one batch through the C ABI:
the ancestor bitmasks of the draft tree, the prefix pass split over the paged
KV cache, the tree-masked suffix pass and the log-sum-exp merge.  With the
default layout it is one tree_attn_verify_tree call (the masks are built
inside the suffix/merge kernel); --layout paged_tree / full_mask call
tree_mask_build first.

    python bench.py [--config chain] [--steps K] [--warmup W]
    python -m torch.distributed.run --nproc-per-node N bench.py --gpus N ...
    python bench.py --impl reference     # the fp64 CPU oracle, timed alone

Prints one JSON line (rank 0).  ``value`` is verified tree tokens per second
over all ranks (B*T tokens per step and rank; each rank runs an independent
replica, so scaling is weak).  Inputs stay resident in HBM during the timed
region; the KV cache is replicated R times on the device and the steps rotate
through the replicas so that every step reads K/V that is not in L2
(R * KV bytes >= 4 x L2).  The timed steps are replayed from one CUDA graph.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

_ROOT = os.path.dirname(os.path.abspath(__file__))
if _ROOT not in sys.path:
    sys.path.insert(0, _ROOT)

from workloads import CONFIGS, make_workload  # noqa: E402

METRIC = "verified tree tokens/s per layer"
# kernels one step launches, per layout
LAUNCHES_PER_STEP = {"shared": 2, "per_seq": 2, "paged_tree": 3, "full_mask": 4}
UNIT = "tokens/s"
FALLBACK_HBM_GBS = 6800.0

# dram__bytes_read.sum + dram__bytes_write.sum per launch of the prefix-pass
# kernel from an ncu capture, keyed by workload, valid only for the kernel
# source whose SHA-256 is recorded with it (see profiles/).
NCU_TRAFFIC = {
    # profiles/prefix_pass_traffic_long_context.md
    "chain": ("f88e1f9741214b41", 2376858624),
    "maverick": ("f88e1f9741214b41", 540920576),
    "llama70b": ("f88e1f9741214b41", 338890496),
    "llama8b": ("f88e1f9741214b41", 33741824),
}


def parse_args():
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--config", choices=sorted(CONFIGS), default="chain",
                   help="headline workload (default: the largest single-GPU one, the "
                        "64-sequence chain)")
    p.add_argument("--layout", choices=["shared", "per_seq", "paged_tree", "full_mask"],
                   default="shared",
                   help="shared: one draft tree for the batch, tree K/V in their own buffers; "
                        "per_seq: one tree per sequence; paged_tree: tree K/V padded into the "
                        "paged cache at positions L_b + j; full_mask: the one-pass ablation "
                        "(paged_tree layout, explicit [B][T][L+T] mask, no split into prefix "
                        "and tree passes)")
    p.add_argument("--path", choices=["verify", "accept_commit"], default="verify",
                   help="verify: the split tree attention step (default); accept_commit: "
                        "greedy acceptance of the verified tree plus the KV commit of the "
                        "accepted path (tree tokens in the paged cache)")
    p.add_argument("--cpu-seconds", type=float, default=10.0,
                   help="bound on the CPU-baseline sample (oracle wall time)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-clocks", action="store_true")
    p.add_argument("--no-early", action="store_true",
                   help="leave the prefix pass's early start off (default: on; the step's "
                        "kernel before each call writes no prefix input)")
    p.add_argument("--no-long-context", action="store_true",
                   help="time only --config (default: also every other long-context "
                        "workload, reported under long_context)")
    return p.parse_args()


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------
def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def measured_hbm_peak():
    path = os.path.join(_ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured (MEASURED_PEAKS.json hbm_gbs)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_sha():
    """SHA-256 prefix of the device sources the prefix-pass kernel is built from,
    with comments and whitespace removed (a comment edit does not make a traffic
    record stale; any code change does)."""
    import hashlib
    import re
    h = hashlib.sha256()
    for name in ("kernels.cu", "prefix_early.cu", "layout.h", "ptx.cuh"):
        with open(os.path.join(_ROOT, "speculative_decoding_tree_split_gb300", "csrc", name),
                  encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def workload_desc(cfg, layout="shared"):
    return cfg.describe() + ("" if layout == "shared" else f" layout={layout}")


def make_layout_workload(cfg, layout, seed=None):
    return make_workload(cfg, seed=seed, per_sequence_trees=(layout == "per_seq"),
                         tree_in_cache=(layout in ("paged_tree", "full_mask")))


def algorithmic_bytes(wl):
    """Bytes one verify call must move (prefix K/V dominates)."""
    c = wl.cfg
    kv = wl.kv_bytes()
    q = c.B * c.T * c.Hq * c.d * 2
    tree = c.B * c.T * c.Hkv * c.d * 2 * 2
    out = c.B * c.T * c.Hq * c.d * 2
    lse = c.B * c.T * c.Hq * 4
    tables = wl.block_table.numel() * 4 + c.B * 4 + c.T * 8 + c.T * 4
    return {"kv": kv, "prefix_kernel": kv + q, "call": kv + q + tree + out + lse + tables}


class ClockSampler:
    """nvidia-smi clocks sampled every 200 ms while the GPU is loaded."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k] == "Active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def smi_gpu_id(props, local):
    """An nvidia-smi -i selector for this process's GPU."""
    uuid = getattr(props, "uuid", None)
    if uuid:
        u = str(uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    ids = [x for x in vis.split(",") if x.strip()]
    if local < len(ids):
        return ids[local].strip()
    return str(local)


def max_over_ranks(values, device=None):
    """Element-wise maximum of `values` over all ranks (identity when not
    distributed); the device follows the process group's backend."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    if device is None:
        device = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def emit(obj):
    print(json.dumps(obj), flush=True)


# ---------------------------------------------------------------------------
# CPU side: the fp64 oracle (baseline leg and the reference arm)
# ---------------------------------------------------------------------------
def oracle_token_fn(wl, layout="shared", threads=None):
    """f(b, i): the oracle on one tree token (all Hq query heads of sequence b,
    node i), with sequence b's own tree mask (the one-pass oracle under the
    explicit mask for the full_mask layout).  threads: the oracle's OpenMP
    threads (default: every core this process may run on)."""
    import oracle
    orc = oracle.get()
    c = wl.cfg
    if threads is None:
        threads = len(os.sched_getaffinity(0))
    if layout == "full_mask":
        from oracle.dense import dense_mask
        tm = orc.tree_mask(wl.parents.tolist())
        cols = int(wl.seq_lens.max()) + c.T
        dense, key_lens = dense_mask(tm, wl.seq_lens.numpy(), c.T, cols)

        def f_dense(b, i):
            rows = np.array([(b, i, h) for h in range(c.Hq)], dtype=np.int32)
            orc.dense_rows(wl, key_lens, dense, rows)

        return f_dense, 1
    if wl.parents.dim() == 2:
        seqs = [wl.sequence(b) for b in range(c.B)]
        masks = [orc.tree_mask(s.parents.tolist()) for s in seqs]
    else:
        seqs, masks = None, orc.tree_mask(wl.parents.tolist())

    def f(b, i):
        if seqs is None:
            rows = np.array([(b, i, h) for h in range(c.Hq)], dtype=np.int32)
            orc.verify_rows(wl, masks, rows, threads=threads)
        else:
            rows = np.array([(0, i, h) for h in range(c.Hq)], dtype=np.int32)
            orc.verify_rows(seqs[b], masks[b], rows, threads=threads)

    return f, threads


def oracle_tokens_per_s(wl, budget_s, max_tokens=None, layout="shared", threads=None):
    """Time the oracle on whole tree tokens (all Hq heads of one (b, i)),
    round-robin over the batch, until `budget_s` of wall time is spent."""
    c = wl.cfg
    f, threads = oracle_token_fn(wl, layout, threads)
    tokens = [(b, i) for b in range(c.B) for i in range(c.T)]
    done = 0
    t0 = time.perf_counter()
    while True:
        f(*tokens[done % len(tokens)])
        done += 1
        el = time.perf_counter() - t0
        if el >= budget_s or (max_tokens is not None and done >= max_tokens):
            break
    return done / el, done, el, threads


def run_reference(args):
    world, rank, _ = dist_info()
    if rank != 0:
        return
    cfg = CONFIGS[args.config]
    wl = make_layout_workload(cfg, args.layout)
    f, threads = oracle_token_fn(wl, args.layout)
    tokens = [(b, i) for b in range(cfg.B) for i in range(cfg.T)]

    def step(n):
        f(*tokens[n % len(tokens)])

    for n in range(args.warmup):
        step(n)
    t0 = time.perf_counter()
    for n in range(args.steps):
        step(args.warmup + n)
    el = time.perf_counter() - t0
    value = args.steps / el
    emit({"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
          "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
          "ms_per_step": 1e3 * el / args.steps, "higher_is_better": True, "scaling": "weak",
          "vs_baseline": None, "dtype": "f64", "data": "synthetic",
          "config": {"workload": workload_desc(cfg, args.layout)},
          "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                           "sample": f"each step = one tree token (all {cfg.Hq} query heads of "
                                     f"one (sequence, node)) of the workload, round-robin"},
          "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                  "d2h_bytes_per_step": 0}})


# ---------------------------------------------------------------------------
# GPU side
# ---------------------------------------------------------------------------
# Workloads whose prefix pass the >= 70 %-of-HBM target is defined on (the
# 70B layer is reported beside them); each is timed in the same run as the
# headline workload.
LONG_CONTEXT = ("llama8b", "llama70b", "chain", "maverick")


class StepBench:
    """Device state and CUDA graphs of one workload: `step` is one pass of
    the whole hot path, `prefix_only` the prefix-pass kernel alone."""

    def __init__(self, ta, cfg, layout, dev, seed, K, W):
        self.ta, self.cfg, self.layout, self.dev, self.K, self.W = ta, cfg, layout, dev, K, W
        wl = make_layout_workload(cfg, layout, seed=seed)
        self.wl = wl
        props = torch.cuda.get_device_properties(dev)
        self.l2 = int(getattr(props, "L2_cache_size", 0) or 0) or 132 * 1024 * 1024
        self.kv_alloc = wl.k_pages.numel() * 2 * 2
        R = max(2, math.ceil(4 * self.l2 / max(self.kv_alloc, 1)))
        self.R = R
        # resident inputs
        self.parents = wl.parents.to(dev)
        self.q = wl.q.to(dev)
        self.bt = wl.block_table.to(dev)
        self.sl = wl.seq_lens.to(dev)
        self.tk = wl.tree_k.to(dev)
        self.tv = wl.tree_v.to(dev)
        self.kps = [wl.k_pages.to(dev) for _ in range(R)]
        self.vps = [wl.v_pages.to(dev) for _ in range(R)]
        self.mask = torch.empty(tuple(wl.parents.shape), dtype=torch.int64, device=dev)
        self.out = torch.empty_like(self.q)
        self.lse = torch.empty(cfg.B, cfg.T, cfg.Hq, dtype=torch.float32, device=dev)
        ws_bytes = ta.workspace_size(cfg.B, cfg.Hq, cfg.Hkv, cfg.d, cfg.T, 0, cfg.page)
        self.ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        if layout == "full_mask":
            self.cols = ta.dense_cols_for(int(wl.seq_lens.max()) + cfg.T)
            self.dense = torch.empty((cfg.B, cfg.T, self.cols), dtype=torch.uint8, device=dev)
            self.key_lens = torch.empty(cfg.B, dtype=torch.int32, device=dev)

    def hot_path(self, par, q_, k_, v_, bt_, sl_, tk_, tv_):
        """One pass of the whole path: masks, then tree attention."""
        ta, cfg, wl = self.ta, self.cfg, self.wl
        layout, mask, out, lse, ws, status = (self.layout, self.mask, self.out, self.lse,
                                              self.ws, self.status)
        if layout == "full_mask":
            ta.mask_build(par, mask_out=mask, status=status)
            ta.dense_mask_build(mask, sl_, cfg.T, self.cols, dense_out=self.dense,
                                key_lens=self.key_lens, status=status)
            ta.verify_dense(q_, k_, v_, bt_, self.key_lens, self.dense, out=out, lse=lse,
                            workspace=ws, status=status, softmax_scale=wl.scale)
        elif layout == "paged_tree":
            ta.mask_build(par, mask_out=mask, status=status)
            ta.verify_paged_tree(q_, k_, v_, bt_, sl_, mask, out=out, lse=lse, workspace=ws,
                                 status=status, softmax_scale=wl.scale)
        else:
            # shared / per_seq: tree_mask_build + tree_attn_verify in one call
            # (tree_attn_verify_tree): the ancestor masks are built inside the
            # attention kernels and written out
            ta.verify_tree(q_, k_, v_, bt_, sl_, tk_, tv_, par, mask_out=mask, out=out, lse=lse,
                           workspace=ws, status=status, softmax_scale=wl.scale)

    def step(self, r):
        self.hot_path(self.parents, self.q, self.kps[r % self.R], self.vps[r % self.R], self.bt,
                      self.sl, self.tk, self.tv)

    def prefix_only(self, r):
        ta, wl = self.ta, self.wl
        k_, v_ = self.kps[r % self.R], self.vps[r % self.R]
        if self.layout == "full_mask":   # the one-pass kernel has no separate entry
            ta.verify_dense(self.q, k_, v_, self.bt, self.key_lens, self.dense, out=self.out,
                            lse=self.lse, workspace=self.ws, status=self.status,
                            softmax_scale=wl.scale)
            return
        ta.prefix_pass(self.q, k_, v_, self.bt, self.sl, self.ws, status=self.status,
                       softmax_scale=wl.scale)

    def prepare(self):
        """Eager warm-up (also applies the kernels' shared-memory opt-in before
        capture), then the CUDA graphs; each graph is launched once, untimed:
        a graph's first launch uploads it to the device."""
        side = torch.cuda.Stream(self.dev)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for r in range(max(self.W, 1)):
                self.step(r)
                self.prefix_only(r)
        torch.cuda.synchronize()
        self.check_status("warm-up")

        def capture(fn, n):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for r in range(n):
                    fn(r)
            return g

        self.g_timed = capture(self.step, self.K)
        self.g_warm = capture(self.step, max(self.W, 1))
        self.g_prefix = capture(self.prefix_only, self.K)
        self.g_timed.replay()
        self.g_prefix.replay()
        torch.cuda.synchronize()

    def check_status(self, where):
        if int(self.status.item()) != 0:
            raise RuntimeError(f"{self.cfg.name}: device status {int(self.status.item())} "
                               f"during {where}")

    def warm(self, seconds):
        """W warm-up steps, then replays for about `seconds` (clocks settle and
        the sampler sees the GPU under load)."""
        self.g_warm.replay()
        t_end = time.perf_counter() + seconds
        while time.perf_counter() < t_end:
            self.g_warm.replay()
            torch.cuda.synchronize()


def timed_replay(graph, barrier):
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier()
    s.record()
    graph.replay()
    e.record()
    torch.cuda.synchronize()
    barrier()
    return s.elapsed_time(e)


def traffic_for(name, layout, sha):
    rec = NCU_TRAFFIC.get(name) if layout == "shared" else None
    return rec[1] if rec is not None and rec[0] == sha else None


def run_ours(args):
    import speculative_decoding_tree_split_gb300 as ta

    world, rank, local = dist_info()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ta.build()
    ta.load()
    # The kernel before each timed call is the previous call's last kernel,
    # which writes no seq_lens, block table or prefix K/V: the promise the
    # early start needs holds (captured into the graphs below).
    ta.set_early_prefix_loads(not args.no_early)

    cfg = CONFIGS[args.config]
    layout = args.layout
    K, W = args.steps, args.warmup
    main = StepBench(ta, cfg, layout, dev, cfg.seed + rank, K, W)
    main.prepare()
    # The other long-context workloads, timed in the same run (one layout and
    # one K for all, so the figures compare).
    others = []
    if not args.no_long_context and args.path == "verify":
        for name in LONG_CONTEXT:
            if name != args.config:
                b = StepBench(ta, CONFIGS[name], layout, dev, CONFIGS[name].seed + rank, K, W)
                b.prepare()
                others.append(b)
    props = torch.cuda.get_device_properties(dev)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    # clocks are sampled from the first warm-up replay to the last timed one
    sampler = ClockSampler(smi_gpu_id(props, local))
    if not args.no_clocks:
        sampler.start()
    main.warm(0.0 if args.no_clocks else 1.2)
    ms_total = timed_replay(main.g_timed, barrier)
    ms_prefix_total = timed_replay(main.g_prefix, barrier)
    other_ms = []
    for b in others:
        b.warm(0.0 if args.no_clocks else 0.3)
        other_ms.append((timed_replay(b.g_timed, barrier), timed_replay(b.g_prefix, barrier)))
    clocks = sampler.stop() if not args.no_clocks else None
    main.check_status("the timed region")
    for b in others:
        b.check_status("the timed region")

    ms_step = ms_total / K
    ms_prefix = ms_prefix_total / K
    ms_step, ms_prefix = max_over_ranks([ms_step, ms_prefix], dev)
    # Run-to-run spread: the same K-step graph replayed five more times, each
    # timed alone.  Reported beside `value`, which is the one timed region above.
    reps = sorted(max_over_ranks([timed_replay(main.g_timed, barrier) / K for _ in range(5)],
                                 dev))
    spread = {"replays": len(reps), "us_per_step_min": reps[0] * 1e3,
              "us_per_step_median": reps[len(reps) // 2] * 1e3, "us_per_step_max": reps[-1] * 1e3}
    tokens_per_step = cfg.B * cfg.T * world
    value = tokens_per_step / (ms_step * 1e-3)

    nbytes = algorithmic_bytes(main.wl)
    peak, peak_src = measured_hbm_peak()
    achieved = nbytes["prefix_kernel"] / (ms_prefix * 1e-3) / 1e9
    sha = kernel_source_sha()
    traffic = traffic_for(args.config, layout, sha)

    def long_context_entry(b, ms_s, ms_p):
        nb = algorithmic_bytes(b.wl)
        c = b.cfg
        gbs = nb["prefix_kernel"] / (ms_p * 1e-3) / 1e9
        call_gbs = nb["kv"] / (ms_s * 1e-3) / 1e9
        return {"workload": workload_desc(c, layout), "us_per_call": ms_s * 1e3,
                "tokens_per_s": c.B * c.T * world / (ms_s * 1e-3),
                "prefix_kernel_us": ms_p * 1e3, "prefix_gbs": gbs,
                "prefix_frac_of_measured": gbs / peak, "prefix_frac_of_8tbs": gbs / 8000.0,
                "call_kv_gbs": call_gbs, "call_frac_of_measured": call_gbs / peak,
                "algorithmic_bytes_per_prefix_launch": nb["prefix_kernel"],
                "traffic": traffic_for(c.name, layout, sha)}

    long_context = None
    if others:
        long_context = {args.config: long_context_entry(main, ms_step, ms_prefix)}
        for b, (ms_s, ms_p) in zip(others, other_ms):
            ms_s, ms_p = max_over_ranks([ms_s / K, ms_p / K], dev)
            long_context[b.cfg.name] = long_context_entry(b, ms_s, ms_p)
    for b in others:   # free their device memory before the end-to-end leg
        del b.kps, b.vps
    others.clear()
    torch.cuda.empty_cache()

    # end to end through the public API: pinned host inputs -> device, the
    # step, out/lse -> pinned host, every step
    e2e = None
    wl = main.wl
    if not args.no_e2e:
        host = dict(parents=wl.parents, q=wl.q, k=wl.k_pages, v=wl.v_pages, bt=wl.block_table,
                    sl=wl.seq_lens, tk=wl.tree_k, tv=wl.tree_v)
        d = dict(parents=main.parents, q=main.q, k=main.kps[0], v=main.vps[0], bt=main.bt,
                 sl=main.sl, tk=main.tk, tv=main.tv)
        if layout in ("paged_tree", "full_mask"):   # the tree K/V travel inside the pages
            del host["tk"], host["tv"]
        h = {k: v.pin_memory() for k, v in host.items()}
        h_out = torch.empty(main.out.shape, dtype=main.out.dtype).pin_memory()
        h_lse = torch.empty(main.lse.shape, dtype=main.lse.dtype).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in h.values())
        d2h = h_out.numel() * 2 + h_lse.numel() * 4
        n_e2e = max(3, min(K, int(20e9 // max(h2d, 1))))

        def e2e_step():
            for key in h:
                d[key].copy_(h[key], non_blocking=True)
            main.hot_path(d["parents"], d["q"], d["k"], d["v"], d["bt"], d["sl"], d["tk"],
                          d["tv"])
            h_out.copy_(main.out, non_blocking=True)
            h_lse.copy_(main.lse, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        barrier()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(n_e2e):
            e2e_step()
        e.record()
        torch.cuda.synchronize()
        ms_e2e = s.elapsed_time(e) / n_e2e
        ms_e2e = max_over_ranks([ms_e2e], dev)[0]
        e2e = {"value": tokens_per_step / (ms_e2e * 1e-3), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n_e2e,
               "ms_per_step": ms_e2e}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, n_tok, el, threads = oracle_tokens_per_s(wl, args.cpu_seconds, layout=layout)
        # the same on one core, for a third of the time
        v1, n1, el1, _ = oracle_tokens_per_s(wl, args.cpu_seconds / 3, layout=layout, threads=1)
        cpu = {"value": v, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"{n_tok} tree tokens (all {cfg.Hq} query heads each) of this "
                         f"workload, round-robin, {el:.1f} s of fp64 oracle time",
               "value_1_core": v1,
               "sample_1_core": f"{n1} tree tokens, {el1:.1f} s, one thread"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": W, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": workload_desc(cfg, layout),
                       "tokens_per_step_per_gpu": cfg.B * cfg.T,
                       "l2": f"{main.R} rotating device copies of the KV cache "
                             f"({main.R * main.kv_alloc / 2**20:.0f} MiB > L2 "
                             f"{main.l2 / 2**20:.0f} MiB)",
                       "parallelism": f"replicas x{world}", "timing": "one CUDA graph of the "
                       "K steps, CUDA events on the replay stream",
                       "early_prefix_loads": not args.no_early},
            "us_per_call": ms_step * 1e3,
            "call_hbm_gbs": nbytes["call"] / (ms_step * 1e-3) / 1e9,
            "prefix_kernel_us": ms_prefix * 1e3,
            "roofline": {"bound": "hbm",
                         "kernel": "prefix_pass_kernel" if layout != "full_mask" else
                         "prefix_pass_kernel (explicit mask) + merge, timed together",
                         "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "algorithmic_bytes_per_launch": nbytes["prefix_kernel"],
                         "peak_source": peak_src, "kernel_sha": sha},
            "clocks": clocks, "e2e": e2e,
            "gpu_launches": LAUNCHES_PER_STEP[layout] * K,
            "cpu_baseline": cpu, "spread": spread,
        }
        if long_context is not None:
            line["long_context"] = long_context
        emit(line)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# the step after verification: greedy acceptance + KV commit
# ---------------------------------------------------------------------------
ACCEPT_METRIC = "committed sequences/s per layer"
ACCEPT_UNIT = "sequences/s"


def accept_inputs(cfg, seed):
    """Per-sequence trees with the tree tokens in the paged cache, plus draft
    and target tokens from a 2-token alphabet (about half the edges match, so
    paths of several nodes are common)."""
    wl = make_workload(cfg, seed=seed, per_sequence_trees=True, tree_in_cache=True)
    g = torch.Generator().manual_seed(1000 + seed)
    draft = torch.randint(0, 2, (cfg.B, cfg.T), generator=g, dtype=torch.int32)
    target = torch.randint(0, 2, (cfg.B, cfg.T), generator=g, dtype=torch.int32)
    return wl, draft, target


def oracle_accept_commit_per_s(wl, draft, target, budget_s, steps=None):
    """Time the acceptance / commit oracle on the whole batch, step after step."""
    from workloads import bf16_bits
    import oracle.accept as acc
    k = bf16_bits(wl.k_pages)
    v = bf16_bits(wl.v_pages)
    bt = wl.block_table.numpy()
    sl = wl.seq_lens.numpy()
    par, dr, tg = wl.parents.numpy(), draft.numpy(), target.numpy()
    done = 0
    t0 = time.perf_counter()
    while True:
        n, path, _ = acc.greedy_accept_batch(par, dr, tg)
        acc.kv_commit(k, v, bt, sl, None, None, path, n, wl.cfg.page)
        done += 1
        el = time.perf_counter() - t0
        if (steps is not None and done >= steps) or (steps is None and el >= budget_s):
            break
    return done * wl.cfg.B / el, done, el


def run_accept_commit(args):
    import speculative_decoding_tree_split_gb300 as ta

    world, rank, local = dist_info()
    cfg = CONFIGS[args.config]
    if args.impl == "reference":
        if rank != 0:
            return
        wl, draft, target = accept_inputs(cfg, cfg.seed)
        oracle_accept_commit_per_s(wl, draft, target, 0, steps=max(args.warmup, 1))
        v, n_steps, el = oracle_accept_commit_per_s(wl, draft, target, 0, steps=args.steps)
        emit({"impl": "reference", "metric": ACCEPT_METRIC, "value": v, "unit": ACCEPT_UNIT,
              "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
              "ms_per_step": 1e3 * el / n_steps, "higher_is_better": True, "scaling": "weak",
              "vs_baseline": None, "dtype": "int32", "data": "synthetic",
              "config": {"workload": workload_desc(cfg, "paged_tree") + " path=accept_commit"},
              "cpu_baseline": {"value": v, "unit": ACCEPT_UNIT, "cores": 1, "kind": "oracle",
                               "sample": f"{n_steps} whole steps"},
              "e2e": {"value": v, "unit": ACCEPT_UNIT, "h2d_bytes_per_step": 0,
                      "d2h_bytes_per_step": 0}})
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ta.build()
    ta.load()
    wl, draft, target = accept_inputs(cfg, cfg.seed + rank)
    parents = wl.parents.to(dev)
    d_draft, d_target = draft.to(dev), target.to(dev)
    k, v = wl.k_pages.to(dev), wl.v_pages.to(dev)
    bt, sl = wl.block_table.to(dev), wl.seq_lens.to(dev)
    B, T = cfg.B, cfg.T
    masks = torch.empty((B, T), dtype=torch.int64, device=dev)
    n = torch.empty(B, dtype=torch.int32, device=dev)
    path = torch.empty((B, T), dtype=torch.int32, device=dev)
    bonus = torch.empty(B, dtype=torch.int32, device=dev)
    sl_out = torch.empty(B, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ta.mask_build_batched(parents, mask_out=masks, status=status)

    def accept_only(_r=0):
        ta.greedy_accept(masks, d_draft, d_target, accept_len=n, accept_path=path,
                         bonus_token=bonus)

    def commit_only(_r=0):
        ta.kv_commit(k, v, bt, sl, path, n, seq_lens_out=sl_out, status=status)

    def step(_r=0):
        # greedy acceptance and the commit in one launch (tree_accept_commit)
        ta.accept_commit(masks, d_draft, d_target, k, v, bt, sl, accept_len=n, accept_path=path,
                         bonus_token=bonus, seq_lens_out=sl_out, status=status)

    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(max(args.warmup, 1)):
            step()
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} during warm-up")
    K = args.steps

    def graph_of(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(K):
                fn()
        return g

    def timed(g):
        s_, e_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        s_.record()
        g.replay()
        e_.record()
        torch.cuda.synchronize()
        return s_.elapsed_time(e_) / K

    g_step, g_acc, g_com = graph_of(step), graph_of(accept_only), graph_of(commit_only)
    # first launches upload the graphs; keep that out of the timed replays
    g_step.replay()
    g_acc.replay()
    g_com.replay()
    sampler = ClockSampler(smi_gpu_id(torch.cuda.get_device_properties(dev), local))
    if not args.no_clocks:
        sampler.start()
        t_end = time.perf_counter() + 1.2
        while time.perf_counter() < t_end:
            g_step.replay()
            torch.cuda.synchronize()
    ms_step = timed(g_step)
    ms_acc = timed(g_acc)
    ms_com = timed(g_com)
    clocks = sampler.stop() if not args.no_clocks else None
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in the timed region")
    ms_step, ms_acc, ms_com = max_over_ranks([ms_step, ms_acc, ms_com], dev)
    n_h = n.cpu()
    rows = int(n_h.sum().item())
    commit_bytes = rows * cfg.Hkv * cfg.d * 2 * 2 * 2   # K and V rows, read + write
    peak, peak_src = measured_hbm_peak()
    achieved = commit_bytes / (ms_step * 1e-3) / 1e9

    e2e = None
    if not args.no_e2e:
        h_draft, h_target = draft.pin_memory(), target.pin_memory()
        h_n = torch.empty(B, dtype=torch.int32).pin_memory()
        h_bonus = torch.empty(B, dtype=torch.int32).pin_memory()
        h2d = 2 * B * T * 4
        d2h = 2 * B * 4

        def e2e_step():
            d_draft.copy_(h_draft, non_blocking=True)
            d_target.copy_(h_target, non_blocking=True)
            step()
            h_n.copy_(n, non_blocking=True)
            h_bonus.copy_(bonus, non_blocking=True)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        s_, e_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s_.record()
        for _ in range(K):
            e2e_step()
        e_.record()
        torch.cuda.synchronize()
        ms_e2e = max_over_ranks([s_.elapsed_time(e_) / K], dev)[0]
        e2e = {"value": B * world / (ms_e2e * 1e-3), "unit": ACCEPT_UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        vcpu, n_steps, el = oracle_accept_commit_per_s(wl, draft, target, args.cpu_seconds)
        cpu = {"value": vcpu, "unit": ACCEPT_UNIT, "cores": 1, "kind": "oracle",
               "sample": f"{n_steps} whole steps ({el:.1f} s)"}
    if rank == 0:
        emit({
            "metric": ACCEPT_METRIC, "value": B * world / (ms_step * 1e-3), "unit": ACCEPT_UNIT,
            "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32",
            "data": "synthetic",
            "config": {"workload": workload_desc(cfg, "paged_tree") + " path=accept_commit",
                       "l2": "inputs are a few KB and stay in L2 (latency-bound step)",
                       "accepted_rows_per_step": rows,
                       "timing": "one CUDA graph of the K steps, CUDA events"},
            "separate_accept_kernel_us": ms_acc * 1e3, "separate_commit_kernel_us": ms_com * 1e3,
            "roofline": {"bound": "hbm", "kernel": "accept_commit_kernel", "achieved": achieved,
                         "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "traffic": None, "algorithmic_bytes_per_launch": commit_bytes,
                         "peak_source": peak_src,
                         "note": "latency-bound: a few KB per launch"},
            "clocks": clocks, "e2e": e2e, "gpu_launches": K, "cpu_baseline": cpu,
        })
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    args = parse_args()
    if args.path == "accept_commit":
        run_accept_commit(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
