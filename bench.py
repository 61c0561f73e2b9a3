"""Benchmark: GDN tree-verify nodes/s per layer on one GB300, with the
roofline fraction of the dominant kernel and the fp64 CPU oracle as a
reported baseline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one decoding iteration of the whole path over one batch: the
delayed commitment of the previous tree's accepted path and the verification
of every node of the next tree, as one gdn_tree_commit_verify call (state
buffers and U buffers ping-pong between steps).  The same work done as the two
separate calls (gdn_tree_verify, then gdn_tree_commit) is timed as well and
reported under "separate_calls".  The workload is the serving-scale case: 32
sequences x 32 v-heads (16 q/k heads), dk = dv = 128, bf16 q/k/v, fp32 state,
128-node random trees (branching 1-4, depth <= 24), accepted paths of up to 24
nodes.  L2 is flushed (a 256 MiB write) before every timed step, outside the
timed events.  Under torchrun each rank runs its own independent batch (weak
scaling, no collective on the data path) and rank 0 prints one JSON line.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "GDN tree-verify nodes/sec per layer on 1 GB300; % of HBM/tensor roofline"
UNIT = "nodes/s"
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, nominal (context beside the measured peak)
WORKLOAD_CFG = 3
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "verify_traffic.json")
KERNEL_SOURCES = [os.path.join(ROOT, "gated_deltanet_tree_gdn_gb300", "csrc", f)
                  for f in ("verify_generic.cu", "verify_tc.cu", "common.cuh", "sm100.cuh")]


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ---------------------------------------------------------------------------
# byte / FLOP model (per launch)
# ---------------------------------------------------------------------------

def verify_bytes(w: W.Workload) -> int:
    es = 2 if w.dtype == W.BF16 else 4
    B, N, Hqk, Hv, dk, dv = w.B, w.N, w.Hqk, w.Hv, w.dk, w.dv
    return (B * Hv * dk * dv * 4            # S0 read
            + 2 * B * N * Hqk * dk * es     # q, k read (once per q/k head)
            + B * N * Hv * dv * es          # v read
            + 2 * B * N * Hv * 4            # log_alpha, beta read
            + B * N * 4                     # parent read
            + B * N * Hv * dv * es          # o write
            + B * Hv * N * dv * 4)          # U write


def commit_bytes(w: W.Workload) -> int:
    es = 2 if w.dtype == W.BF16 else 4
    Lsum = int(w.path_len.sum())
    return (2 * w.B * w.Hv * w.dk * w.dv * 4   # S0 read + S1 write
            + Lsum * w.Hv * w.dv * 4           # U rows of the accepted paths
            + Lsum * w.Hqk * w.dk * es         # k rows (once per q/k head)
            + Lsum * w.Hv * 4                  # log_alpha along the paths
            + w.B * (w.Lmax + 1) * 4)          # path + path_len


def iteration_bytes(w: W.Workload) -> int:
    """One fused decoding iteration: the verify's traffic (the previous state is
    read once), the committed state written once, and the previous accepted
    path's rows (U, k, log alpha, parent links)."""
    es = 2 if w.dtype == W.BF16 else 4
    Lsum = int(w.path_len.sum())
    return (verify_bytes(w)
            + w.B * w.Hv * w.dk * w.dv * 4           # S1 write
            + Lsum * w.Hv * w.dv * 4                 # U rows of the accepted paths
            + Lsum * w.Hqk * w.dk * es               # k rows (once per q/k head)
            + Lsum * w.Hv * 4                        # log_alpha along the paths
            + Lsum * 4                               # parent links checked
            + w.B * (w.Lmax + 1) * 4)                # path + path_len


def verify_flops(w: W.Workload) -> int:
    B, N, Hqk, Hv, d = w.B, w.N, w.Hqk, w.Hv, w.dk
    return (B * Hv * (2 * 2 * N * d * d        # Q S0 and K S0
                      + N * N * d              # solve (dense lower-triangular)
                      + N * N * d)             # Y U
            + B * Hqk * (2 * N * N * d + N * N * d))  # Q K^T, K K^T (symmetric)


def commit_flops(w: W.Workload) -> int:
    return int(w.path_len.sum()) * w.Hv * 2 * w.dk * w.dv


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def measured_peaks() -> tuple[dict, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def kernel_source_sha() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        if os.path.exists(p):
            with open(p, "rb") as f:
                h.update(f.read())
    return h.hexdigest()[:16]


def verify_kernel_name(w: W.Workload) -> str:
    """The verify kernel the library dispatches for this shape (mirrors the
    C-ABI's rule: for bf16 with dk = dv = 128, the tensor-core kernel up to 128
    nodes, the 256-node kernel up to 256 and the chunk pass with R on the tensor
    cores beyond; the last two run single-chain units in the chunkwise form)."""
    forced = os.environ.get("GDN_TREE_KERNEL", "auto")
    tc_shape = w.dtype == W.BF16 and w.dk == 128 and w.dv == 128
    if tc_shape and forced not in ("generic", "long", "long_cuda"):
        if w.N <= 128 and forced != "mid":
            return "verify_tc_kernel"
        if w.N <= 256:
            return "verify_mid_kernel"
    if w.N > 256 or forced in ("long", "long_cuda"):
        if tc_shape and forced not in ("generic", "long_cuda"):
            # (past 256 nodes the units whose tree is one chain go to a kernel of their
            # own, launched first; past 128 the 256-node kernel runs them itself)
            return ("verify_chain_kernel + " if forced == "auto" else "") + "verify_long_tc_kernel"
        return "verify_long_kernel"
    return "verify_generic_kernel"


def topw_kernel_name(N: int, c: int, w: int) -> str:
    """The top-w kernel the library dispatches: the sorted-list kernel for rounds of
    at most 32 offers (w c <= 32), else the general one."""
    return "tree_topw_list_kernel" if w * c <= 32 and N <= 256 else "tree_topw_kernel"


def commit_kernel_name(w: W.Workload) -> str:
    """The commit kernel the library dispatches (mirrors the C-ABI's rule: the
    tensor-core commit for bf16, dk = dv = 128 and paths of more than 32 entries)."""
    if (w.dtype == W.BF16 and w.dk == 128 and w.dv == 128 and w.Lmax > 32
            and os.environ.get("GDN_TREE_KERNEL", "auto") != "generic"):
        return "commit_tc_kernel"
    return "commit_kernel"


def iteration_kernel_name(w: W.Workload) -> str:
    """The kernel one fused decoding iteration runs on (the tensor-core kernel
    with the delayed commitment fused in, where it takes the shape)."""
    if verify_kernel_name(w) == "verify_tc_kernel":
        return "verify_tc_kernel<fused commit>"
    return commit_kernel_name(w) + " + " + verify_kernel_name(w)


def arithmetic_dtype(kernel: str) -> str:
    # tensor-core kernel: bf16 products (fp32 accumulate, split-bf16 where the
    # state needs fp32 accuracy) and an fp32 solve; CUDA-core kernel: fp32
    return "bf16" if kernel.startswith("verify_tc_kernel") else "f32"


def profiled_traffic(kernel: str):
    """dram read+write bytes per launch of `kernel` from the committed ncu record,
    or None when the record was taken on a different kernel source or lacks it."""
    try:
        with open(PROFILE_TRAFFIC) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("source_sha") != kernel_source_sha():
        return None
    return rec.get("kernels", {}).get(kernel, {}).get("traffic_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 50 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        # the raw samples: $GDN_BENCH_CLOCKS_DIR if set, else the temporary directory
        out = os.environ.get("GDN_BENCH_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(out, f"gdn_bench_clocks_gpu{gpu_index}.csv")

    def sample_once(self) -> None:
        """One synchronous sample appended to the record (taken right before and
        right after the timed loop, so that a loop shorter than the sampling
        period still has clock readings)."""
        try:
            r = subprocess.run(["nvidia-smi", f"--query-gpu={self.FIELDS}",
                                "--format=csv,noheader,nounits", "-i", str(self.gpu)],
                               capture_output=True, text=True, timeout=10)
        except (OSError, subprocess.TimeoutExpired):
            return
        if r.returncode == 0 and r.stdout.strip():
            self.extra.append(r.stdout.strip())

    def __enter__(self):
        self.extra = []
        self.sample_once()
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "50"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()
        self.sample_once()

    def summary(self):
        lines = list(self.extra)
        if self.proc is not None and os.path.exists(self.path):
            with open(self.path) as f:
                lines += f.read().splitlines()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        if True:
            for line in lines:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax = float(parts[2])
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "samples": len(sm),
                "reasons": sorted(reasons)}


def max_over_ranks(x: float, dist, device=None) -> float:
    """Largest value of x over all ranks (identity when not distributed)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, B: int, N: int, ms_per_step: float) -> float:
    """Whole-job nodes/s: every rank verifies its own B x N nodes per step and
    the step time is the slowest rank's."""
    return world * B * N / (ms_per_step * 1e-3)


def rank_workload(cfg: int, rank: int, make=None) -> W.Workload:
    """Rank r's batch: its own seeded draw of the workload (seed 1000 + cfg + r),
    so that under N ranks the job is the concatenation of N independent batches,
    sequences of rank r first at index r * B (weak scaling, no data exchange)."""
    make = make or W.make_config
    return make(cfg, seed=1000 + cfg + rank)


def gather_sequences(x, dist, world: int):
    """The ranks' per-sequence results (leading axis = sequences) concatenated in
    rank order, on every rank (identity when not distributed)."""
    if dist is None or world == 1:
        return x
    import torch
    parts = [torch.empty_like(x) for _ in range(world)]
    dist.all_gather(parts, x)
    return torch.cat(parts, dim=0)


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def workload_config(w: W.Workload, world: int) -> dict:
    """The workload a step runs (the same dictionary for both arms)."""
    return {"workload": f"{w.name}: B={w.B} seqs x Hv={w.Hv} v-heads (Hqk={w.Hqk}), "
                        f"dk=dv={w.dk}, {w.dtype} q/k/v, fp32 S0, N={w.N}-node random trees "
                        "(branching 1-4, depth<=24), accepted paths <=24",
            "B": w.B, "N": w.N, "Hqk": w.Hqk, "Hv": w.Hv, "dk": w.dk, "dv": w.dv,
            "l2": "flushed before every timed step (256 MiB write, outside the events)",
            "parallelism": f"dp{world}",
            "step": "one decoding iteration: commit of the previous accepted path and "
                    "verification of the next tree"}


# ---------------------------------------------------------------------------
# reference arm: the fp64 CPU oracle, timed on the host cores
# ---------------------------------------------------------------------------

def run_reference(args, rank: int) -> None:
    """The oracle as it stands, timed on the host cores: every step verifies the
    whole layer's trees (all sequences and heads, memoised fp64 recurrence) and
    commits every accepted path, exactly the work of one step of our arm."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    w = W.make_config(WORKLOAD_CFG)
    cores = cpu_cores()

    def step():
        t0 = time.perf_counter()
        oracle.verify_workload(w, mode="memo", threads=cores)
        oracle.commit_workload(w, threads=cores)
        return time.perf_counter() - t0

    for _ in range(args.warmup):
        step()
    ts = [step() for _ in range(args.steps)]
    t_step = sum(ts) / len(ts)
    value = w.B * w.N / t_step
    line = {"metric": METRIC, "value": value, "unit": UNIT, "impl": "reference",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * t_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, args.gpus),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"each step: the whole layer ({w.B * w.Hv} (sequence, "
                                       "head) units), memoised fp64 recurrence + commit, "
                                       f"{cores} threads"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def first_sequences(w: W.Workload, nb: int) -> W.Workload:
    """The first nb sequences of a workload (every head, tree and path of each)."""
    import dataclasses
    sl = slice(0, nb)
    return dataclasses.replace(
        w, name=f"{w.name}[:{nb}]", B=nb, q=w.q[sl], k=w.k[sl], v=w.v[sl],
        log_alpha=w.log_alpha[sl], beta=w.beta[sl], parent=w.parent[sl], S0=w.S0[sl],
        path=w.path[sl], path_len=w.path_len[sl])


def cpu_baseline(w: W.Workload) -> dict:
    """The oracle as it stands on the host cores.  Headline: the whole workload,
    memoised fp64 recurrence + commit, all cores.  Beside it: the same on one
    core (a sample of sequences, scaled per node), and the literal path walk
    (every node re-runs its whole root-to-node path: the single-branch
    recurrent verification) on the small workloads and on a sample of this one."""
    import oracle
    oracle.build()
    cores = cpu_cores()
    t0 = time.perf_counter()
    oracle.verify_workload(w, mode="memo", threads=cores)
    oracle.commit_workload(w, threads=cores)
    dt = time.perf_counter() - t0
    out = {"value": w.B * w.N / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
           "sample": f"the whole workload ({w.B * w.Hv} (sequence, head) units), memoised "
                     f"fp64 recurrence + commit, {dt:.2f} s wall"}
    extra = []

    def timed(ww, mode, threads, label):
        t = time.perf_counter()
        oracle.verify_workload(ww, mode=mode, threads=threads)
        oracle.commit_workload(ww, threads=threads)
        sec = time.perf_counter() - t
        extra.append({"workload": label, "mode": mode, "cores": threads, "seconds": sec,
                      "nodes_per_s": ww.B * ww.N / sec})

    nb = 4  # sequences of the sample (each with all its heads)
    ws = first_sequences(w, nb)
    timed(ws, "memo", 1, f"{w.name}, first {nb} sequences")
    timed(ws, "path", cores, f"{w.name}, first {nb} sequences")
    for cfg in (0, 1, 2):
        wc = W.make_config(cfg)
        if wc.S0 is None:
            wc.S0 = oracle.warmup_state(wc.warmup["k"], wc.warmup["v"], wc.warmup["log_alpha"],
                                        wc.warmup["beta"], wc.Hv, wc.dk, wc.dv)
        timed(wc, "path", cores, wc.name)
    out["modes"] = extra
    return out


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def run_ours(args, rank: int, world: int, local_rank: int) -> None:
    import torch
    import gated_deltanet_tree_gdn_gb300 as gt
    from gated_deltanet_tree_gdn_gb300 import build as gbuild

    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    gbuild.build_library()
    gt.load()
    dev = torch.device("cuda", local_rank)

    w = rank_workload(WORKLOAD_CFG, rank)
    dt = torch.bfloat16 if w.dtype == W.BF16 else torch.float32

    def host(x, dtype=None):
        return torch.from_numpy(np.ascontiguousarray(x)).to(dtype=dtype).pin_memory()

    hin = dict(q=host(w.q, dt), k=host(w.k, dt), v=host(w.v, dt), log_alpha=host(w.log_alpha),
               beta=host(w.beta), parent=host(w.parent), S0=host(w.S0), path=host(w.path),
               path_len=host(w.path_len))
    x = {kk: t.to(dev) for kk, t in hin.items()}
    o = torch.empty((w.B, w.N, w.Hv, w.dv), dtype=dt, device=dev)
    U = torch.empty((w.B, w.Hv, w.N, w.dv), dtype=torch.float32, device=dev)
    S1 = torch.empty_like(x["S0"])
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step(xx, oo, UU, SS):
        gt.verify(xx["q"], xx["k"], xx["v"], xx["log_alpha"], xx["beta"], xx["parent"],
                  xx["S0"], o=oo, U=UU)
        gt.commit(xx["path"], xx["path_len"], UU, xx["k"], xx["log_alpha"], xx["S0"], S1=SS,
                  parent=xx["parent"])

    # ping-pong buffers of a decoding loop: step i commits the accepted path of
    # the tree verified at step i-1 (its U rows) and verifies the next tree
    Sbuf = [x["S0"].clone(), torch.empty_like(x["S0"])]
    Ubuf = [torch.empty_like(U), torch.empty_like(U)]
    gt.verify(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["parent"], Sbuf[0],
              o=o, U=Ubuf[0])

    def iteration(i, xx=None, oo=None):
        xx = xx or x
        cur, nxt = i & 1, (i + 1) & 1
        gt.commit_verify(xx["path"], xx["path_len"], Ubuf[cur], xx["k"], xx["log_alpha"],
                         Sbuf[cur], xx["q"], xx["k"], xx["v"], xx["log_alpha"], xx["beta"],
                         xx["parent"], S1=Sbuf[nxt], o=o if oo is None else oo, U=Ubuf[nxt],
                         prev_parent=xx["parent"])

    for i in range(args.warmup):
        flush.zero_()
        iteration(i)
        flush.zero_()
        step(x, o, U, S1)
    torch.cuda.synchronize()

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        wall0 = time.perf_counter()
        for i in range(K):
            flush.zero_()
            ev[i][0].record(stream)
            iteration(i)
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t_it = [ev[i][0].elapsed_time(ev[i][1]) for i in range(K)]
    ms_per_step = max_over_ranks(float(sum(t_it)), dist, dev) / K
    value = job_throughput(world, w.B, w.N, ms_per_step)

    # the same work as two separate calls (verify, then commit)
    Ks = min(K, 1000)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(Ks)]
    for i in range(Ks):
        flush.zero_()
        evs[i][0].record(stream)
        gt.verify(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["parent"], x["S0"],
                  o=o, U=U)
        evs[i][1].record(stream)
        gt.commit(x["path"], x["path_len"], U, x["k"], x["log_alpha"], x["S0"], S1=S1,
                  parent=x["parent"])
        evs[i][2].record(stream)
    torch.cuda.synchronize()
    t_ver = [evs[i][0].elapsed_time(evs[i][1]) for i in range(Ks)]   # ms
    t_com = [evs[i][1].elapsed_time(evs[i][2]) for i in range(Ks)]
    sep_ms = max_over_ranks(float(sum(t_ver) + sum(t_com)), dist, dev) / Ks

    # for scale: a plain device copy of the state bytes the commit streams (S0 in,
    # S1 out), under the same flush and events
    evc = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(Ks)]
    for i in range(Ks):
        flush.zero_()
        evc[i][0].record(stream)
        S1.copy_(x["S0"])
        evc[i][1].record(stream)
    torch.cuda.synchronize()
    state_copy_us = 1e3 * statistics.mean(evc[i][0].elapsed_time(evc[i][1]) for i in range(Ks))

    # the page's measurement baseline: single-branch recurrent verification of the
    # same trees (one recurrent pass per root-to-leaf branch), against which the
    # tree verification is compared
    Kr = min(K, 100)
    evr = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(Kr)]
    for i in range(Kr):
        flush.zero_()
        evr[i][0].record(stream)
        gt.verify_recurrent(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["parent"],
                            x["S0"], o=o, U=U)
        evr[i][1].record(stream)
    torch.cuda.synchronize()
    rec_ms = max_over_ranks(float(sum(evr[i][0].elapsed_time(evr[i][1]) for i in range(Kr))),
                            dist, dev) / Kr

    # the step before the verification: top-w best-first construction of trees of
    # the same size (c = w = 4 candidates and pops, depth <= 24), from seeded
    # candidate log-probabilities
    lp = torch.from_numpy(np.log(np.random.default_rng(7).uniform(
        1e-6, 1.0, size=(w.B, w.N, 4))).astype(np.float32)).to(dev)
    tb_par = torch.empty((w.B, w.N), dtype=torch.int32, device=dev)
    tb_j = torch.empty_like(tb_par)
    tb_s = torch.empty((w.B, w.N), dtype=torch.float32, device=dev)
    tb_n = torch.empty((w.B,), dtype=torch.int32, device=dev)
    # device time per call: the calls replayed back to back from a CUDA graph, as a
    # serving loop launches its iteration (timed call by call, a launch of this size
    # mostly measures the host's launch latency)
    Kt = 20
    tb_stream = torch.cuda.Stream()
    tb_stream.wait_stream(stream)
    with torch.cuda.stream(tb_stream):
        for _ in range(3):
            gt.build_topw(lp, 4, 24, parent=tb_par, cand_index=tb_j, score=tb_s, n_built=tb_n)
    torch.cuda.synchronize()
    tb_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(tb_graph, stream=tb_stream):
        for _ in range(Kt):
            gt.build_topw(lp, 4, 24, parent=tb_par, cand_index=tb_j, score=tb_s, n_built=tb_n)
    tb_runs = []
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(tb_stream):  # the graph runs on the current stream
            e0.record(tb_stream)
            tb_graph.replay()
            e1.record(tb_stream)
        torch.cuda.synchronize()
        tb_runs.append(1e3 * e0.elapsed_time(e1) / Kt)
    tb_us = statistics.median(tb_runs)
    del tb_graph

    # trees past the on-chip limit: the two-level chunk pass (verify, then the commit
    # of paths into them) on 1024-node random trees of the same family (branching
    # 1-4, depth <= 24), 8 sequences x the same heads
    wl = W.make_custom(seed=1024 + rank, B=8, N=1024, Hqk=w.Hqk, Hv=w.Hv, dk=w.dk, dv=w.dv,
                       dtype=w.dtype, tree="random", max_depth=24)
    xl = {kk: torch.from_numpy(np.ascontiguousarray(getattr(wl, kk))).to(
        device=dev, dtype=dt if kk in ("q", "k", "v") else None)
        for kk in ("q", "k", "v", "log_alpha", "beta", "parent", "S0", "path", "path_len")}
    ol = torch.empty((wl.B, wl.N, wl.Hv, wl.dv), dtype=dt, device=dev)
    Ul = torch.empty((wl.B, wl.Hv, wl.N, wl.dv), dtype=torch.float32, device=dev)
    S1l = torch.empty_like(xl["S0"])
    Kl = max(3, min(K, 10))
    evl = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(Kl + 1)]
    for i in range(Kl + 1):  # the first iteration is a warm-up
        flush.zero_()
        evl[i][0].record(stream)
        gt.verify(xl["q"], xl["k"], xl["v"], xl["log_alpha"], xl["beta"], xl["parent"],
                  xl["S0"], o=ol, U=Ul)
        evl[i][1].record(stream)
        gt.commit(xl["path"], xl["path_len"], Ul, xl["k"], xl["log_alpha"], xl["S0"], S1=S1l,
                  parent=xl["parent"])
        evl[i][2].record(stream)
    torch.cuda.synchronize()
    lv_us = 1e3 * statistics.mean(evl[i][0].elapsed_time(evl[i][1]) for i in range(1, Kl + 1))
    lc_us = 1e3 * statistics.mean(evl[i][1].elapsed_time(evl[i][2]) for i in range(1, Kl + 1))

    # one decoding step of one sequence (the decode shape: 1 sequence x 32 v-heads, a
    # 16-node tree; the state drawn at random, which changes no timing): what a serving
    # loop waits when the GPU is idle at the call (binding, launch and kernel, read by
    # the host after a synchronize), the host's part of it, and the device time alone
    w1 = W.make_config(1)
    w1.S0 = W.draw_state(np.random.Generator(np.random.PCG64(1001)), w1.B, w1.Hv, w1.dk, w1.dv)
    x1 = {kk: torch.from_numpy(np.ascontiguousarray(getattr(w1, kk))).to(
        device=dev, dtype=dt if kk in ("q", "k", "v") else None)
        for kk in ("q", "k", "v", "log_alpha", "beta", "parent", "S0")}
    o1 = torch.empty((w1.B, w1.N, w1.Hv, w1.dv), dtype=dt, device=dev)
    U1 = torch.empty((w1.B, w1.Hv, w1.N, w1.dv), dtype=torch.float32, device=dev)

    def decode_call():
        gt.verify(x1["q"], x1["k"], x1["v"], x1["log_alpha"], x1["beta"], x1["parent"],
                  x1["S0"], o=o1, U=U1)

    for _ in range(10):
        decode_call()
    torch.cuda.synchronize()
    d_host, d_done = [], []
    for _ in range(50):
        t0 = time.perf_counter()
        decode_call()
        t1 = time.perf_counter()
        torch.cuda.synchronize()
        t2 = time.perf_counter()
        d_host.append((t1 - t0) * 1e6)
        d_done.append((t2 - t0) * 1e6)
    d_stream = torch.cuda.Stream()
    d_stream.wait_stream(stream)
    with torch.cuda.stream(d_stream):
        decode_call()
    torch.cuda.synchronize()
    d_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(d_graph, stream=d_stream):
        for _ in range(20):
            decode_call()
    d_dev = []
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(d_stream):
            e0.record(d_stream)
            d_graph.replay()
            e1.record(d_stream)
        torch.cuda.synchronize()
        d_dev.append(1e3 * e0.elapsed_time(e1) / 20)
    del d_graph, x1, o1, U1
    decode_step = {"workload": f"decode-B{w1.B}-Hv{w1.Hv}-N{w1.N}: B={w1.B} x Hv={w1.Hv} "
                               f"(Hqk={w1.Hqk}), N={w1.N}-node tree, d={w1.dk}, bf16, state "
                               "drawn at random (timing only)",
                   "kernel": verify_kernel_name(w1),
                   "call_to_done_us": statistics.median(d_done),
                   "host_us": statistics.median(d_host),
                   "device_us": statistics.median(d_dev),
                   "timing": "median of 50 calls with the GPU idle at each call (host clock, "
                             "synchronize included); device time from a CUDA graph of 20"}

    # the stress shapes: 64 sequences of 256-node trees mixing 256-deep chains,
    # stars and random trees, strong decay and beta up to 0.99 (the CUDA-core
    # on-chip kernel: the tensor-core kernel takes trees of up to 128 nodes)
    w4 = W.make_config(4)
    x4 = {kk: torch.from_numpy(np.ascontiguousarray(getattr(w4, kk))).to(
        device=dev, dtype=dt if kk in ("q", "k", "v") else None)
        for kk in ("q", "k", "v", "log_alpha", "beta", "parent", "S0", "path", "path_len")}
    o4 = torch.empty((w4.B, w4.N, w4.Hv, w4.dv), dtype=dt, device=dev)
    U4 = torch.empty((w4.B, w4.Hv, w4.N, w4.dv), dtype=torch.float32, device=dev)
    S14 = torch.empty_like(x4["S0"])
    K4 = max(3, min(K, 10))
    ev4 = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K4 + 1)]
    for i in range(K4 + 1):  # the first iteration is a warm-up
        flush.zero_()
        ev4[i][0].record(stream)
        gt.verify(x4["q"], x4["k"], x4["v"], x4["log_alpha"], x4["beta"], x4["parent"],
                  x4["S0"], o=o4, U=U4)
        ev4[i][1].record(stream)
        gt.commit(x4["path"], x4["path_len"], U4, x4["k"], x4["log_alpha"], x4["S0"], S1=S14,
                  parent=x4["parent"])
        ev4[i][2].record(stream)
    torch.cuda.synchronize()
    c4v_us = 1e3 * statistics.mean(ev4[i][0].elapsed_time(ev4[i][1]) for i in range(1, K4 + 1))
    c4c_us = 1e3 * statistics.mean(ev4[i][1].elapsed_time(ev4[i][2]) for i in range(1, K4 + 1))
    del x4, o4, U4, S14

    # end to end through the public API: every step copies the tree's inputs and
    # the accepted path from pinned host memory (the recurrent state stays
    # resident on the device, as in a decoding loop), runs one decoding
    # iteration, and reads its result, the tree's outputs o, back into pinned
    # memory.  The inputs of a step sit in one packed pinned staging buffer and
    # cross in ONE host-to-device copy (16-byte aligned sub-buffers, viewed as
    # the call's tensors on the device); o comes back in one copy.  As a serving
    # loop runs it: step i's inputs copy in on one stream while step i - 1
    # computes, and step i - 1's outputs copy out on another (staging and o
    # double-buffered; every copy of every step is inside the timed region).
    per_step_inputs = [kk for kk in hin if kk != "S0"]
    offs, pos = {}, 0
    for kk in per_step_inputs:
        nbytes = hin[kk].numel() * hin[kk].element_size()
        offs[kk] = (pos, nbytes)
        pos += (nbytes + 255) // 256 * 256
    stage_bytes = pos
    h_stage = torch.empty(stage_bytes, dtype=torch.uint8).pin_memory()
    for kk in per_step_inputs:
        a, nbytes = offs[kk]
        h_stage[a:a + nbytes].copy_(hin[kk].reshape(-1).view(torch.uint8))
    d_stage = [torch.empty(stage_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]

    def staged_views(buf):
        out = {}
        for kk in per_step_inputs:
            a, nbytes = offs[kk]
            out[kk] = buf[a:a + nbytes].view(hin[kk].dtype).view(hin[kk].shape)
        return out

    xe = [staged_views(d_stage[j]) for j in range(2)]
    h_o = torch.empty(o.shape, dtype=dt).pin_memory()
    h2d = stage_bytes
    d2h = h_o.numel() * h_o.element_size()
    Ke = max(3, min(K, 50))
    oe = [o, torch.empty_like(o)]
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_step(i, first):
        j = i & 1
        if not first[j]:
            s_in.wait_event(ev_comp[j])    # step i - 2 has read this staging buffer
            stream.wait_event(ev_out[j])   # and its o has been copied out
        with torch.cuda.stream(s_in):
            d_stage[j].copy_(h_stage, non_blocking=True)
            ev_in[j].record(s_in)
        stream.wait_event(ev_in[j])
        xx = dict(xe[j], S0=x["S0"])
        iteration(i, xx, oe[j])
        ev_comp[j].record(stream)
        s_out.wait_event(ev_comp[j])
        with torch.cuda.stream(s_out):
            h_o.copy_(oe[j], non_blocking=True)
            ev_out[j].record(s_out)
        first[j] = False

    def e2e_run(n):
        first = [True, True]
        for i in range(n):
            e2e_step(i, first)
        stream.wait_event(ev_out[(n - 1) & 1])
        if n > 1:
            stream.wait_event(ev_out[n & 1])

    e2e_run(3)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    e2e_run(Ke)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / Ke, dist, dev)

    # the link itself: the same staging copy alone, host to device and back
    c0 = torch.cuda.Event(enable_timing=True)
    c1 = torch.cuda.Event(enable_timing=True)
    c2 = torch.cuda.Event(enable_timing=True)
    for _ in range(2):
        d_stage[0].copy_(h_stage, non_blocking=True)
    c0.record(stream)
    for _ in range(5):
        d_stage[0].copy_(h_stage, non_blocking=True)
    c1.record(stream)
    for _ in range(5):
        h_o.copy_(o, non_blocking=True)
    c2.record(stream)
    torch.cuda.synchronize()
    h2d_gbs = 5 * stage_bytes / (c0.elapsed_time(c1) * 1e-3) / 1e9
    d2h_gbs = 5 * d2h / (c1.elapsed_time(c2) * 1e-3) / 1e9

    if rank == 0:
        peaks, peak_kind = measured_peaks()
        vb, cb, ib = verify_bytes(w), commit_bytes(w), iteration_bytes(w)
        vf, cf = verify_flops(w), commit_flops(w)
        it_ms = ms_per_step
        hbm = float(peaks["hbm_gbs"])
        tflops = float(peaks["bf16_tflops"])
        kernel = iteration_kernel_name(w)
        achieved = ib / (statistics.mean(t_it) * 1e-3) / 1e9
        traffic = profiled_traffic(kernel)
        t_roof = max(ib / (hbm * 1e9), (vf + cf) / (tflops * 1e12))
        t_roof_sep = max((vb + cb) / (hbm * 1e9), (vf + cf) / (tflops * 1e12))
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": arithmetic_dtype(kernel),
            "data": "synthetic",
            "config": workload_config(w, world),
            "clocks": clk.summary(),
            "e2e": {"value": job_throughput(world, w.B, w.N, e2e_ms), "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_ms, "copies_per_step": {"h2d": 1, "d2h": 1},
                    "link": {"h2d_gbs_copy_alone": h2d_gbs, "d2h_gbs_copy_alone": d2h_gbs,
                             "h2d_ms_copy_alone": stage_bytes / (h2d_gbs * 1e9) * 1e3}},
            "gpu_launches": K,
            "roofline": {"bound": "hbm", "kernel": kernel, "achieved": achieved, "peak": hbm,
                         "unit": "GB/s", "frac": achieved / hbm, "traffic": traffic,
                         "algorithmic_bytes_per_launch": ib, "peak_source": peak_kind,
                         "peak_nominal": NOMINAL_HBM_GBS,
                         "frac_nominal": achieved / NOMINAL_HBM_GBS},
            "step": {"iteration_us": 1e3 * it_ms, "iteration_bytes": ib,
                     "roofline_us": 1e6 * t_roof, "roofline_frac": t_roof / (it_ms * 1e-3),
                     "wall_s_timed_loop": wall},
            "separate_calls": {"value": job_throughput(world, w.B, w.N, sep_ms),
                               "ms_per_step": sep_ms,
                               "verify_us": 1e3 * statistics.mean(t_ver),
                               "commit_us": 1e3 * statistics.mean(t_com),
                               "verify_bytes": vb, "commit_bytes": cb,
                               "verify_roofline_frac": vb / (statistics.mean(t_ver) * 1e-3)
                               / (hbm * 1e9),
                               "roofline_frac": t_roof_sep / (sep_ms * 1e-3),
                               "verify_flops": vf, "commit_flops": cf,
                               "state_copy_us": state_copy_us,
                               "state_copy_bytes": 2 * x["S0"].numel() * 4,
                               "verify_kernel": verify_kernel_name(w),
                               "commit_kernel": commit_kernel_name(w),
                               "verify_traffic": profiled_traffic(verify_kernel_name(w))},
        }
        line["recurrent_baseline"] = {
            "kernel": "verify_recurrent_kernel", "verify_us": 1e3 * rec_ms,
            "nodes_per_s": job_throughput(world, w.B, w.N, rec_ms),
            "tree_verify_speedup": rec_ms / statistics.mean(t_ver),
            "page": "fused tree kernel 7.1x faster than single-branch recurrent verification "
                    "at 126 tree tokens, NVIDIA B200 (DFlash-TfM, results)"}
        line["decode_step"] = decode_step
        line["tree_build"] = {"kernel": topw_kernel_name(w.N, 4, 4), "us": tb_us,
                              "timing": "device time per call, 20 calls replayed from a CUDA "
                                        "graph (median of 5 replays)",
                              "B": w.B, "N": w.N,
                              "c": 4, "w": 4, "max_depth": 24,
                              "rounds": -(-(w.N - 1) // 4)}
        line["long_trees"] = {
            "kernel": verify_kernel_name(wl) + " + " + commit_kernel_name(wl),
            "workload": f"B={wl.B} seqs x Hv={wl.Hv} v-heads (Hqk={wl.Hqk}), N={wl.N}-node random "
                        "trees (branching 1-4, depth<=24), accepted paths <= depth",
            "verify_us": lv_us, "commit_us": lc_us,
            "nodes_per_s": wl.B * wl.N / ((lv_us + lc_us) * 1e-6),
            "verify_roofline_frac": verify_bytes(wl) / (lv_us * 1e-6) / (hbm * 1e9),
            "commit_roofline_frac": commit_bytes(wl) / (lc_us * 1e-6) / (hbm * 1e9)}
        line["config4"] = {
            "kernel": verify_kernel_name(w4) + " + " + commit_kernel_name(w4),
            "workload": W.CONFIG_NAMES[4] + ": B=64 seqs x Hv=32 v-heads (Hqk=16), dk=dv=128, "
                        "bf16, N=256-node trees (256-deep chains, stars, random trees), "
                        "log alpha down to -4, beta up to 0.99",
            "verify_us": c4v_us, "commit_us": c4c_us,
            "nodes_per_s": w4.B * w4.N / ((c4v_us + c4c_us) * 1e-6),
            "verify_roofline_frac": verify_bytes(w4) / (c4v_us * 1e-6) / (hbm * 1e9),
            "commit_roofline_frac": commit_bytes(w4) / (c4c_us * 1e-6) / (hbm * 1e9)}
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(w)
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
    else:
        run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
