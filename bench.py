"""Benchmark: one decode-attention step over a paged GQA KV cache.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

A step is the whole hot path on one batch: host plan, the split kernel and
(when the plan splits) the ordered combine.  The metric is the effective
KV-read bandwidth (algorithmic K+V bytes / step time) with the fraction of
the HBM roofline and the microseconds per step.  Default workload: the long
context (B=4, 131072 tokens each, 64 query / 8 KV heads, head_dim 128,
page 64; 2 GiB of K+V, larger than L2, so no flush is needed; smaller
workloads flush L2 between timed steps and time each step with events).

With N > 1 (torchrun) every rank runs an independent replica on its own GPU
("replicas only": the path needs no exchange), a barrier brackets the timed
region, the time is the max over ranks and ``value`` counts all ranks' bytes.

``--impl reference`` times the f64 CPU oracle on the host cores instead, on
bounded samples of the same workload, in the same units.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import glob
import json
import os
import platform
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attention effective KV-read TB/s (% of HBM peak); µs per decode step"
FALLBACK_HBM_GBS = 6800.0
WORKLOAD_DESC = {
    "long": "B=4, seq 131072 each, Hq=64, Hkv=8, D=128, page 64, full context",
    "long_b1": "B=1, seq 131072, Hq=64, Hkv=8, D=128, page 64, full context",
    "long_w4096": "B=4, seq 131072 each, Hq=64, Hkv=8, D=128, page 64, window 4096",
    "long_d256": "B=1, seq 131072, Hq=16, Hkv=4, D=256, page 64, full context",
    "batched": "B=64, Hq=32, Hkv=8, D=128, seq_lens U[1,8192], page 16",
    "llama": "B=1, Hq=32, Hkv=8, D=128, context 3060, page 16 (Llama-3.1-8B shape)",
    "sweep_d64": "B=1, Hq=32, Hkv=8, D=64, context 3060, page 16",
    "sweep_d128": "B=1, Hq=32, Hkv=8, D=128, context 3060, page 16",
    "sweep_d256": "B=1, Hq=16, Hkv=4, D=256, context 3060, page 16",
    "tiny": "B=1, Hq=4, Hkv=1, D=64, context 256, page 16",
    "many_short": "B=1000, Hq=32, Hkv=8, D=128, seq_lens U[1,512], page 16",
}


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="long", choices=sorted(WORKLOAD_DESC))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-budget", type=float, default=15.0,
                    help="seconds of oracle work for the cpu_baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--variant", type=int, default=0)
    ap.add_argument("--force-chunk", type=int, default=0)
    ap.add_argument("--dtype", default="fp16", choices=["fp16", "bf16"],
                    help="element format of q, K/V and out")
    ap.add_argument("--queries", type=int, default=1,
                    help="query positions per sequence (the last T positions, causal)")
    ap.add_argument("--append", action="store_true",
                    help="time the fused append + attention launch (new rows at the last "
                         "T positions)")
    ap.add_argument("--schedule", type=int, default=0,
                    help="0 planner, 1 grid (workspace merge), 2 cluster merge")
    ap.add_argument("--eager", action="store_true",
                    help="launch each step from the host instead of replaying a CUDA graph")
    ap.add_argument("--dump", default="",
                    help="write the step's output (fp32), the workload and the plan to this "
                         ".npz for offline comparison with the oracle")
    ap.add_argument("--config-steps", type=int, default=200,
                    help="timed steps of each per_config entry (0 skips the block)")
    ap.add_argument("--context-sweep", action="store_true",
                    help="threshold A/B instead of the bench line: contexts 1..512 of the "
                         "three head-dim shapes, split threshold 256 (default), always split, "
                         "or single pass up to 512; one JSON line per point")
    return ap.parse_args(argv)


# ------------------------------------------------------------ distributed

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(backend):
    import torch.distributed as dist
    if int(os.environ.get("WORLD_SIZE", "1")) > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend)
    return dist.is_initialized()


def max_over_ranks(x: float, device=None) -> float:
    """Largest value of x over all ranks (x itself without a process group)."""
    import torch
    import torch.distributed as dist
    if not dist.is_initialized():
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not dist.is_initialized():
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_initialized():
        dist.barrier()


# ------------------------------------------------------------ peaks / clocks

def load_peak_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            for k in ("hbm_gbs", "hbm_GBs", "hbm_copy_gbs"):
                if k in d:
                    return float(d[k]), "measured (MEASURED_PEAKS.json)"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, earlier GB300 copy measurement)"


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 100 ms."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader",
                 "-i", str(self.index), "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self, t0: float, t1: float):
        samples = []
        for l in self.lines:
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                sm = float(parts[2].split()[0])
                smax = float(parts[3].split()[0])
            except ValueError:
                continue
            reasons = [name for name, v in zip(
                ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"),
                parts[6:10]) if v.lower() == "active"]
            samples.append((ts, sm, smax, reasons))
        if not samples:
            return None
        inside = [s for s in samples if t0 - 0.05 <= s[0] <= t1 + 0.05]
        window = "timed"
        if not inside:  # timed region shorter than the sampling period
            inside = [s for s in samples if s[0] <= t1 + 0.2]
            window = "warmup+timed"
        if not inside:
            inside, window = samples, "whole run"
        reasons = sorted({r for s in inside for r in s[3]})
        return {"sm_mhz": statistics.median(s[1] for s in inside),
                "sm_max_mhz": max(s[2] for s in inside), "reasons": reasons,
                "samples": len(inside), "window": window}


# ------------------------------------------------------------ traffic record

def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in sorted(glob.glob(os.path.join(ROOT, "paged_gqa_decode_06_gb300", "csrc", "*"))):
        with open(f, "rb") as fh:
            h.update(os.path.basename(f).encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kernel: str):
    """DRAM bytes per launch of the split kernel from the committed ncu
    summary, if it was taken of the same kernel on the current kernel
    sources (the summaries are captured with the default options: fp16, one
    query position, no append; the caller passes None for other runs)."""
    path = os.path.join(ROOT, "profiles", f"split_kernel_{workload}.md")
    if kernel is None or not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    kn = re.search(r"^kernel:\s*(\S+)", text, re.M)
    hsh = re.search(r"kernel_source_sha256:\s*([0-9a-f]+)", text)
    if not m or not kn or kn.group(1) != kernel or not hsh or \
            hsh.group(1) != kernel_source_hash():
        return None
    return float(m.group(1))


# ------------------------------------------------------------ CPU oracle

def split_kernel_name(plan, head_dim: int) -> str:
    """The split kernel a plan launches (the one the roofline is taken on)."""
    if plan.variant == 1:
        return "split_simt_kernel"
    if plan.cluster > 0:
        return "split_mma_kernel_cluster"
    if plan.ring_stages == (4 if head_dim == 64 else 2):
        return "split_mma_kernel_shallow"
    if not plan.split:
        return "split_mma_kernel_single"
    return "split_mma_kernel"


def cpu_model() -> str:
    """The host CPU's name from /proc/cpuinfo (x86 'model name'; on Arm the
    implementer/part codes when no name is given)."""
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
    except OSError:
        return platform.machine()
    for key in ("model name", "Model Name", "Hardware"):
        m = re.search(rf"^{key}\s*:\s*(.+)$", info, re.M)
        if m:
            return m.group(1).strip()
    imp = re.search(r"^CPU implementer\s*:\s*(\S+)", info, re.M)
    part = re.search(r"^CPU part\s*:\s*(\S+)", info, re.M)
    if imp and part:
        return f"{platform.machine()} implementer {imp.group(1)} part {part.group(1)}"
    return platform.machine()


def percentiles_us(ms_list):
    """p10 / median / p90 of per-step times given in ms, in us."""
    import numpy as np
    a = np.asarray(ms_list, dtype=np.float64) * 1e3
    return {"p10": float(np.percentile(a, 10)), "p50": float(np.percentile(a, 50)),
            "p90": float(np.percentile(a, 90))}


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class OracleSample:
    """Times the oracle on whole GQA groups (all G query heads of one KV head
    of one sequence) over the last n_tok attended positions.  The sample is
    sized once (calibrate) to about budget_s seconds; run() then repeats it."""

    def __init__(self, w_cpu, threads: int):
        import numpy as np
        self.w, self.threads = w_cpu, threads
        self.G = w_cpu.num_q_heads // w_cpu.num_kv_heads
        L = w_cpu.seq_lens.to("cpu").numpy().astype(np.int64)
        self.L_max = int(L.max())
        self.L_att = np.minimum(L, w_cpu.window) if w_cpu.window > 0 else L
        self.n_groups_all = w_cpu.batch * w_cpu.num_kv_heads
        self.ng = min(self.n_groups_all, max(1, (threads + self.G - 1) // self.G))
        self.ntok = int(min(4096, self.L_att.max()))

    def _rows(self):
        import numpy as np
        w, rows = self.w, []
        for gi in range(self.ng):
            b, h = divmod(gi, w.num_kv_heads)
            rows += [b * w.num_q_heads + h * self.G + g for g in range(self.G)]
        return np.array(rows, dtype=np.int32)

    def run(self):
        """(algorithmic K+V bytes of the sample, seconds)."""
        import oracle
        w = self.w
        win = self.ntok if self.ntok < self.L_max else w.window
        rows = self._rows()
        t0 = time.perf_counter()
        oracle.decode_attn(w.q, w.k_pages, w.v_pages, w.page_table, w.seq_lens, w.scale, win,
                           rows=rows, threads=self.threads)
        dt = time.perf_counter() - t0
        toks = sum(int(min(self.L_att[gi // w.num_kv_heads], self.ntok))
                   for gi in range(self.ng))
        return toks * 4 * w.head_dim, dt

    def calibrate(self, budget_s: float):
        nbytes, dt = self.run()
        target = nbytes / max(dt, 1e-9) * budget_s
        per_tok = 4 * self.w.head_dim
        self.ntok = int(min(self.L_att.max(), max(1, target / (per_tok * self.ng))))
        if self.ntok >= self.L_att.max():
            self.ng = int(min(self.n_groups_all,
                              max(self.ng, target / (per_tok * max(1.0, self.L_att.mean())))))
        return self

    def describe(self, nbytes):
        return (f"{self.ng} GQA groups x {self.G} query heads, last {self.ntok} attended "
                f"positions each ({nbytes / 1e6:.1f} MB of K+V), {self.threads} threads")


# ------------------------------------------------------------ GPU arm

# The configurations the per_config block times besides the headline (every
# workload of the benchmark's config list: the tiny decode, the Llama-3.1-8B
# shape, the head_dim sweep at 3060 tokens, the batched serving mix and the
# long context with a 4096-position window).
PER_CONFIG = ("tiny", "llama", "sweep_d64", "sweep_d128", "sweep_d256", "batched",
              "long_w4096")


def l2_policy(kv_bytes: int, l2_bytes: int):
    """(flush?, description): steps whose K/V fit in twice the L2 flush it
    between timed steps; larger inputs stream from HBM anyway."""
    if kv_bytes < 2 * l2_bytes:
        return True, "flushed between timed steps (write of 4x L2, then read of 4x L2)"
    return False, f"inputs {kv_bytes / 2**30:.2f} GiB > L2, no flush"


def time_config(pkg, workloads, name, dev, local, steps, dtype, peak_gbs, flush_l2, l2):
    """One per_config entry: the workload's decode step (decode_attn_split,
    one launch) captured in a CUDA graph and replayed `steps` times, each
    replay bracketed by events on the launching stream, L2 flushed before each
    step when the workload fits in twice the L2."""
    import torch
    w = workloads.make(name, device=dev, dtype=dtype)
    kv_bytes = w.kv_bytes()
    max_len = w.max_seq_len()
    params = pkg.make_params(w.q, w.k_pages, w.page_table, w.scale, w.window, max_len)
    props = torch.cuda.get_device_properties(dev)
    plan = pkg.decode_attn_make_plan(params, props.multi_processor_count)
    ws = torch.zeros(max(pkg.decode_attn_workspace_size(params, local), 256), dtype=torch.uint8,
                     device=dev)
    out = torch.empty_like(w.q)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush, l2_desc = l2_policy(kv_bytes, l2)

    def step():
        pkg.decode_attn_split(w.q, w.k_pages, w.v_pages, w.page_table, w.seq_lens, w.scale,
                              window=w.window, out=out, max_seq_len=max_len, workspace=ws,
                              err_flag=err)

    for _ in range(3):
        if flush:
            flush_l2()
        step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(3):
        if flush:
            flush_l2()
        g.replay()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for e0, e1 in evs:
        if flush:
            flush_l2()
        e0.record(stream)
        g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    ms = [a.elapsed_time(b) for a, b in evs]
    if int(err.item()) != 0:
        raise RuntimeError(f"{name}: device error bits {int(err.item())}")
    mean_ms = statistics.mean(ms)
    gbs = kv_bytes / (mean_ms * 1e-3) / 1e9
    entry = {"desc": WORKLOAD_DESC[name], "us_per_step": mean_ms * 1e3,
             "us_percentiles": percentiles_us(ms), "kv_bytes_per_step": kv_bytes,
             "kv_tbs": gbs / 1e3, "frac": gbs / peak_gbs, "steps": steps, "l2": l2_desc,
             "kernel": split_kernel_name(plan, w.head_dim),
             "plan": {k: plan.as_dict()[k] for k in ("split", "chunk_tokens", "max_shards",
                                                     "grid_x", "grid_y", "grid_z", "cluster",
                                                     "ring_stages")}}
    del g, w, ws, out
    torch.cuda.empty_cache()
    return entry


def gpu_arm(args):
    import torch
    import paged_gqa_decode_06_gb300 as pkg
    from paged_gqa_decode_06_gb300 import build, workloads

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init("nccl")
    build.build()
    pkg.load_library()

    edt = torch.bfloat16 if args.dtype == "bf16" else torch.float16
    w = workloads.make(args.workload, device=dev, dtype=edt)
    T = max(1, args.queries)
    gen = torch.Generator(device=dev)
    gen.manual_seed(1234)
    if T > 1:  # T query positions per sequence: q [B, T, Hq, D]
        w.q = torch.randn(w.batch, T, w.num_q_heads, w.head_dim, generator=gen, device=dev,
                          dtype=torch.float32).to(edt)
    k_new = v_new = None
    if args.append:
        shape = (w.batch, T, w.num_kv_heads, w.head_dim) if T > 1 else \
            (w.batch, w.num_kv_heads, w.head_dim)
        k_new = torch.randn(*shape, generator=gen, device=dev, dtype=torch.float32).to(edt)
        v_new = torch.randn(*shape, generator=gen, device=dev, dtype=torch.float32).to(edt)
    max_len = w.max_seq_len()
    kv_bytes = w.kv_bytes()
    if T > 1 and w.window > 0:  # the first query's window starts T - 1 earlier
        L = w.seq_lens.to("cpu").to(torch.int64)
        kv_bytes = int(torch.clamp(L, max=w.window + T - 1).sum()) * w.num_kv_heads * \
            w.head_dim * 4
    params = pkg.make_params(w.q, w.k_pages, w.page_table, w.scale, w.window, max_len,
                             args.variant, 0, args.force_chunk, args.schedule)
    props = torch.cuda.get_device_properties(dev)
    plan = pkg.decode_attn_make_plan(params, props.multi_processor_count)
    ws_bytes = pkg.decode_attn_workspace_size(params, local)
    ws = torch.zeros(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    out = torch.empty_like(w.q)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    l2 = getattr(props, "L2_cache_size", 128 << 20) or (128 << 20)
    resident = (w.k_pages.numel() + w.v_pages.numel()) * 2
    flush, l2_desc = l2_policy(kv_bytes, l2)
    # the flush buffers: for this workload when it fits in twice the L2, and
    # for the per_config block's small workloads
    need_flush = flush or args.config_steps > 0
    flush_buf = torch.empty(4 * l2 // 4, dtype=torch.float32, device=dev) if need_flush else None
    flush_read = torch.ones(4 * l2 // 4, dtype=torch.float32, device=dev) if need_flush else None

    def flush_l2():
        # write 4x L2 (evicts the step's data), then read another 4x L2 so the
        # dirty lines are written back before the timed step, not during it
        flush_buf.zero_()
        flush_read.sum()

    def split_call():
        if args.append:
            pkg.decode_attn_append(w.q, k_new, v_new, w.k_pages, w.v_pages, w.page_table,
                                   w.seq_lens, w.scale, window=w.window, out=out,
                                   max_seq_len=max_len, workspace=ws, err_flag=err,
                                   variant=args.variant, force_chunk=args.force_chunk,
                                   schedule=args.schedule)
            return
        pkg.decode_attn_split(w.q, w.k_pages, w.v_pages, w.page_table, w.seq_lens, w.scale,
                              window=w.window, out=out, max_seq_len=max_len, workspace=ws,
                              err_flag=err, variant=args.variant, force_chunk=args.force_chunk,
                              schedule=args.schedule)

    def step_call():
        # one launch: the split kernel's last CTA per group merges the partials
        split_call()

    for _ in range(args.warmup):
        if flush:
            flush_l2()
        step_call()
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise RuntimeError(f"device error bits {int(err.item())}")

    # The step is captured once as a CUDA graph (the tickets' memset and the
    # split kernel); replays carry no host launch work.  The roofline loop
    # replays it again with events around every launch.
    if args.eager:
        run_step, run_split = step_call, split_call
    else:
        g_step, g_split = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_step):
            step_call()
        with torch.cuda.graph(g_split):
            split_call()
        run_step, run_split = g_step.replay, g_split.replay
        for _ in range(3):
            run_step()
            run_split()
        torch.cuda.synchronize()

    K = args.steps

    def timed_loop(fn):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
        if flush:
            for i in range(K):
                flush_l2()  # between steps, outside the events
                evs[i][0].record(stream)
                fn()
                evs[i][1].record(stream)
            torch.cuda.synchronize()
            per = [e0.elapsed_time(e1) for e0, e1 in evs]
            return sum(per), per
        e0, e1 = evs[0]
        e0.record(stream)
        for _ in range(K):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        total = e0.elapsed_time(e1)
        return total, None

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    total_ms, step_ms = timed_loop(run_step)
    t_wall1 = time.time()
    barrier()
    # split kernel alone, each launch bracketed by events on its stream
    split_evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(K)]
    for i in range(K):
        if flush:
            flush_l2()
        split_evs[i][0].record(stream)
        run_split()
        split_evs[i][1].record(stream)
    torch.cuda.synchronize()
    sampler.stop()
    split_ms = [a.elapsed_time(b) for a, b in split_evs]
    split_avg_ms = statistics.mean(split_ms)
    ms_local = total_ms / K
    ms_max = max_over_ranks(ms_local, dev)
    bytes_all = sum_over_ranks(kv_bytes, dev)
    value_tbs = bytes_all / (ms_max * 1e-3) / 1e12
    peak_gbs, peak_src = load_peak_hbm()
    split_achieved_gbs = kv_bytes / (split_avg_ms * 1e-3) / 1e9
    default_run = T == 1 and not args.append and args.dtype == "fp16"
    traffic = recorded_traffic(args.workload,
                               split_kernel_name(plan, w.head_dim) if default_run else None)
    # ---- every other configuration of the benchmark, timed the same way
    per_config = None
    if rank == 0 and args.config_steps > 0 and T == 1 and not args.append and \
            args.variant == 0 and args.schedule == 0 and args.force_chunk == 0:
        per_config = {}
        for name in PER_CONFIG:
            if name == args.workload:
                continue
            per_config[name] = time_config(pkg, workloads, name, dev, local, args.config_steps,
                                           edt, peak_gbs, flush_l2, l2)
    # ---- end to end from pinned host buffers through the C ABI
    e2e = None
    if args.e2e_steps > 0 and T == 1 and not args.append:
        pin = lambda t: t.to("cpu").contiguous().pin_memory()
        qh, kh, vh, th, lh = map(pin, (w.q, w.k_pages, w.v_pages, w.page_table, w.seq_lens))
        out_h = torch.empty_like(qh).pin_memory()
        d_bufs = [torch.empty_like(t, device=dev) for t in (qh, kh, vh, th, lh, qh)]
        h2d = sum(t.numel() * t.element_size() for t in (qh, kh, vh, th, lh))
        d2h = out_h.numel() * out_h.element_size()
        for _ in range(2):
            pkg.decode_attn_host(params, qh, kh, vh, th, lh, out_h, *d_bufs, ws, 0, err)
        torch.cuda.synchronize()
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.e2e_steps):
            pkg.decode_attn_host(params, qh, kh, vh, th, lh, out_h, *d_bufs, ws, 0, err)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.e2e_steps, dev)
        if not torch.equal(out_h, out.cpu()):
            raise RuntimeError("host-buffer path disagrees with the device path")
        e2e = {"value": bytes_all / (e2e_ms * 1e-3) / 1e12, "unit": "TB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e2e_ms, "steps": args.e2e_steps,
               "path": "decode_attn_host: pinned host -> device copies, kernels, out -> host"}
        del d_bufs, qh, kh, vh

    if int(err.item()) != 0:
        raise RuntimeError(f"device error bits {int(err.item())}")

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cores = cpu_cores()
        smp = OracleSample(w.to("cpu"), cores).calibrate(args.cpu_budget)
        nbytes, secs = smp.run()
        cpu = {"value": nbytes / secs / 1e12, "unit": "TB/s", "cores": cores, "kind": "oracle",
               "sample": smp.describe(nbytes), "seconds": round(secs, 2), "cpu": cpu_model()}
        if w.kv_bytes() < (1 << 30) and cores > 1:
            # the smaller workloads: the same sample on one thread as well
            one = OracleSample(w.to("cpu"), 1).calibrate(min(5.0, args.cpu_budget))
            nb1, secs1 = one.run()
            cpu["one_thread"] = {"value": nb1 / secs1 / 1e12, "unit": "TB/s",
                                 "sample": one.describe(nb1), "seconds": round(secs1, 2)}

    clocks = sampler.summary(t_wall0, t_wall1)
    if rank == 0:
        line = {
            "metric": METRIC, "value": value_tbs, "unit": "TB/s", "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": ms_max,
            "us_per_step": ms_max * 1e3, "hbm_frac": value_tbs * 1e3 / peak_gbs,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": f"{args.dtype} in / fp32 accumulate",
            "data": f"synthetic (seeded N(0,1) {args.dtype})",
            "config": {"workload": args.workload, "desc": WORKLOAD_DESC[args.workload],
                       "queries_per_seq": T, "fused_append": bool(args.append),
                       "kv_bytes_per_step": kv_bytes, "resident_kv_bytes": resident,
                       "l2": l2_desc, "parallelism": f"replicas x{world}"},
            "plan": plan.as_dict(),
            "roofline": {"bound": "hbm", "kernel": split_kernel_name(plan, w.head_dim),
                         "achieved": split_achieved_gbs, "peak": peak_gbs, "unit": "GB/s",
                         "frac": split_achieved_gbs / peak_gbs, "peak_source": peak_src,
                         "traffic": traffic,
                         # every byte the launch moves (ncu DRAM read + write:
                         # K/V, q, page table, partials, out) over its time
                         "traffic_gbs": (traffic / (split_avg_ms * 1e-3) / 1e9
                                         if traffic else None),
                         "algorithmic_bytes_per_launch": kv_bytes,
                         "launch_us": split_avg_ms * 1e3,
                         "launch_us_percentiles": percentiles_us(split_ms)},
            "step_us_percentiles": percentiles_us(step_ms) if step_ms else None,
            "cpu_baseline": cpu, "e2e": e2e, "per_config": per_config,
            "gpu_launches": K,
            "launch_mode": "eager" if args.eager else "cuda graph replay",
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
        if args.dump:
            import numpy as np
            np.savez(args.dump, out=out.float().cpu().numpy(), workload=args.workload,
                     dtype=args.dtype, queries=T, append=bool(args.append),
                     plan=json.dumps(plan.as_dict()))


# ------------------------------------------------------------ context sweep

SWEEP_CONTEXTS = (1, 2, 3, 8, 32, 64, 128, 192, 255, 256, 257, 320, 384, 448, 512)


def context_sweep(args):
    """Threshold A/B over short contexts (the 256-token split threshold):
    every point is timed like the bench's small workloads (graph replay, L2
    flushed before each step, events around it)."""
    import torch
    import paged_gqa_decode_06_gb300 as pkg
    from paged_gqa_decode_06_gb300 import build, workloads

    rank, world, local = dist_env()
    if rank != 0:
        return
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build.build()
    pkg.load_library()
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 128 << 20) or (128 << 20)
    flush_w = torch.empty(4 * l2 // 4, dtype=torch.float32, device=dev)
    flush_r = torch.ones(4 * l2 // 4, dtype=torch.float32, device=dev)
    K = max(10, min(args.steps, 300))
    modes = (("threshold 256", 0), ("always split", 1), ("single pass to 512", 512))
    summary = {}
    for shape in ("d64", "d128", "d256"):
        for ctx in SWEEP_CONTEXTS:
            w = workloads.make(f"ctx{ctx}_{shape}", device=dev)
            out = torch.empty_like(w.q)
            for label, split_min in modes:
                params = pkg.make_params(w.q, w.k_pages, w.page_table, w.scale, 0, ctx, 0,
                                         split_min)
                plan = pkg.decode_attn_make_plan(params, props.multi_processor_count)
                ws = torch.zeros(max(pkg.decode_attn_workspace_size(params, local), 256),
                                 dtype=torch.uint8, device=dev)

                def step():
                    pkg.decode_attn(w.q, w.k_pages, w.v_pages, w.page_table, w.seq_lens, w.scale,
                                    out=out, max_seq_len=ctx, workspace=ws, split_min=split_min)

                for _ in range(3):
                    step()
                torch.cuda.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    step()
                evs = []
                for _ in range(K):
                    flush_w.zero_()
                    flush_r.sum()
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record()
                    g.replay()
                    e1.record()
                    evs.append((e0, e1))
                torch.cuda.synchronize()
                us = statistics.median(a.elapsed_time(b) for a, b in evs) * 1e3
                summary.setdefault(label, []).append(us)
                print(json.dumps({"sweep": "context", "shape": shape, "context": ctx,
                                  "mode": label, "split": plan.split,
                                  "shards": plan.max_shards, "us_per_step_median": us,
                                  "steps": K}), flush=True)
                del g, ws
    print(json.dumps({"sweep": "context", "summary_mean_us": {
        k: statistics.mean(v) for k, v in summary.items()}, "points": len(SWEEP_CONTEXTS) * 3,
        "l2": "flushed before every step (write of 4x L2, then read of 4x L2)"}), flush=True)


# ------------------------------------------------------------ reference arm

def reference_arm(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return  # rank 0 alone times the oracle
    import torch
    from paged_gqa_decode_06_gb300 import workloads
    import oracle
    oracle.build()
    w = workloads.make(args.workload, device="cpu")
    kv_bytes = w.kv_bytes()
    resident = (w.k_pages.numel() + w.v_pages.numel()) * 2
    # the GPU arm's L2 rule, so both arms name the same configuration
    l2 = 126 << 20
    if torch.cuda.is_available():
        l2 = getattr(torch.cuda.get_device_properties(0), "L2_cache_size", l2) or l2
    cores = cpu_cores()
    steps = args.steps + args.warmup
    per_step = max(0.02, min(5.0, 120.0 / steps))
    smp = OracleSample(w, cores).calibrate(per_step)  # untimed
    times, nbytes = [], 0
    for i in range(steps):
        b, secs = smp.run()
        if i >= args.warmup:
            times.append(secs)
            nbytes += b
    desc = smp.describe(nbytes / max(1, len(times)))
    total = sum(times)
    value = nbytes / total / 1e12
    ms = total / max(1, len(times)) * 1e3
    line = {
        "metric": METRIC, "value": value, "unit": "TB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1) fp16)",
        "impl": "reference",
        "config": {"workload": args.workload, "desc": WORKLOAD_DESC[args.workload],
                   "queries_per_seq": 1, "fused_append": False,
                   "kv_bytes_per_step": kv_bytes, "resident_kv_bytes": resident,
                   "l2": l2_policy(kv_bytes, l2)[1], "parallelism": f"replicas x{world}"},
        "cpu_baseline": {"value": value, "unit": "TB/s", "cores": cores, "kind": "oracle",
                         "sample": f"per step: {desc}", "cpu": cpu_model()},
        "e2e": {"value": value, "unit": "TB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    del torch
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        reference_arm(args)
    elif args.context_sweep:
        context_sweep(args)
    else:
        gpu_arm(args)
    import torch.distributed as dist
    if dist.is_initialized():
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
