"""Benchmark of the fused attention forward pass on GB300.

python bench.py --gpus N --steps K --warmup W [--impl reference] [--causal]

One step = one forward pass over the whole workload (bf16 B=2 H=16 N=8192
d=128, non-causal, the long-sequence head-dim-128 setting) with Q, K, V
already resident in HBM.  W untimed steps, then exactly K timed steps
bracketed by a barrier and a device synchronise.  L2 is flushed (a 256 MiB
write) before every timed step, outside the kernel's events.  The kernel
time is measured with CUDA events on the launching stream; `value` is the
whole-job throughput in TFLOP/s (4*B*H*N^2*d FLOPs per step, halved when
causal), the max over ranks.  With N GPUs every rank runs its own copy of
the workload (independent heads; no exchange), so scaling is weak.  Under
torchrun the ranks come from its environment; `--gpus N` without it starts
the N ranks itself (torch.distributed.run on 127.0.0.1, one rank per GPU).

Also reported: `e2e` (the same metric through the public C-ABI call with the
inputs copied from pinned host memory and O/LSE copied back every step),
`roofline` (achieved TFLOP/s of the kernel against the measured dense bf16
peak), `clocks` (nvidia-smi during the timed region), `per_config` (at one
GPU: the causal bf16 and the e4m3 N=8192 d=128 workloads, timed the same way
after the headline) and `cpu_baseline` (the fp64 oracle timed on the host
cores on a bounded sample of the workload).

--impl reference times that oracle alone, on the same workload, metric and
unit (each step a bounded sample of rows), and prints the same JSON line
with "impl": "reference".
"""
from __future__ import annotations

import argparse
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import attn_inputs as ai  # noqa: E402

WORKLOAD = "bf16_n8192_d128"
METRIC = "attention fwd TFLOPs/s on 1 GB300 (and % of dense BF16/FP8 tensor peak)"
UNIT = "TFLOP/s"
FALLBACK_BF16_TFLOPS = 1900.0
L2_FLUSH_BYTES = 256 << 20
KERNEL_NAME = "attn_fwd_kernel"


# ----------------------------------------------------------------- helpers

def dist_env():
    """(rank, local_rank, world) from the torchrun environment."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def free_port() -> int:
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def launch_command(nproc: int, argv, port: int):
    """torch.distributed.run command that re-runs this script as nproc ranks
    on this node (rendezvous on 127.0.0.1)."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
            f"--nproc-per-node={nproc}", "--master-addr", "127.0.0.1", "--master-port",
            str(port), os.path.abspath(__file__), *argv]


def check_world(gpus: int):
    """None when this process should run as a rank; otherwise the number of
    ranks to start.  Raises ValueError when a launcher's world size
    contradicts --gpus."""
    env = os.environ.get("WORLD_SIZE")
    if env is None:
        return gpus if gpus > 1 else None
    if int(env) != gpus:
        raise ValueError(f"WORLD_SIZE={env} but --gpus {gpus}")
    return None


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The max of x over all ranks (x itself when world == 1)."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(flops_per_step: float, steps: int, world: int, max_time_s: float) -> float:
    """Whole-job TFLOP/s: every rank ran `steps` steps of the workload."""
    return world * steps * flops_per_step / max_time_s / 1e12


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops, burst)"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback (no MEASURED_PEAKS.json)"


# The sources the timed forward kernel is built from (a change to any of
# them invalidates the profiled traffic figure).
KERNEL_SOURCES = ("ptx_sm103.cuh", "attn_fwd_kernel.cuh", "attn_fwd_tail.cuh", "attn_launch.h",
                  "attn_instance.cuh", "inst_bf16.cu")


def kernel_source_digest() -> str:
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "warp_specialized_gb300", "csrc")
    for name in KERNEL_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch of the timed kernel from the committed ncu
    summary, if it was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", f"{KERNEL_NAME}_{WORKLOAD}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*(\d+)\s+source_digest:\s*([0-9a-f]+)", text)
    if not m or m.group(2) != kernel_source_digest():
        return None
    return int(m.group(1))


class ClockSampler:
    """nvidia-smi sampling of SM clock, power and throttle reasons; only the
    samples taken inside the timed region (by their timestamps) count."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 20):
        self.gpu = gpu_index
        self.period = period_ms
        self.proc = None
        self.out = None

    def start(self):
        try:
            self.out = tempfile.TemporaryFile(mode="w+")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 f"-lms", str(self.period), "-i", str(self.gpu)],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    @staticmethod
    def summarise(lines, t_begin=None, t_end=None):
        """Median SM clock, max clock and power, and the throttle reasons seen,
        over the samples whose timestamps (host wall clock, seconds) lie in
        [t_begin, t_end]; all samples when no window is given or none falls
        in it (then "window" says so)."""
        import datetime
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        parsed = []
        for line in lines:
            r = [x.strip() for x in line.split(",")]
            if len(r) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                vals = (float(r[2]), float(r[3]), float(r[4]))
            except ValueError:
                continue
            active = [n for n, v in zip(names, r[6:10]) if v.lower().startswith("active")]
            parsed.append((ts, vals, active))
        window = "timed region"
        sel = parsed
        if t_begin is not None:
            sel = [p for p in parsed if t_begin <= p[0] <= t_end]
            if not sel:
                sel, window = parsed, "whole run (no sample inside the timed region)"
        sm = [p[1][0] for p in sel]
        reasons = sorted({n for p in sel for n in p[2]})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(p[1][1] for p in sel) if sel else None,
                "power_w_max": max(p[1][2] for p in sel) if sel else None,
                "reasons": reasons, "samples": len(sel), "samples_total": len(parsed),
                "window": window}

    def stop(self, t_begin=None, t_end=None):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.seek(0)
        return self.summarise(self.out.read().strip().splitlines(), t_begin, t_end)


# ----------------------------------------------------------------- GPU arm

def run_gpu(args):
    import torch
    import torch.distributed as dist

    import warp_specialized_gb300 as ws

    rank, local_rank, world = dist_env()
    if local_rank >= torch.cuda.device_count():
        raise RuntimeError(f"rank {rank}: local rank {local_rank} but only "
                           f"{torch.cuda.device_count()} GPU(s) visible")
    if world > 1:
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    ws.load_library(build_if_missing=True)

    inp = ai.workload(WORKLOAD)
    B, H, N, d = inp.shape
    causal = bool(args.causal)
    flops = ai.workload_flops(B, H, N, d, causal)
    q, k, v = (t.to(dev) for t in (inp.q, inp.k, inp.v))
    o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream
    qp, kp, vp, op, lp = q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr()

    # the library's own advice on splitting the work left after whole rounds
    # (attn_fwd_ws) for this shape; the kernels one call launches
    split = ws.attn_fwd_split_advised(B, H, N, d, causal, ws.ATTN_BF16)
    wsp = None
    launches = 1
    if split:
        wsp = torch.empty(ws.attn_fwd_workspace_size(d, ws.ATTN_BF16), dtype=torch.uint8,
                          device=dev)
        n_items = B * H * -(-(-(-N // 128)) // 2)
        launches = 2 if n_items >= torch.cuda.get_device_properties(dev).multi_processor_count else 1

    def fwd_call(qp_, kp_, vp_, op_, lp_, sh_):
        if wsp is None:
            return ws.attn_fwd_raw(qp_, kp_, vp_, op_, lp_, B, H, N, d, inp.scale, causal,
                                   ws.ATTN_BF16, sh_)
        return ws.attn_fwd_ws_raw(qp_, kp_, vp_, op_, lp_, B, H, N, d, inp.scale, causal,
                                  ws.ATTN_BF16, wsp.data_ptr(), wsp.numel(), sh_)

    def step():
        rc = fwd_call(qp, kp, vp, op, lp, sh)
        if rc != 0:
            raise ws.AttnError(rc)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    if ws.attn_fwd_status() != 0:
        raise RuntimeError("watchdog fired during warm-up")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sampler = ClockSampler(local_rank if world > 1 else torch.cuda.current_device())
    sampler.start()
    time.sleep(0.3)  # let the sampler start before the timed region
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_begin = time.time()
    t0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    t_end = time.time()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop(t_begin, t_end)
    if ws.attn_fwd_status() != 0:
        raise RuntimeError("watchdog fired during the timed region")
    kernel_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_s = sum(kernel_ms) / 1e3
    # the same steps back to back, without the L2 flush between them
    # (reported beside the flushed number, not used for `value`)
    nf_steps = max(3, min(args.steps, 50))
    nf0, nf1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    nf0.record(stream)
    for _ in range(nf_steps):
        step()
    nf1.record(stream)
    torch.cuda.synchronize()
    no_flush_ms = nf0.elapsed_time(nf1) / nf_steps
    sorted_ms = sorted(kernel_ms)
    max_total_s = max_over_ranks(total_s, world, dev)
    value = weak_scaling_value(flops, args.steps, world, max_total_s)
    avg_ms = max_total_s / args.steps * 1e3
    achieved = flops / (avg_ms / 1e3) / 1e12

    # End to end through the public call: every step copies its inputs from
    # pinned host memory, runs the forward pass and copies O and LSE back.
    # Steps are independent, so they are pipelined the way a serving loop
    # would run them: two device buffer sets, the input copies of step i+1
    # (one stream) overlap the kernel of step i (a second stream) and the
    # output copies of step i-1 (a third), ordered by events.
    e2e_steps = 0 if args.no_e2e else max(2, min(args.steps, 100))
    hq, hk, hv = (t.pin_memory() for t in (inp.q, inp.k, inp.v))
    ho = [torch.empty((B, H, N, d), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    hl = [torch.empty((B, H, N), dtype=torch.float32).pin_memory() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = ho[0].numel() * ho[0].element_size() + hl[0].numel() * hl[0].element_size()
    e2e_value = None
    if e2e_steps:
        bufs = [dict(q=q, k=k, v=v, o=o, l=lse)]
        bufs.append(dict(q=torch.empty_like(q), k=torch.empty_like(k), v=torch.empty_like(v),
                         o=torch.empty_like(o), l=torch.empty_like(lse)))
        s_in, s_run, s_out = (torch.cuda.Stream(device=dev) for _ in range(3))
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_run = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]
        for b in range(2):  # mark every buffer free
            ev_run[b].record(s_run)
            ev_out[b].record(s_out)

        def e2e_step(i):
            b = i & 1
            bb = bufs[b]
            with torch.cuda.stream(s_in):
                s_in.wait_event(ev_run[b])          # the kernel of step i-2 has read them
                bb["q"].copy_(hq, non_blocking=True)
                bb["k"].copy_(hk, non_blocking=True)
                bb["v"].copy_(hv, non_blocking=True)
                ev_in[b].record(s_in)
            s_run.wait_event(ev_in[b])
            s_run.wait_event(ev_out[b])             # O / LSE of step i-2 are copied out
            rc = fwd_call(bb["q"].data_ptr(), bb["k"].data_ptr(), bb["v"].data_ptr(),
                          bb["o"].data_ptr(), bb["l"].data_ptr(), s_run.cuda_stream)
            if rc != 0:
                raise ws.AttnError(rc)
            ev_run[b].record(s_run)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_run[b])
                ho[b].copy_(bb["o"], non_blocking=True)
                hl[b].copy_(bb["l"], non_blocking=True)
                ev_out[b].record(s_out)

        for i in range(6):  # warm-up: both buffer sets, the copy engines, the host pages
            e2e_step(i)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        es.record(s_in)
        for i in range(e2e_steps):
            e2e_step(i)
        s_out.wait_event(ev_out[(e2e_steps - 1) & 1])
        ee.record(s_out)
        torch.cuda.synchronize()
        e2e_s = max_over_ranks(es.elapsed_time(ee) / 1e3, world, dev)
        e2e_value = round(weak_scaling_value(flops, e2e_steps, world, e2e_s), 2)
        if ws.attn_fwd_status() != 0:
            raise RuntimeError("watchdog fired during the end-to-end leg")

    peak, peak_src = load_peaks()
    per_config = None
    if world == 1 and not args.no_per_config:
        per_config = time_other_configs(ws, dev, peak, stream)
    result = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(avg_ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"{WORKLOAD} (B={B} H={H} N={N} d={d}, "
                               f"{'causal' if causal else 'non-causal'}, N(0,1) inputs)",
                   "B": B, "H": H, "N": N, "d": d, "causal": causal,
                   "flops_per_step": flops,
                   "l2": "flushed before every timed step (256 MiB write, outside the events)",
                   "parallelism": f"replica per GPU x{world} (independent heads, no exchange)"},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "schedule": "steps pipelined over two buffer sets: H2D(i+1) || kernel(i) || D2H(i-1)"},
        "gpu_launches": launches * (args.steps + nf_steps + e2e_steps),
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
                     "unit": UNIT, "frac": round(achieved / peak, 4),
                     "traffic": profiled_traffic(), "peak_source": peak_src,
                     "kernel": KERNEL_NAME},
        "timing": {"ms_per_step_median": round(sorted_ms[len(sorted_ms) // 2], 4),
                   "ms_per_step_min": round(sorted_ms[0], 4),
                   "ms_per_step_no_l2_flush": round(no_flush_ms, 4),
                   "no_l2_flush_steps": nf_steps},
        "clocks": clocks,
        "wall_s_timed_region": round(wall, 4),
    }
    if per_config is not None:
        result["per_config"] = per_config
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return result, rank, world


def time_other_configs(ws, dev, peak: float, stream, steps: int = 10):
    """CUDA-event TFLOP/s and roofline fraction of the causal bf16 workload
    and of the e4m3 workload (per-tensor descales, its peak taken as twice
    the measured bf16 one, the nominal dense ratio), each step after an L2
    flush, median of `steps`."""
    import torch
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    out = {}
    for name, causal in (("bf16_n8192_d128", True), ("fp8_n8192_d128", False)):
        inp = ai.workload(name)
        B, H, N, d = inp.shape
        q, k, v = (t.to(dev) for t in (inp.q, inp.k, inp.v))
        o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        sh = stream.cuda_stream
        lib = ws.load_library()
        if inp.dtype == "fp8":
            ds = inp.descale
            call = lambda: lib.attn_fwd_fp8(q.data_ptr(), k.data_ptr(), v.data_ptr(),  # noqa: E731
                                            o.data_ptr(), lse.data_ptr(), B, H, N, d, inp.scale,
                                            int(causal), ds["q"], ds["k"], ds["v"], sh)
            pk, dt = 2.0 * peak, "e4m3"
        else:
            call = lambda: ws.attn_fwd_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(),  # noqa: E731
                                           o.data_ptr(), lse.data_ptr(), B, H, N, d, inp.scale,
                                           causal, ws.ATTN_BF16, sh)
            pk, dt = peak, "bf16"
        for _ in range(3):
            flush.zero_()
            if call() != 0:
                raise RuntimeError(f"{name}: launch failed")
        ms = []
        for _ in range(steps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            call()
            e1.record(stream)
            e1.synchronize()
            ms.append(e0.elapsed_time(e1))
        if ws.attn_fwd_status() != 0:
            raise RuntimeError(f"{name}: watchdog fired")
        med = sorted(ms)[len(ms) // 2]
        tf = ai.workload_flops(B, H, N, d, causal) / med / 1e9
        out[f"{name}{'_causal' if causal else ''}"] = {
            "dtype": dt, "causal": causal, "B": B, "H": H, "N": N, "d": d,
            "ms_median": round(med, 4), "tflops": round(tf, 1), "peak": pk,
            "frac": round(tf / pk, 4), "steps": steps,
            "peak_source": "measured bf16 burst" + (" x 2 (nominal e4m3:bf16 dense ratio)"
                                                    if dt == "e4m3" else "")}
        del q, k, v, o, lse
    return out


# ------------------------------------------------------------- CPU oracle

def oracle_sample(target_s: float, seed: int = 0):
    """Times the fp64 oracle on seeded rows of every head of the workload,
    sized to take about target_s seconds.  Returns (TFLOP/s, seconds, rows,
    threads, description)."""
    import numpy as np

    import oracle
    inp = ai.workload(WORKLOAD)
    B, H, N, d = inp.shape
    q, k, v = (x.numpy() for x in inp.as_float64())
    g = np.random.default_rng(seed)
    # warm the thread pool, then calibrate on 8 rows per head
    oracle.attn_fwd(q, k, v, inp.scale, False, rows=g.choice(N, size=1, replace=False))
    rows = g.choice(N, size=8, replace=False)
    t0 = time.perf_counter()
    oracle.attn_fwd(q, k, v, inp.scale, False, rows=rows)
    dt = time.perf_counter() - t0
    per_row = dt / (8 * B * H)
    n_rows = int(max(2, min(N, target_s / max(per_row, 1e-9) / (B * H))))
    rows = g.choice(N, size=n_rows, replace=False)
    t0 = time.perf_counter()
    oracle.attn_fwd(q, k, v, inp.scale, False, rows=rows)
    dt = time.perf_counter() - t0
    fl = 4.0 * N * d * n_rows * B * H
    desc = (f"{n_rows} seeded query rows x all {B * H} heads of {WORKLOAD} "
            f"({n_rows * B * H} rows, {fl / 1e9:.1f} GFLOP), non-causal, fp64")
    return fl / dt / 1e12, dt, n_rows, oracle.max_threads(), desc


def run_reference(args):
    """The oracle alone on the host cores, same metric/unit/workload."""
    rank, _, world = dist_env()
    if rank != 0:
        return None, rank, world
    per_step_target = max(0.5, min(10.0, 60.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(per_step_target / 4)
    rates, times = [], []
    desc = ""
    cores = 1
    for i in range(args.steps):
        tf, dt, n_rows, cores, desc = oracle_sample(per_step_target, seed=i + 1)
        rates.append(tf)
        times.append(dt)
    value = statistics.median(rates)
    inp_shape = ai.WORKLOADS[WORKLOAD][:4]
    B, H, N, d = inp_shape
    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": statistics.median(times) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": {"workload": f"{WORKLOAD} (B={B} H={H} N={N} d={d}, non-causal, N(0,1) "
                               "inputs); each step a bounded row sample",
                   "B": B, "H": H, "N": N, "d": d, "causal": False},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    return result, rank, world


def launch_selftest():
    """One rank of the launcher check: gloo process group, the max over
    ranks of (rank + 1), and rank 0 prints the world it saw."""
    import torch.distributed as dist
    rank, local_rank, world = dist_env()
    if world > 1:
        dist.init_process_group("gloo")
    m = max_over_ranks(rank + 1.0, world)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps({"launch_selftest": True, "n_gpus": world, "max_over_ranks": m}),
              flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--causal", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end leg (profiling)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the causal and e4m3 timings after the headline")
    ap.add_argument("--launch-selftest", action="store_true",
                    help="start the ranks, exchange one value over gloo and report; no GPU work")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.gpus < 1:
        ap.error("--gpus must be >= 1")
    try:
        nproc = check_world(args.gpus)
    except ValueError as e:
        ap.error(str(e))
    if nproc is not None:
        sys.exit(subprocess.call(launch_command(nproc, sys.argv[1:], free_port())))

    if args.launch_selftest:
        launch_selftest()
        return

    if args.impl == "reference":
        result, rank, _ = run_reference(args)
        if rank == 0:
            print(json.dumps(result), flush=True)
        return

    result, rank, world = run_gpu(args)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            tf, dt, n_rows, cores, desc = oracle_sample(args.cpu_seconds)
            result["cpu_baseline"] = {"value": tf, "unit": UNIT, "cores": cores,
                                      "kind": "oracle", "sample": desc,
                                      "seconds": round(dt, 2),
                                      "full_workload_s_extrapolated":
                                          round(result["config"]["flops_per_step"] / (tf * 1e12), 1)}
        print(json.dumps(result), flush=True)


if __name__ == "__main__":
    main()
