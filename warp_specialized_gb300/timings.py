"""Kernel timings behind the results tables: the forward pass on every
workload and mask, the backward pass, and the e4m3 quantiser.

    python -m warp_specialized_gb300.timings [--only fwd,bwd,quant] [--steps 20] [--json FILE]

Attention steps are timed one at a time with CUDA events on the current
stream, each after a 256 MiB write that flushes L2, and the median is
reported.  The quantiser's inputs (268 MB and more) are larger than L2, so
its launches are timed back to back.  Every input is the seeded synthetic
workload of `attn_inputs`; the watchdog word is read after every case.
"""
from __future__ import annotations

import argparse
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

FWD_CASES = [("bf16_n8192_d128", None), ("bf16_n2048_d128", None), ("outlier_d64", "bf16"),
             ("outlier_d64", "fp16"), ("outlier_d256", "bf16"), ("outlier_d256", "fp16"),
             ("fp8_n8192_d128", None)]
BWD_CASES = ["bf16_n8192_d128", "bf16_n2048_d128"]
QUANT_CASES = [("bf16", 128), ("bf16", 64), ("fp16", 128), ("fp32", 128), ("fp32", 64)]


def _hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"])
    except (OSError, KeyError, ValueError):
        return None


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--only", default="fwd,bwd,quant")
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--json", default=None, help="also write the results to this file")
    ap.add_argument("--cases", default=None,
                    help="forward cases to run, comma-separated workload[:dtype]:mask, e.g. "
                         "fp8_n8192_d128:nc,outlier_d64:bf16:causal (default: all)")
    ap.add_argument("--split", choices=["auto", "on", "off"], default="auto",
                    help="the forward's split tail launch: where it pays (auto), always, never")
    ap.add_argument("--exp2-fma", action="store_true",
                    help="time the forward with ATTN_OPT_EXP2_FMA (4 of every 32 exponentials "
                         "on the FMA pipe; bf16 d = 64 / 128 and e4m3 d = 128)")
    ap.add_argument("--shape", default=None,
                    help="time only this forward shape B,H,N,d (bf16, N(0,1) inputs, both "
                         "masks unless --cases names one: e.g. --cases x:nc)")
    args = ap.parse_args(argv)
    parts = set(args.only.split(","))

    import torch

    import attn_inputs as ai
    import warp_specialized_gb300 as ws

    ws.load_library(build_if_missing=True)
    flush = torch.empty(64 << 20, dtype=torch.float32, device="cuda")
    results = {}

    def median_ms(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(args.steps):
            flush.zero_()
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            fn()
            e.record()
            e.synchronize()
            ts.append(s.elapsed_time(e))
        return sorted(ts)[len(ts) // 2]

    def record(key, **kw):
        status = ws.attn_fwd_status()
        if status != 0:
            raise RuntimeError(f"{key}: watchdog status {status}")
        results[key] = kw
        print(key, " ".join(f"{k}={v}" for k, v in kw.items()), flush=True)

    if "fwd" in parts:
        wanted = None
        if args.cases:
            wanted = set()
            for c in args.cases.split(","):
                f = c.split(":")
                wanted.add((f[0], f[1] if len(f) == 3 else None, f[-1] == "causal"))
        fwd_cases = FWD_CASES
        if args.shape:
            fwd_cases = [("shape", None)]
            if wanted is not None:
                wanted = {("shape", None, m) for (_, _, m) in wanted}
        for name, dt in fwd_cases:
            masks = [m for m in (False, True) if wanted is None or (name, dt, m) in wanted]
            if not masks:
                continue
            if name == "shape":
                Bs, Hs, Ns, ds_ = (int(x) for x in args.shape.split(","))
                inp = ai.make_inputs(Bs, Hs, Ns, ds_, "bf16", seed=11)
                name = f"B{Bs}_H{Hs}_N{Ns}_d{ds_}"
            else:
                inp = ai.workload(name, dt)
            q, k, v = (t.cuda() for t in (inp.q, inp.k, inp.v))
            B, H, N, d = inp.shape
            split = {"auto": None, "on": True, "off": False}[args.split]
            wsp = None
            if split is not False and not args.exp2_fma:
                code = ws.ATTN_FP8_E4M3 if inp.dtype == "fp8" else ws.ATTN_BF16
                wsp = torch.empty(ws.attn_fwd_workspace_size(d, code), dtype=torch.uint8,
                                  device="cuda")
            o = torch.empty((B, H, N, d), dtype=torch.bfloat16 if inp.dtype == "fp8" else q.dtype,
                            device="cuda")
            lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
            for causal in masks:
                if inp.dtype == "fp8":
                    ds = inp.descale
                    fn = lambda: ws.attn_fwd_fp8(q, k, v, ds["q"], ds["k"], ds["v"],  # noqa: E731
                                                 scale=inp.scale, causal=causal, out=o, lse=lse,
                                                 split_tail=split, workspace=wsp,
                                                 exp2_fma=args.exp2_fma)
                else:
                    fn = lambda: ws.attn_fwd(q, k, v, scale=inp.scale, causal=causal,  # noqa: E731
                                             out=o, lse=lse, split_tail=split, workspace=wsp,
                                             exp2_fma=args.exp2_fma)
                ms = median_ms(fn)
                fl = ai.workload_flops(B, H, N, d, causal)
                record(f"fwd {name}:{inp.dtype}:{'causal' if causal else 'nc'}"
                       + (":exp2_fma" if args.exp2_fma else ""),
                       ms=round(ms, 4), tflops=round(fl / ms / 1e9, 1))
            del q, k, v, o, lse, wsp

    if "bwd" in parts:
        for name in BWD_CASES:
            inp = ai.workload(name)
            B, H, N, d = inp.shape
            q, k, v = (t.cuda() for t in (inp.q, inp.k, inp.v))
            dout = ai.make_inputs(B, H, N, d, "bf16", seed=7).q.cuda()
            for causal in (False, True):
                o, lse = ws.attn_fwd(q, k, v, scale=inp.scale, causal=causal)
                wsp = torch.empty(ws.attn_bwd_workspace_size(B, H, N), dtype=torch.uint8,
                                  device="cuda")
                dq, dk, dv = (torch.empty_like(q) for _ in range(3))
                ms = median_ms(lambda: ws.attn_bwd(q, k, v, o, lse, dout, scale=inp.scale,
                                                   causal=causal, dq=dq, dk=dk, dv=dv,
                                                   workspace=wsp))
                fl = 2.5 * ai.workload_flops(B, H, N, d, causal)
                record(f"bwd {name}:{'causal' if causal else 'nc'}", ms=round(ms, 4),
                       tflops_2p5x_fwd=round(fl / ms / 1e9, 1))
            del q, k, v, dout

    if "quant" in parts:
        peak = _hbm_peak()
        for dtype, d in QUANT_CASES:
            x = ai.make_inputs(8, 16, 8192, d, dtype, seed=3).q.cuda()
            B, H, N, _ = x.shape
            codes = torch.empty(x.shape, dtype=torch.float8_e4m3fn, device="cuda")
            scales = torch.empty((B, H, N // 128), dtype=torch.float32, device="cuda")
            nbytes = x.numel() * x.element_size() + x.numel() + scales.numel() * 4
            for had in (False, True):
                fn = lambda: ws.attn_quantize_fp8(x, hadamard=had, codes=codes,  # noqa: E731
                                                  scales=scales)
                for _ in range(3):
                    fn()
                s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                s.record()
                for _ in range(args.steps):
                    fn()
                e.record()
                e.synchronize()
                us = s.elapsed_time(e) / args.steps * 1e3
                gbs = nbytes / us / 1e3
                kw = dict(us=round(us, 1), gbs=round(gbs))
                if peak:
                    kw["frac_of_measured_hbm"] = round(gbs / peak, 3)
                record(f"quant {dtype} d={d} {'hadamard' if had else 'plain'}", **kw)
            del x, codes

    if args.json:
        with open(args.json, "w") as f:
            json.dump(results, f, indent=1)


if __name__ == "__main__":
    main()
