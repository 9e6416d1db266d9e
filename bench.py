#!/usr/bin/env python3
"""Benchmark of the DCP MLA decode hot path on GB300.

One step = dcp_mla_decode_partial + dcp_lse_combine over one batch of the
workload (default: long-context decode, B=1, 120,000 context tokens, 128
heads, D=8 shards, interleave 1, block size 64), all inputs resident in HBM.
The metric is KV tokens/s of the whole step; the line also carries the
decode kernel's HBM roofline fraction (algorithmic bytes / event-timed
duration), the combine's GB/s, an end-to-end figure through the C ABI with
host buffers, and the float64 CPU oracle timed on this host.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
                  [--workload NAME]

Under torchrun (N > 1) each rank runs an independent replica (the path has no
exchange on one GPU); value = all ranks' tokens / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "MLA DCP decode KV tokens/s + combine GB/s, % of GB300 HBM roofline"
UNIT = "KV tokens/s"
L2_FLUSH_BYTES = 512 << 20
KV_ROW_BYTES = 576 * 2
# DRAM bytes (read + write) of one tensor-core decode launch on the 120k
# long-context workload, from one ncu capture of that launch.  They describe
# only the kernel source they were taken on, so they are reported only while
# that file's hash matches.
MEASURED_TRAFFIC = {
    "workload": "long_ctx_120k_b1_d8_i1",
    "source": "mla_decode_context_gb300/csrc/dcp_decode_tc.cu",
    "sha256": "087b48f9079aa297584983834872647c73c7b55ea0dbce2e4812179de1992fe6",
    "bytes": 138481152 + 3569664,
}


def measured_traffic(workload: str):
    import hashlib
    if workload != MEASURED_TRAFFIC["workload"] or os.environ.get("DCP_FORCE_SIMT") == "1":
        return None
    try:
        with open(os.path.join(ROOT, MEASURED_TRAFFIC["source"]), "rb") as f:
            digest = hashlib.sha256(f.read()).hexdigest()
    except OSError:
        return None
    return MEASURED_TRAFFIC["bytes"] if digest == MEASURED_TRAFFIC["sha256"] else None


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def tensor_peak():
    """Dense bf16 tensor peak (TFLOP/s): the burst cuBLAS figure, since one
    decode launch is timed on its own."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def decode_flops(inp) -> int:
    """Algorithmic tensor work of one decode launch: every row scores each of
    its causal tokens (L_r = seq_len - (q_len - 1 - i)) on 576 dims and
    accumulates 512 value dims, for all H heads."""
    seq = np.asarray(inp["seq_lens"], dtype=np.int64)
    qsl = np.asarray(inp["query_start_loc"], dtype=np.int64)
    rows = 0
    for b in range(inp["B"]):
        q = int(qsl[b + 1] - qsl[b])
        if seq[b] <= 0 or q <= 0:
            continue
        rows += int(np.clip(seq[b] - (q - 1 - np.arange(q)), 0, None).sum())
    return 2 * inp["H"] * (576 + 512) * rows


def kv_tokens(inp) -> int:
    """KV tokens one step streams: every request's context once (its
    verification rows share the load)."""
    return int(np.asarray(inp["seq_lens"], dtype=np.int64).sum())


def decode_bytes(inp) -> int:
    """Algorithmic HBM bytes of one decode launch: each live KV latent row once
    (1152 B), the query rows, and the partial outputs + LSEs written."""
    T, H, D = inp["T"], inp["H"], inp["D"]
    return kv_tokens(inp) * KV_ROW_BYTES + T * H * 576 * 2 + D * T * H * (512 + 1) * 4


def combine_bytes(inp, lse_part_host=None) -> int:
    """Algorithmic bytes of one combine: live partials read (skipped empty and
    padding pairs excluded), LSEs read, bf16 outputs + fp32 LSEs written."""
    T, H, D = inp["T"], inp["H"], inp["D"]
    if lse_part_host is not None:
        live = int(np.isfinite(lse_part_host).sum())
    else:
        live = D * T * H
    return live * 512 * 4 + D * T * H * 4 + T * H * (512 * 2 + 4)


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during timing."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.p = None
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(index), "--query-gpu=" + self.Q,
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.p = None

    def stop(self):
        if self.p is None:
            return None
        time.sleep(0.25)
        self.p.terminate()
        try:
            out, _ = self.p.communicate(timeout=5)
        except Exception:
            self.p.kill()
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower() in ("active", "1"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def cpu_oracle_rate(inp, min_seconds: float = 10.0):
    """The float64 oracle as it stands, on the whole workload, repeated until
    about min_seconds of CPU time; returns (tokens/s, passes, seconds)."""
    import oracle
    req, L, pad = oracle.row_lengths(inp["seq_lens"], inp["query_start_loc"], inp["T"])
    passes, t0 = 0, time.perf_counter()
    while True:
        O, lse, rows = oracle.decode_partial(inp)
        oracle.lse_combine(O, lse, pad)
        passes += 1
        el = time.perf_counter() - t0
        if el >= min_seconds or passes >= 50:
            break
    return kv_tokens(inp) * passes / el, passes, el


def cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, device) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_rate(world_size: int, tokens_per_rank: int, max_ms: float) -> float:
    """Whole-job rate of a weak-scaling replica run: every rank processes the
    same workload, and the job takes as long as its slowest rank."""
    return world_size * tokens_per_rank / (max_ms * 1e-3)


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def run_reference(args, spec):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    inp = wl.make_decode_inputs(spec)
    import oracle
    req, L, pad = oracle.row_lengths(inp["seq_lens"], inp["query_start_loc"], inp["T"])

    def step():
        O, lse, _ = oracle.decode_partial(inp)
        oracle.lse_combine(O, lse, pad)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    v = kv_tokens(inp) * args.steps / el
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": spec.name, "B": spec.B, "seq_len": int(inp["max_seq_len"]), "H": spec.H,
                   "D": spec.D, "interleave": spec.interleave, "block_size": spec.block_size},
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores(), "kind": "oracle",
                         "sample": "the whole workload per step (decode partials for all 8 shards "
                                   "+ combine, float64 numpy; BLAS threads = all host cores)"},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_gb300(args, spec):
    import torch
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)
    import mla_decode_context_gb300 as dcp

    inp = wl.make_decode_inputs(spec)
    t = wl.to_torch(inp, dev)
    D, T, H, I = inp["D"], inp["T"], inp["H"], inp["interleave"]
    B = inp["B"]
    msl, mql = max(1, inp["max_seq_len"]), max(1, inp["max_q_len"])
    O = torch.empty((D, T, H, 512), dtype=torch.float32, device=dev)
    lse = torch.empty((D, T, H), dtype=torch.float32, device=dev)
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev)
    out_lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    wsz = dcp.dcp_decode_workspace_size(B, T, H, D, msl, mql)
    work = torch.empty(max(wsz, 16), dtype=torch.uint8, device=dev) if wsz else None
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    derr = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def check_device_flags(where):
        # a kernel that reported a bad input or a timed-out wait did not do
        # the work being timed: stop instead of printing a number
        flags = int(derr.item())
        if flags:
            raise SystemExit(f"bench: device error flags 0x{flags:x} after {where}")

    def decode():
        dcp.dcp_mla_decode_partial(t["q"], t["kv_cache"], t["block_table"], t["seq_lens"],
                                   t["query_start_loc"], O, lse, D=D, interleave=I, scale=inp["scale"],
                                   max_seq_len=msl, max_q_len=mql, workspace=work, dev_error=derr,
                                   stream=stream)

    def combine():
        dcp.dcp_lse_combine(O, lse, t["seq_lens"], t["query_start_loc"], out, out_lse, stream=stream)

    for _ in range(max(3, args.warmup)):
        decode()
        combine()
    torch.cuda.synchronize()
    check_device_flags("warm-up")
    launches_per_step = 1 + dcp.dcp_decode_kernel_launches(B, T, H, D, I, msl, mql, work.numel() if work is not None else 0)

    # ---- device-timed steps (inputs resident, L2 flushed before each) ----
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    clocks = Clocks(dev.index) if rank == 0 else None
    time.sleep(0.3 if clocks else 0)
    wall0 = time.perf_counter()
    for k in range(args.steps):
        flush.zero_()
        ev[k][0].record(stream)
        decode()
        ev[k][1].record(stream)
        combine()
        ev[k][2].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    barrier()
    ck = clocks.stop() if clocks else None
    dec_ms = [ev[k][0].elapsed_time(ev[k][1]) for k in range(args.steps)]
    com_ms = [ev[k][1].elapsed_time(ev[k][2]) for k in range(args.steps)]
    step_ms = sum(a + b for a, b in zip(dec_ms, com_ms)) / args.steps
    step_ms = max_over_ranks(step_ms, dev)
    dec_avg = sum(dec_ms) / len(dec_ms)
    com_avg = sum(com_ms) / len(com_ms)

    # ---- end to end through the C ABI with host buffers ----
    hq = torch.empty_like(t["q"], device="cpu").pin_memory()
    hq.copy_(t["q"].cpu())
    htab = t["block_table"].cpu().pin_memory()
    hseq = t["seq_lens"].cpu().pin_memory()
    hqsl = t["query_start_loc"].cpu().pin_memory()
    hout = torch.empty_like(out, device="cpu").pin_memory()
    hlse = torch.empty_like(out_lse, device="cpu").pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in (hq, htab, hseq, hqsl))
    d2h = hout.numel() * hout.element_size() + hlse.numel() * hlse.element_size()
    e2e_ms = []
    for k in range(args.steps):
        flush.zero_()
        torch.cuda.synchronize()
        w0 = time.perf_counter()
        t["q"].copy_(hq, non_blocking=True)
        t["block_table"].copy_(htab, non_blocking=True)
        t["seq_lens"].copy_(hseq, non_blocking=True)
        t["query_start_loc"].copy_(hqsl, non_blocking=True)
        decode()
        combine()
        hout.copy_(out, non_blocking=True)
        hlse.copy_(out_lse, non_blocking=True)
        torch.cuda.synchronize()
        e2e_ms.append(1e3 * (time.perf_counter() - w0))
    e2e_avg = max_over_ranks(sum(e2e_ms) / len(e2e_ms), dev)
    check_device_flags("the timed steps")

    tokens = kv_tokens(inp)
    peak, peak_kind = peaks()
    dbytes = decode_bytes(inp)
    achieved = dbytes / (dec_avg * 1e-3) / 1e9
    # the bound is the roof the workload meets first: HBM unless its flop
    # per byte exceeds the measured ridge (verification rows, q_len > 1)
    tpeak, tpeak_kind = tensor_peak()
    dflops = decode_flops(inp)
    tflops = dflops / (dec_avg * 1e-3) / 1e12
    tensor_bound = dflops / dbytes > tpeak * 1e12 / (peak * 1e9)
    cbytes = combine_bytes(inp, lse.cpu().numpy())
    res = None
    if rank == 0:
        rate, passes, secs = cpu_oracle_rate(inp)
        res = {
            "metric": METRIC, "value": aggregate_rate(ws, tokens, step_ms), "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": dcp.compute_dtype(), "data": "synthetic",
            "config": {"workload": spec.name, "B": B, "seq_len": int(inp["max_seq_len"]), "H": H, "D": D,
                       "interleave": I, "block_size": inp["block_size"], "q_len": mql,
                       "parallelism": "replicas" if ws > 1 else "single",
                       "l2": "flushed before every step (512 MB write, untimed)"},
            "decode_ms": dec_avg, "combine_ms": com_avg,
            "decode_ms_median": float(np.median(dec_ms)), "combine_ms_median": float(np.median(com_ms)),
            "decode_gbs": achieved, "combine_gbs": cbytes / (com_avg * 1e-3) / 1e9,
            "combine_hbm_frac": cbytes / (com_avg * 1e-3) / 1e9 / peak,
            "roofline": ({"bound": "tensor", "kernel": "dcp_mla_decode_partial", "achieved": tflops,
                          "peak": tpeak, "unit": "TFLOP/s", "frac": tflops / tpeak,
                          "peak_source": tpeak_kind + " (MEASURED_PEAKS.json bf16_tflops, burst)"
                          if tpeak_kind == "measured" else "fallback 1.9 PFLOP/s",
                          "hbm_achieved_gbs": achieved, "hbm_frac": achieved / peak,
                          "traffic": measured_traffic(spec.name),
                          "algorithmic_flops_per_launch": dflops, "algorithmic_bytes_per_launch": dbytes}
                         if tensor_bound else
                         {"bound": "hbm", "kernel": "dcp_mla_decode_partial", "achieved": achieved,
                          "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                          "peak_source": peak_kind + " (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                          else "fallback 6.8 TB/s", "traffic": measured_traffic(spec.name),
                          "tensor_achieved_tflops": tflops, "tensor_frac": tflops / tpeak,
                          "algorithmic_bytes_per_launch": dbytes}),
            "e2e": {"value": aggregate_rate(ws, tokens, e2e_avg), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "note": "host-pinned per-step inputs (q, block table, "
                    "seq_lens, query_start_loc) copied in and out/out_lse copied back inside the timed "
                    "region; the paged KV cache is resident device state"},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": ck,
            "wall_s_timed": wall,
            "cpu_baseline": {"value": rate, "unit": UNIT, "cores": cores(), "kind": "oracle",
                             "sample": "whole workload x %d passes (%.1f s): float64 numpy decode "
                                       "partials + combine" % (passes, secs)},
        }
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if res is not None:
        print(json.dumps(res), flush=True)
    return 0


def run_decode_only(args, spec):
    """For profilers: warmup + steps calls of the decode on one GPU, nothing
    timed or printed but a one-line summary; exits nonzero on a device error."""
    import torch
    import mla_decode_context_gb300 as dcp
    inp = wl.make_decode_inputs(spec)
    t = wl.to_torch(inp, "cuda:0")
    err = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    for _ in range(args.warmup + args.steps):
        dcp.decode_partial(t["q"], t["kv_cache"], t["block_table"], t["seq_lens"], t["query_start_loc"],
                           D=inp["D"], interleave=inp["interleave"], scale=inp["scale"],
                           max_seq_len=inp["max_seq_len"], max_q_len=inp["max_q_len"], dev_error=err)
    torch.cuda.synchronize()
    flags = int(err.item())
    print("%s: %d decode calls, dev_error 0x%x, KV bytes %d"
          % (spec.name, args.warmup + args.steps, flags, kv_tokens(inp) * KV_ROW_BYTES), flush=True)
    return 1 if flags else 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default=wl.LONG_120K.name, choices=sorted(wl.DECODE_WORKLOADS))
    ap.add_argument("--decode-only", action="store_true",
                    help="only call the decode warmup + steps times (for ncu captures)")
    args = ap.parse_args(argv)
    spec = wl.DECODE_WORKLOADS[args.workload]
    if args.decode_only:
        return run_decode_only(args, spec)
    if args.impl == "reference":
        return run_reference(args, spec)
    return run_gb300(args, spec)


if __name__ == "__main__":
    sys.exit(main())
