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
    "sha256": "b201b4f053abdd1da9cc1496dd66c9790436a005f19d792309a54d3321f617e1",
    "bytes": 138486016 + 3622400,
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


def decode_bytes(inp, o_bytes: int = 4) -> int:
    """Algorithmic HBM bytes of one decode launch: each live KV latent row once
    (1152 B in bf16; 576 B of FP8 codes + a 4 B scale in fp8), the query rows,
    and the partial outputs (o_bytes per element) + fp32 LSEs written."""
    T, H, D = inp["T"], inp["H"], inp["D"]
    row = 576 + 4 if inp.get("kv_dtype", "bf16") == "fp8_e4m3" else KV_ROW_BYTES
    return kv_tokens(inp) * row + T * H * 576 * 2 + D * T * H * (512 * o_bytes + 4)


def combine_bytes(inp, lse_part_host=None, o_bytes: int = 4) -> int:
    """Algorithmic bytes of one combine: live partials read (o_bytes per
    element; skipped empty and padding pairs excluded), LSEs read, bf16
    outputs + fp32 LSEs written."""
    T, H, D = inp["T"], inp["H"], inp["D"]
    if lse_part_host is not None:
        live = int(np.isfinite(lse_part_host).sum())
    else:
        live = D * T * H
    return live * 512 * o_bytes + D * T * H * 4 + T * H * (512 * 2 + 4)


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


def workload_config(spec, inp, n_gpus: int) -> dict:
    """The `config` object of a bench line, the same for both arms."""
    cfg = {"workload": spec.name, "B": spec.B, "seq_len": int(inp["max_seq_len"]), "H": spec.H,
           "D": spec.D, "interleave": spec.interleave, "block_size": spec.block_size,
           "q_len": int(inp["max_q_len"]), "parallelism": "replicas" if n_gpus > 1 else "single",
           "l2": "flushed before every timed step (512 MB write, untimed)"}
    if spec.layout != "global":
        cfg["block_tables"] = "per-shard (rank-local)"
    if spec.shared_prefix:
        cfg["shared_prefix"] = spec.prefix_len
    if spec.kv_dtype != "bf16":
        cfg["kv_cache"] = spec.kv_dtype
    return cfg


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
        "data": "synthetic", "config": workload_config(spec, inp, args.gpus),
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores(), "kind": "oracle",
                         "sample": "the whole workload per step (decode partials for all 8 shards "
                                   "+ combine, float64 numpy; BLAS threads = all host cores; host "
                                   "caches are not flushed)"},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def capture(fn, use_graphs: bool):
    """A CUDA graph of `fn` (library calls on the current stream), or None
    when graphs are off or the capture fails (the caller then runs fn
    eagerly).  Graph replay launches the same kernels without the host's
    per-call launch gaps, as a serving loop replays its decode step."""
    import torch
    if not use_graphs:
        return None
    try:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            fn()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="thread_local"):
            fn()
        torch.cuda.synchronize()
        return g
    except Exception as e:  # pragma: no cover - depends on the driver
        print("bench: graph capture failed (%s); timing eager calls" % e, file=sys.stderr)
        torch.cuda.synchronize()
        return None


def packed(tensors, dev):
    """One uint8 device buffer holding copies of `tensors` (each at a
    256-byte-aligned offset) and a view of it shaped like each tensor."""
    import torch
    offs, n = [], 0
    for x in tensors:
        offs.append(n)
        n += (x.numel() * x.element_size() + 255) // 256 * 256
    buf = torch.empty(n, dtype=torch.uint8, device=dev)
    views = []
    for x, o in zip(tensors, offs):
        v = buf[o:o + x.numel() * x.element_size()].view(x.dtype).view(x.shape)
        v.copy_(x)
        views.append(v)
    return buf, views


class DecodeBench:
    """One decode workload resident on the device, with its outputs,
    workspace and the two library calls of a step (decode, combine).  A
    step's own inputs (q, block table, seq_lens, query_start_loc) share one
    device buffer and its outputs (out, out_lse) another, so that an
    end-to-end step moves each with a single copy; the paged KV cache is
    resident state."""

    def __init__(self, spec, dev, use_graphs=True, o_dtype=None):
        import torch
        import mla_decode_context_gb300 as dcp
        o_dtype = torch.float32 if o_dtype is None else o_dtype
        self.spec, self.dev = spec, dev
        self.o_bytes = 2 if o_dtype == torch.bfloat16 else 4
        self.inp = inp = wl.make_decode_inputs(spec)
        self.t = t = wl.to_torch(inp, dev)
        D, T, H, I, B = inp["D"], inp["T"], inp["H"], inp["interleave"], inp["B"]
        self.msl, self.mql = msl, mql = max(1, inp["max_seq_len"]), max(1, inp["max_q_len"])
        self.O = O = torch.empty((D, T, H, 512), dtype=o_dtype, device=dev)
        self.lse = lse = torch.empty((D, T, H), dtype=torch.float32, device=dev)
        self.step_in, views = packed([t["q"], t["block_table"], t["seq_lens"], t["query_start_loc"]], dev)
        t["q"], t["block_table"], t["seq_lens"], t["query_start_loc"] = views
        self.step_out, (out, out_lse) = packed([torch.zeros((T, H, 512), dtype=torch.bfloat16),
                                                torch.zeros((T, H), dtype=torch.float32)], dev)
        self.out, self.out_lse = out, out_lse
        wsz = dcp.dcp_decode_workspace_size(B, T, H, D, msl, mql)
        self.work = work = torch.empty(max(wsz, 16), dtype=torch.uint8, device=dev) if wsz else None
        self.derr = derr = torch.zeros(1, dtype=torch.int32, device=dev)
        self.launches = 1 + dcp.dcp_decode_kernel_launches(B, T, H, D, I, msl, mql,
                                                           work.numel() if work is not None else 0)

        general = spec.kv_dtype != "bf16" or spec.layout != "global" or o_dtype != torch.float32

        def decode():
            if general:  # fp8 cache, per-shard tables or bf16 partials
                dcp.dcp_mla_decode_partial_v2(t["q"], t["kv_cache"], t["block_table"], t["seq_lens"],
                                              t["query_start_loc"], O, lse, D=D, interleave=I, scale=inp["scale"],
                                              max_seq_len=msl, max_q_len=mql, kv_scale=t.get("kv_scale"),
                                              workspace=work, dev_error=derr)
            else:
                dcp.dcp_mla_decode_partial(t["q"], t["kv_cache"], t["block_table"], t["seq_lens"],
                                           t["query_start_loc"], O, lse, D=D, interleave=I, scale=inp["scale"],
                                           max_seq_len=msl, max_q_len=mql, workspace=work, dev_error=derr)

        def combine():
            dcp.dcp_lse_combine(O, lse, t["seq_lens"], t["query_start_loc"], out, out_lse)

        self.decode, self.combine = decode, combine
        for _ in range(3):
            decode()
            combine()
        torch.cuda.synchronize()
        self.check_flags("warm-up")
        self.g_dec = capture(decode, use_graphs)
        self.g_com = capture(combine, use_graphs)
        self.graphs = self.g_dec is not None and self.g_com is not None

        def step():
            decode()
            combine()

        # the whole step as one graph (the combine's launch then overlaps the
        # split merge's tail through programmatic dependent launch)
        self.g_step = capture(step, use_graphs and self.graphs)

    def check_flags(self, where):
        # a kernel that reported a bad input or a timed-out wait did not do
        # the work being timed: stop instead of printing a number
        flags = int(self.derr.item())
        if flags:
            raise SystemExit(f"bench: device error flags 0x{flags:x} after {where} ({self.spec.name})")

    def run_decode(self):
        self.g_dec.replay() if self.graphs else self.decode()

    def run_combine(self):
        self.g_com.replay() if self.graphs else self.combine()

    def timed(self, steps, warmup, flush):
        """Per-step (decode ms, combine ms), CUDA events on the launching
        stream, the L2 flushed (untimed) before every step."""
        import torch
        stream = torch.cuda.current_stream(self.dev)
        for _ in range(warmup):
            flush.zero_()
            self.run_decode()
            self.run_combine()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
        torch.cuda.synchronize()
        for k in range(steps):
            flush.zero_()
            ev[k][0].record(stream)
            self.run_decode()
            ev[k][1].record(stream)
            self.run_combine()
            ev[k][2].record(stream)
        torch.cuda.synchronize()
        self.check_flags("the timed steps")
        dec = [ev[k][0].elapsed_time(ev[k][1]) for k in range(steps)]
        com = [ev[k][1].elapsed_time(ev[k][2]) for k in range(steps)]
        return dec, com

    def timed_step(self, steps, warmup, flush):
        """Per-step ms of the whole step replayed as one graph (None without
        graphs), CUDA events on the launching stream, the L2 flushed (untimed)
        before every step."""
        import torch
        if self.g_step is None:
            return None
        stream = torch.cuda.current_stream(self.dev)
        for _ in range(warmup):
            flush.zero_()
            self.g_step.replay()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
        torch.cuda.synchronize()
        for k in range(steps):
            flush.zero_()
            ev[k][0].record(stream)
            self.g_step.replay()
            ev[k][1].record(stream)
        torch.cuda.synchronize()
        self.check_flags("the timed steps")
        return [ev[k][0].elapsed_time(ev[k][1]) for k in range(steps)]

    def roofline(self, dec_ms: float, traffic=None) -> dict:
        """The decode call's roofline record: HBM unless the workload's flop
        per byte pass the measured ridge (verification rows)."""
        inp = self.inp
        peak, peak_kind = peaks()
        tpeak, tpeak_kind = tensor_peak()
        dbytes = decode_bytes(inp, self.o_bytes)
        dflops = decode_flops(inp)
        achieved = dbytes / (dec_ms * 1e-3) / 1e9
        tflops = dflops / (dec_ms * 1e-3) / 1e12
        if dflops / dbytes > tpeak * 1e12 / (peak * 1e9):
            return {"bound": "tensor", "kernel": "dcp_mla_decode_partial", "achieved": tflops, "peak": tpeak,
                    "unit": "TFLOP/s", "frac": tflops / tpeak,
                    "peak_source": tpeak_kind + " (MEASURED_PEAKS.json bf16_tflops, burst)"
                    if tpeak_kind == "measured" else "fallback 1.9 PFLOP/s",
                    "hbm_achieved_gbs": achieved, "hbm_frac": achieved / peak, "traffic": traffic,
                    "algorithmic_flops_per_launch": dflops, "algorithmic_bytes_per_launch": dbytes}
        return {"bound": "hbm", "kernel": "dcp_mla_decode_partial", "achieved": achieved, "peak": peak,
                "unit": "GB/s", "frac": achieved / peak,
                "peak_source": peak_kind + " (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                else "fallback 6.8 TB/s", "traffic": traffic,
                "tensor_achieved_tflops": tflops, "tensor_frac": tflops / tpeak,
                "algorithmic_bytes_per_launch": dbytes}

    def release(self):
        import torch
        for k in list(vars(self)):
            setattr(self, k, None)
        torch.cuda.empty_cache()


def combine_sweep_record(dev, flush, steps: int = 20):
    """The standalone combine over the sweep (D in {2, 4, 8}, T in {1, 64,
    1024, 4096}, H = 128): median µs per call and GB/s of algorithmic bytes
    (live partials + all LSEs read, bf16 out + fp32 out_lse written); the HBM
    fraction is reported where the pages' bandwidth target applies (T >=
    1024; smaller T are latency-bound)."""
    import torch
    import mla_decode_context_gb300 as dcp
    peak, _ = peaks()
    rec = {}
    for D, T in wl.COMBINE_SWEEP:
        O, lse, seq, qsl, empty, pad = wl.make_combine_inputs(D, T, device=dev)
        seq_t, qsl_t = torch.from_numpy(seq).to(dev), torch.from_numpy(qsl).to(dev)
        out = torch.empty((T, wl.COMBINE_H, 512), dtype=torch.bfloat16, device=dev)
        out_lse = torch.empty((T, wl.COMBINE_H), dtype=torch.float32, device=dev)

        def call():
            dcp.dcp_lse_combine(O, lse, seq_t, qsl_t, out, out_lse)

        g = capture(call, True)
        run = g.replay if g is not None else call
        for _ in range(3):
            run()
        stream = torch.cuda.current_stream(dev)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
        torch.cuda.synchronize()
        for k in range(steps):
            flush.zero_()
            ev[k][0].record(stream)
            run()
            ev[k][1].record(stream)
        torch.cuda.synchronize()
        us = statistics.median(ev[k][0].elapsed_time(ev[k][1]) * 1e3 for k in range(steps))
        live = (~empty & ~pad[None, :]).sum() * wl.COMBINE_H
        nbytes = int(live) * 512 * 4 + D * T * wl.COMBINE_H * 4 + T * wl.COMBINE_H * (512 * 2 + 4)
        gbs = nbytes / (us * 1e-6) / 1e9
        r = {"us": us, "gbs": gbs, "algorithmic_bytes": nbytes}
        if T >= 1024:
            r["hbm_frac"] = gbs / peak
        rec["D%d_T%d" % (D, T)] = r
        del O, lse, out, out_lse, g
        torch.cuda.empty_cache()
    return rec


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

    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    bench = DecodeBench(spec, dev, use_graphs=not args.eager)
    inp, t = bench.inp, bench.t

    # ---- device-timed steps (inputs resident, L2 flushed before each) ----
    barrier()
    torch.cuda.synchronize()
    clocks = Clocks(dev.index) if rank == 0 else None
    time.sleep(0.3 if clocks else 0)
    wall0 = time.perf_counter()
    dec_ms, com_ms = bench.timed(args.steps, max(3, args.warmup), flush)
    whole = bench.timed_step(args.steps, max(3, args.warmup), flush)
    wall = time.perf_counter() - wall0
    barrier()
    ck = clocks.stop() if clocks else None
    # a step: the whole hot path, one graph replay (else decode + combine
    # timed back to back)
    step_ms = (sum(whole) if whole is not None else sum(a + b for a, b in zip(dec_ms, com_ms))) / args.steps
    step_ms = max_over_ranks(step_ms, dev)
    dec_avg = sum(dec_ms) / len(dec_ms)
    com_avg = sum(com_ms) / len(com_ms)

    # ---- end to end through the C ABI with host buffers ----
    # the step's inputs (q, block table, seq_lens, query_start_loc) in one
    # pinned host buffer laid out like the device one: one copy in; out and
    # out_lse back with one copy
    hin = bench.step_in.cpu().pin_memory()
    hout = torch.empty_like(bench.step_out, device="cpu").pin_memory()
    h2d = hin.numel()
    d2h = hout.numel()
    def e2e_step():
        bench.step_in.copy_(hin, non_blocking=True)
        bench.decode()
        bench.combine()
        hout.copy_(bench.step_out, non_blocking=True)

    def e2e_times(run):
        ms = []
        for k in range(args.steps):
            flush.zero_()
            torch.cuda.synchronize()
            w0 = time.perf_counter()
            run()
            torch.cuda.synchronize()
            ms.append(1e3 * (time.perf_counter() - w0))
        return max_over_ranks(sum(ms) / len(ms), dev)

    # eager: the copies and the two library calls issued from Python every
    # step; graph: the same step captured once as a CUDA graph (copies,
    # dcp_mla_decode_partial, dcp_lse_combine, copies back) and replayed, as
    # a serving loop runs its decode step
    e2e_eager = e2e_times(e2e_step)
    g_e2e = capture(e2e_step, not args.eager)
    e2e_graph = e2e_times(g_e2e.replay) if g_e2e is not None else None
    e2e_avg = e2e_graph if e2e_graph is not None else e2e_eager
    bench.check_flags("the end-to-end steps")

    tokens = kv_tokens(inp)
    peak, _ = peaks()
    cbytes = combine_bytes(inp, bench.lse.cpu().numpy())
    roof = bench.roofline(dec_avg, measured_traffic(spec.name))
    res = None
    if rank == 0:
        res = {
            "metric": METRIC, "value": aggregate_rate(ws, tokens, step_ms), "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": dcp.compute_dtype(), "data": "synthetic",
            "config": workload_config(spec, inp, ws),
            "timing": ("one CUDA graph of the step's two library calls, replayed (decode_ms / combine_ms: "
                       "each call's own graph)" if whole is not None else
                       "CUDA graphs of the library calls, replayed" if bench.graphs else "eager library calls"),
            "decode_ms": dec_avg, "combine_ms": com_avg,
            "decode_ms_median": float(np.median(dec_ms)), "combine_ms_median": float(np.median(com_ms)),
            "decode_gbs": decode_bytes(inp) / (dec_avg * 1e-3) / 1e9,
            "combine_gbs": cbytes / (com_avg * 1e-3) / 1e9,
            "combine_hbm_frac": cbytes / (com_avg * 1e-3) / 1e9 / peak,
            "roofline": roof,
            "e2e": {"value": aggregate_rate(ws, tokens, e2e_avg), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h,
                    "timing": ("wall clock around one CUDA-graph replay per step (host->device copies, "
                               "dcp_mla_decode_partial, dcp_lse_combine, device->host copies) and a "
                               "synchronize" if e2e_graph is not None else
                               "wall clock around eager library calls per step and a synchronize"),
                    "eager_value": aggregate_rate(ws, tokens, e2e_eager),
                    "note": "host-pinned per-step inputs (q, block table, seq_lens, query_start_loc, packed "
                    "in one buffer) copied in with one copy and out/out_lse copied back with one copy inside "
                    "the timed region; the paged KV cache is resident device state"},
            "gpu_launches": bench.launches * args.steps,
            "clocks": ck,
            "wall_s_timed": wall,
        }
    bench.release()

    # ---- the other workloads: decode records and the combine sweep ----
    if rank == 0 and not args.headline_only:
        recs = {}
        for other in (wl.BATCHED_B64, wl.SPEC_VERIFY_B32, wl.LONG_120K_B2_PREFIX, wl.LONG_120K_B2_PREFIX_LOCAL,
                      wl.BATCHED_B64_LOCAL):
            ob = DecodeBench(other, dev, use_graphs=not args.eager)
            osteps = max(5, min(args.steps, 20))
            d_ms, c_ms = ob.timed(osteps, 3, flush)
            dmed = float(np.median(d_ms))
            recs[other.name] = {
                "config": workload_config(other, ob.inp, 1), "steps": osteps,
                "decode_ms_median": dmed, "combine_ms_median": float(np.median(c_ms)),
                "kv_tokens_per_s": kv_tokens(ob.inp) / ((dmed + float(np.median(c_ms))) * 1e-3),
                "roofline": ob.roofline(dmed), "gpu_launches_per_step": ob.launches}
            ob.release()
        for name, other, od in (("long_ctx_120k_b1_d8_i1 bf16 partials", wl.LONG_120K, torch.bfloat16),
                                ("long_ctx_120k_b1_d8_i1 fp8 cache", wl.LONG_120K_FP8, None)):
            ob = DecodeBench(other, dev, use_graphs=not args.eager, o_dtype=od)
            d_ms, c_ms = ob.timed(max(5, min(args.steps, 20)), 3, flush)
            dmed = float(np.median(d_ms))
            cfg = workload_config(other, ob.inp, 1)
            cfg["partials"] = "bf16" if od is not None else "fp32"
            recs[name] = {
                "config": cfg, "decode_ms_median": dmed, "combine_ms_median": float(np.median(c_ms)),
                "kv_tokens_per_s": kv_tokens(ob.inp) / ((dmed + float(np.median(c_ms))) * 1e-3),
                "roofline": ob.roofline(dmed), "gpu_launches_per_step": ob.launches,
                "kernel": "tensor cores"}
            ob.release()
        recs["combine_sweep_h128"] = combine_sweep_record(dev, flush)
        res["workloads"] = recs
    if rank == 0:
        rate, passes, secs = cpu_oracle_rate(inp)
        res["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": cores(), "kind": "oracle",
                               "sample": "whole workload x %d passes (%.1f s): float64 numpy decode "
                                         "partials + combine" % (passes, secs)}
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
                           max_seq_len=inp["max_seq_len"], max_q_len=inp["max_q_len"], dev_error=err,
                           kv_scale=t.get("kv_scale"))
    torch.cuda.synchronize()
    flags = int(err.item())
    row_bytes = 576 + 4 if inp.get("kv_dtype", "bf16") == "fp8_e4m3" else KV_ROW_BYTES
    print("%s: %d decode calls, dev_error 0x%x, KV bytes %d"
          % (spec.name, args.warmup + args.steps, flags, kv_tokens(inp) * row_bytes), flush=True)
    return 1 if flags else 0


def run_combine_only(args):
    """For profilers: warmup + steps calls of the standalone combine on one
    combine-sweep point (D, T), nothing timed; exits nonzero on failure."""
    import torch
    import mla_decode_context_gb300 as dcp
    D, T = args.combine_only
    O, lse, seq, qsl, empty, pad = wl.make_combine_inputs(D, T, device="cuda:0")
    seq_t, qsl_t = torch.from_numpy(seq).cuda(), torch.from_numpy(qsl).cuda()
    for _ in range(args.warmup + args.steps):
        out, out_lse = dcp.lse_combine(O, lse, seq_t, qsl_t)
    torch.cuda.synchronize()
    ok = not torch.isnan(out).any().item()
    print("combine D=%d T=%d: %d calls, finite=%s" % (D, T, args.warmup + args.steps, ok), flush=True)
    return 0 if ok else 1


def run_probe(name: str) -> int:
    """The measurements behind the kernels' design choices: each probe is a
    small CUDA program (bounded waits, one CTA per SM) that prints its own
    table."""
    from mla_decode_context_gb300 import build_lib
    exe = build_lib.build_probe(name)
    return subprocess.run([exe], check=False).returncode


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default=wl.LONG_120K.name, choices=sorted(wl.DECODE_WORKLOADS))
    ap.add_argument("--decode-only", action="store_true",
                    help="only call the decode warmup + steps times (for ncu captures)")
    ap.add_argument("--eager", action="store_true", help="time eager library calls instead of graph replays")
    ap.add_argument("--combine-only", type=int, nargs=2, metavar=("D", "T"),
                    help="only call the standalone combine on one sweep point (for ncu captures)")
    ap.add_argument("--headline-only", action="store_true",
                    help="skip the other workloads and the combine sweep")
    ap.add_argument("--probe", choices=["mma_rate", "load_rate", "tma_rate", "store_rate"],
                    help="build and run one stand-alone hardware-rate probe (tensor-core issue rate, "
                         "cp.async streaming rate, TMA streaming rate, store rate) instead of the bench")
    args = ap.parse_args(argv)
    if args.probe:
        return run_probe(args.probe)
    spec = wl.DECODE_WORKLOADS[args.workload]
    if args.combine_only:
        return run_combine_only(args)
    if args.decode_only:
        return run_decode_only(args, spec)
    if args.impl == "reference":
        return run_reference(args, spec)
    return run_gb300(args, spec)


if __name__ == "__main__":
    sys.exit(main())
