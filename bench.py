#!/usr/bin/env python
"""Benchmark of the GB300 Flash-Overlap hot path; prints ONE JSON line.

Default workload: the largest single-GPU configuration, the 70B-like MLP layer at
16K tokens with P=8 virtual ranks on one GPU (tokens 16384 sharded by sequence,
hidden 8192, ffn 28672): Flash-AG (gate/up, column-parallel) -> SiLU(gate)*up ->
Flash-RS (down, row-parallel).  A step is one layer over one batch; inputs stay
resident in HBM.  The timed weights (1.4 GB) and activations exceed the 126 MiB
L2, so no flush is used.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload llama8b|tiny|sweep1k..sweep16k|tail_rs|attn|attn1k..attn16k|attn_layer|a2a|mlp_bwd]

With N > 1 (torchrun, one process per GPU) every rank runs an independent
replica of the workload ("replicas only": the virtual ranks of one layer never
span GPUs); value = total FLOP of all ranks / max-over-ranks time.
``--impl reference`` times the CPU oracle (the slow plain restatement under
oracle/) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import fo_workloads as wl  # noqa: E402

METRIC = "overlapped AG-GEMM/GEMM-RS TFLOP/s, % of bf16 tensor peak; exposed copy time"
# sources whose digest a committed ncu summary records (traffic is reported only while they match)
# the kernel and the host code that orders its tiles (fo_api.cu): both set its DRAM traffic
PAIR_KERNEL_SOURCES = ("overlapped_tensor_gemm_gb300/csrc/fo_gemm2.cu",
                       "overlapped_tensor_gemm_gb300/csrc/fo_gemm_common.cuh",
                       "overlapped_tensor_gemm_gb300/csrc/fo_ptx.cuh",
                       "overlapped_tensor_gemm_gb300/csrc/fo_api.cu")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="sweep16k")
    ap.add_argument("--no-extras", action="store_true", help="skip baselines, attention, e2e and the CPU leg")
    ap.add_argument("--no-attn", action="store_true", help="skip the attention sub-benchmark")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle leg")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="target CPU time of the oracle sample")
    ap.add_argument("--attn-order", default="flash", choices=["flash", "serial"],
                    help="order of the attention workload's main timing ('serial' for ncu, as --ag-order)")
    ap.add_argument("--ag-order", default="flash", choices=["flash", "serial"],
                    help="order of the AG projection; 'serial' (ring first, same GEMM kernel after) is what "
                         "runs under ncu, which serialises the ring copies against kernels")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"bf16_burst": d["bf16_tflops"], "bf16_sustained": d["bf16_tflops_sustained"],
                "hbm_gbs": d["hbm_gbs"], "source": "measured"}
    return {"bf16_burst": 1900.0, "bf16_sustained": 1700.0, "hbm_gbs": 6800.0, "source": "fallback"}


def source_digest(sources) -> str:
    import hashlib
    h = hashlib.sha256()
    for src in sources:
        with open(os.path.join(ROOT, src), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profiled_traffic(profile: str, sources):
    """DRAM bytes per launch from a committed ncu summary, if the kernel sources are unchanged."""
    import re
    try:
        text = open(os.path.join(ROOT, "profiles", profile)).read()
        want = re.search(r"sha256 prefix `([0-9a-f]+)`", text).group(1)
        have = source_digest(sources)[:len(want)]
        if have != want:
            return None
        return int(re.search(r"traffic_bytes_per_launch: (\d+)", text).group(1))
    except (OSError, AttributeError):
        return None


def aggregate(flop_per_rank: float, ms_per_rank: float, world: int, reduce_max) -> tuple[float, float]:
    """Whole-job throughput of `world` independent replicas: all ranks' FLOP over the
    slowest rank's time.  Returns (TFLOP/s, max ms)."""
    ms_max = reduce_max(ms_per_rank)
    return world * flop_per_rank / (ms_max * 1e-3) / 1e12, ms_max


def layer_in_one_launch(cfg) -> bool:
    """fo_mlp_layer runs the whole layer in one launch unless its reduce-scatter takes the
    transposed tiles of its own launch (rank slices of 32, 64 or 128 rows with 256/m
    dividing P; include/fo.h, fo_opts.split_layer)."""
    m = cfg.m
    transposed = m <= 128 and m % 32 == 0 and 256 % m == 0 and 256 // m <= cfg.P and cfg.P % (256 // m) == 0
    return not transposed


def mlp_config(name: str):
    if name == "llama8b":
        return wl.LLAMA8B
    if name == "tiny":
        return wl.TINY
    if name.startswith("sweep"):
        return wl.sweep(int(name[5:-1]) * 1024)
    raise SystemExit(f"unknown MLP workload {name}")


# --------------------------------------------------------------------------
# clocks sampler (nvidia-smi during the timed region)
# --------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.tmp = None

    def __enter__(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.tmp, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self) -> dict:
        if self.proc is None or self.tmp is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        self.tmp.flush()
        with open(self.tmp.name) as f:
            rows = [r.strip().split(",") for r in f if r.strip()]
        os.unlink(self.tmp.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for i, n in enumerate(names):
                if len(r) > 5 + i and "Active" in r[5 + i] and "Not" not in r[5 + i]:
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# --------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline and --impl reference)
# --------------------------------------------------------------------------

def oracle_mlp_sample(cfg, inp_f64, rows_per_slice: int, seed: int):
    """Runs the oracle's decomposed MLP layer on a row sample; returns (seconds, flop)."""
    from oracle import ops
    rng = np.random.default_rng(seed)
    rows = [np.sort(rng.choice(cfg.m, size=rows_per_slice, replace=False)) for _ in range(cfg.P)]
    X, Wc, Wr = inp_f64
    t0 = time.perf_counter()
    ops.mlp_layer([X[s][rows[s]] for s in range(cfg.P)], Wc, Wr, gated=cfg.gated)
    dt = time.perf_counter() - t0
    n = rows_per_slice * cfg.P
    flop = 2 * n * cfg.hidden * cfg.n_col * cfg.P + 2 * n * cfg.k_row * cfg.hidden * cfg.P
    return dt, flop


def decode_inputs(inp):
    from oracle import bf16
    return ([bf16.to_f64(x) for x in inp["X_shards"]], [bf16.to_f64(w) for w in inp["W_col"]],
            [bf16.to_f64(w) for w in inp["W_row"]])


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def calibrate_rows(cfg, inp_f64, target_s: float) -> int:
    """Token rows per slice for an oracle sample of about target_s seconds.  A small sample's
    time is mostly the fixed cost of streaming the fp64 weights, so the sample is grown until
    one run takes at least half the target and then scaled in proportion (which, with a fixed
    part in the cost, can only fall short of the target, never overshoot it)."""
    r = 2
    dt, _ = oracle_mlp_sample(cfg, inp_f64, r, 0)
    while dt < 0.5 * target_s and r < cfg.m:
        r = int(min(cfg.m, max(2 * r, r * 0.6 * target_s / max(dt, 1e-3))))
        dt, _ = oracle_mlp_sample(cfg, inp_f64, r, 0)
    return int(max(2, min(cfg.m, r * target_s / max(dt, 1e-3))))


# --------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------

def run_ours(args, rank: int, world: int, device: int):
    import torch
    import overlapped_tensor_gemm_gb300 as fo
    torch.cuda.set_device(device)
    dist = None
    if world > 1:
        import torch.distributed as dist

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    def max_over_ranks(x: float) -> float:
        if dist is None:
            return x
        t = torch.tensor([x], device="cuda", dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    pk = peaks()
    if args.workload == "attn" or (args.workload.startswith("attn") and args.workload.endswith("k")):
        return run_attention_only(args, rank, world, device, pk, barrier, max_over_ranks)
    if args.workload == "tail_rs":
        return run_tail_rs(args, world, device, pk)
    if args.workload == "attn_layer":
        return run_attn_layer(args, world, device, pk)
    if args.workload == "a2a":
        return run_a2a(args, world, device, pk)
    if args.workload == "mlp_bwd":
        return run_mlp_backward(args, world, device, pk)
    cfg = mlp_config(args.workload)
    inp = wl.mlp_inputs(cfg)

    def dev(bits):
        return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).cuda()

    X = [dev(x) for x in inp["X_shards"]]
    Wc = [dev(w) for w in inp["W_col"]]
    Wr = [dev(w) for w in inp["W_row"]]
    Z = [torch.empty((cfg.m, cfg.hidden), dtype=torch.bfloat16, device="cuda") for _ in range(cfg.P)]
    ctx = fo.Context(device)
    stream = torch.cuda.current_stream()
    flops = cfg.flops()

    M = cfg.tokens
    epi = "silu" if cfg.gated else "plain"
    H = [torch.empty((M, cfg.k_row if cfg.gated else cfg.n_col), dtype=torch.bfloat16, device="cuda")
         for _ in range(cfg.P)]

    def layer():
        if args.ag_order == "flash":
            ctx.mlp_layer(X, Wc, Wr, Z, gated=cfg.gated)
        else:
            ctx.ag_gemm(X, Wc, H, order=args.ag_order, epilogue=epi)
            ctx.gemm_rs(H, Wr, Z)

    for _ in range(max(args.warmup, 3)):
        layer()
    torch.cuda.synchronize()
    ctx.poll()

    # ---- main timed region: K layers back to back -------------------------
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(device) as clk:
        e0.record(stream)
        for _ in range(args.steps):
            layer()
        e1.record(stream)
        torch.cuda.synchronize()
    barrier()
    ctx.poll()
    ms = e0.elapsed_time(e1) / args.steps
    value, ms_max = aggregate(flops["total"], ms, world, max_over_ranks)
    one_launch = layer_in_one_launch(cfg) and args.ag_order == "flash"
    launches_per_step = 1 if one_launch else 2  # the whole layer, or Flash-AG + Flash-RS

    out = {"metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max, 4),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
           "data": "synthetic (seeded N(0,1) activations, N(0,0.02) weights, bf16)",
           "config": {"workload": f"{cfg.name}: MLP layer, P={cfg.P} virtual ranks on one GPU, tokens "
                                  f"{cfg.tokens}, hidden {cfg.hidden}, ffn {cfg.ffn}",
                      "P": cfg.P, "tokens": cfg.tokens, "hidden": cfg.hidden, "ffn": cfg.ffn,
                      "global_batch": cfg.tokens, "seq_len": cfg.tokens,
                      "parallelism": f"virtual tp{cfg.P} on one GPU; replicas across GPUs",
                      "l2": "inputs larger than L2 (no flush)"},
           "pct_of_peak": round(100 * value / world / pk["bf16_burst"], 2),
           "gpu_launches": launches_per_step * args.steps,
           "clocks": clk.summary()}

    # ---- per-op timing: roofline of the dominant kernel, baselines, exposure ----
    def timed(fn, iters):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(iters):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        ctx.poll()
        return a.elapsed_time(b) / iters

    def timed_set(fns: dict, iters: int, rounds: int = 5) -> dict:
        """Median ms per call of every function of `fns`, timed in `rounds` interleaved
        rounds of `iters` back-to-back calls (CUDA events on the launching stream): at the
        long sweep points the GPU runs into its power cap, and interleaving gives every
        variant the same mix of clock states."""
        for fn in fns.values():
            fn()
            fn()
        torch.cuda.synchronize()
        samples = {k: [] for k in fns}
        for _ in range(rounds):
            for k, fn in fns.items():
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                for _ in range(iters):
                    fn()
                b.record(stream)
                torch.cuda.synchronize()
                samples[k].append(a.elapsed_time(b) / iters)
        ctx.poll()
        return {k: statistics.median(v) for k, v in samples.items()}

    iters = max(2, min(args.steps, int(40.0 / max(ms_max, 1e-3))))  # ~40 ms of work per sample
    # every variant, and the same variant with its transfers removed (compute_only: the
    # same launches, every ring flag published before the launch, no copy enqueued)
    ag = lambda o, c=False: (lambda: ctx.ag_gemm(X, Wc, H, order=o, epilogue=epi, compute_only=c))  # noqa: E731
    rs = lambda o, c=False: (lambda: ctx.gemm_rs(H, Wr, Z, order=o, compute_only=c))  # noqa: E731
    variants = [("ag", ag, ("flash", "serial", "slicing")), ("rs", rs, ("flash", "naive", "serial", "slicing"))]
    if args.no_extras:
        variants = [("ag", ag, ("flash",)), ("rs", rs, ("flash",))]
    fns = {("layer", "one", False): lambda: ctx.mlp_layer(X, Wc, Wr, Z, gated=cfg.gated),
           ("layer", "two", False): lambda: ctx.mlp_layer(X, Wc, Wr, Z, gated=cfg.gated, split_layer=True)}
    for op, fn, orders in variants:
        for o in orders:
            fns[(op, o, False)] = fn(o if not (op == "ag" and o == "flash") else args.ag_order)
            if not args.no_extras:
                fns[(op, o, True)] = fn(o, True)
    tm = timed_set(fns, iters)
    t_ag, t_rs = tm[("ag", "flash", False)], tm[("rs", "flash", False)]
    t_one, t_two = tm[("layer", "one", False)], tm[("layer", "two", False)]
    ag_tflops = flops["ag"] / (t_ag * 1e-3) / 1e12
    # 256-row tiles on SM pairs when every slice is a multiple of 256 rows, or (all-gather) when
    # 128-row slices pair up two ring steps per tile (P even)
    pair = cfg.m % 256 == 0 or (cfg.m == 128 and cfg.P % 2 == 0 and not one_launch)
    kernel = "gemm_pair_kernel" if pair else "gemm_kernel"
    if one_launch:  # the step is one launch: the whole layer's FLOP over its duration
        dom = {"kernel": f"{kernel} (whole MLP layer in one launch: Flash-AG with the {epi} epilogue, "
                         f"then Flash-RS)", "achieved": flops["total"] / (t_one * 1e-3) / 1e12,
               "flop_per_launch": flops["total"], "ms_per_launch": t_one,
               "profile": f"{kernel}_{cfg.name}_layer.md"}
    else:
        dom = {"kernel": f"{kernel} (Flash-AG launch, {epi} epilogue)", "achieved": ag_tflops,
               "flop_per_launch": flops["ag"], "ms_per_launch": t_ag, "profile": f"{kernel}_{cfg.name}_mlp.md"}
    out["roofline"] = {"bound": "tensor", "kernel": dom["kernel"], "achieved": round(dom["achieved"], 2),
                       "peak": pk["bf16_burst"], "unit": "TFLOP/s", "frac": round(dom["achieved"] / pk["bf16_burst"], 4),
                       "peak_kind": f"bf16 burst ({pk['source']})",
                       "frac_of_sustained_peak": round(dom["achieved"] / pk["bf16_sustained"], 4),
                       "flop_per_launch": dom["flop_per_launch"], "ms_per_launch": round(dom["ms_per_launch"], 4),
                       "traffic": profiled_traffic(dom["profile"], PAIR_KERNEL_SOURCES),
                       "traffic_unit": "bytes per launch (dram read + write, ncu)"}
    breakdown = {"layer_one_launch_ms": round(t_one, 4), "layer_two_launches_ms": round(t_two, 4),
                 "ag_flash_ms": round(t_ag, 4), "rs_flash_ms": round(t_rs, 4),
                 "ag_tflops": round(ag_tflops, 2), "rs_tflops": round(flops["rs"] / (t_rs * 1e-3) / 1e12, 2)}
    if not args.no_extras:
        def phase(fn):
            fn()
            torch.cuda.synchronize()
            return ctx.phase_ms()
        t = {(op, o): v for (op, o, c), v in tm.items() if not c}
        tc = {(op, o): v for (op, o, c), v in tm.items() if c}
        ag_coll, ag_gemm = phase(ag("serial"))
        rs_coll, rs_gemm = phase(rs("serial"))
        exposed = {o: (t[("ag", "flash" if o == "naive" else o)] - tc[("ag", "flash" if o == "naive" else o)])
                   + (t[("rs", o)] - tc[("rs", o)]) for o in ("flash", "naive", "serial", "slicing")}
        breakdown.update({
            "ag_serial_ms": round(t[("ag", "serial")], 4), "ag_slicing_ms": round(t[("ag", "slicing")], 4),
            "ag_serial_phases_ms": {"ring": round(ag_coll, 4), "gemm": round(ag_gemm, 4)},
            "rs_serial_ms": round(t[("rs", "serial")], 4), "rs_slicing_ms": round(t[("rs", "slicing")], 4),
            "rs_naive_ms": round(t[("rs", "naive")], 4),
            "rs_serial_phases_ms": {"gemm": round(rs_gemm, 4), "ring_reduce": round(rs_coll, 4)},
            "compute_only_ms": {f"{op}_{o}": round(v, 4) for (op, o), v in tc.items()},
            "timing": f"medians of 5 interleaved rounds of {iters} calls per variant",
        })
        ser = exposed["serial"]
        out["exposed_copy"] = {
            "flash_ms": round(exposed["flash"], 4), "flash_frac_of_layer": round(exposed["flash"] / (t_ag + t_rs), 4),
            "serial_ms": round(ser, 4), "slicing_ms": round(exposed["slicing"], 4),
            "naive_rs_ms": round(exposed["naive"], 4),
            "hidden_frac_vs_serial": round(1 - exposed["flash"] / ser, 4) if ser > 0 else None,
            "slicing_hidden_frac_vs_serial": round(1 - exposed["slicing"] / ser, 4) if ser > 0 else None,
            "definition": "per projection T_variant - T_compute_only(variant): the same launches of that variant "
                          "with every ring flag published before the launch and no copy enqueued; summed over "
                          "the AG and RS projections (naive: Flash-AG + naive-order RS)",
            "pages_context": "about 99.8% of communication overhead hidden vs about 84% for data slicing "
                             "(FlashOverlap summary, section 4; hardware not named)"}
        # ---- end to end through the public API with host buffers -------------
        Xh = [torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).pin_memory()
              for x in inp["X_shards"]]
        Zh = [torch.empty((cfg.m, cfg.hidden), dtype=torch.bfloat16).pin_memory() for _ in range(cfg.P)]
        t_e2e = timed(lambda: ctx.mlp_layer_host(Xh, Wc, Wr, Zh, gated=cfg.gated), args.steps)
        t_e2e = max_over_ranks(t_e2e)
        nbytes = sum(x.numel() * 2 for x in Xh)
        out["e2e"] = {"value": round(world * flops["total"] / (t_e2e * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                      "ms_per_step": round(t_e2e, 4), "h2d_bytes_per_step": nbytes,
                      "d2h_bytes_per_step": sum(z.numel() * 2 for z in Zh)}
        # ---- query-split attention (config 5) -------------------------------
        if not args.no_attn:
            out["attention"] = attention_bench(ctx, pk, max(3, args.steps // 4))
    out["breakdown"] = breakdown
    ctx.close()

    if rank == 0 and not args.no_extras and not args.no_cpu:
        inp_f64 = decode_inputs(inp)
        rows = calibrate_rows(cfg, inp_f64, args.cpu_seconds)
        dt, fl = oracle_mlp_sample(cfg, inp_f64, rows, 1)
        out["cpu_baseline"] = {"value": round(fl / dt / 1e12, 6), "unit": "TFLOP/s", "cores": cpu_cores(),
                               "kind": "oracle", "seconds": round(dt, 2),
                               "sample": f"{rows} token rows per slice x {cfg.P} slices of the {cfg.name} layer "
                                         f"(oracle fp64 numpy, decomposed ring)"}
    return out


def attention_bench(ctx, pk, iters: int, order: str = "flash", baselines: bool = True, c=None):
    import torch
    c = c or wl.ATTN
    g = torch.Generator(device="cuda")
    g.manual_seed(c.seed)
    shape = (c.m, c.heads * c.head_dim)
    Q = [torch.randn(shape, generator=g, device="cuda").to(torch.bfloat16) for _ in range(c.P)]
    K = [torch.randn(shape, generator=g, device="cuda").to(torch.bfloat16) for _ in range(c.P)]
    V = [torch.randn(shape, generator=g, device="cuda").to(torch.bfloat16) for _ in range(c.P)]
    O = [torch.empty(shape, dtype=torch.bfloat16, device="cuda") for _ in range(c.P)]
    stream = torch.cuda.current_stream()

    def call(o, compute_only=False, prune=True):
        # causal-pruned forwarding (a K/V slice goes only to the ranks that use it; the same
        # output as the full ring) unless prune is False
        kw = dict(heads=c.heads, head_dim=c.head_dim, order=o, compute_only=compute_only, causal_prune=prune)
        return lambda: ctx.qsplit_attn(Q, K, V, O, **kw)

    fns = {"main": call(order)}
    if baselines:
        # the same launches with every arrival flag published and no copy: T_compute of each order
        fns.update({"full": call(order, prune=False), "serial": call("serial"),
                    "main_c": call(order, compute_only=True), "serial_c": call("serial", compute_only=True)})
    for fn in fns.values():
        fn()
        fn()
    torch.cuda.synchronize()
    # medians of interleaved rounds, so that a slow moment of the GPU hits every variant alike
    samples = {k: [] for k in fns}
    for _ in range(5):
        for k, fn in fns.items():
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(iters):
                fn()
            b.record(stream)
            torch.cuda.synchronize()
            samples[k].append(a.elapsed_time(b) / iters)
    ctx.poll()
    t = {k: statistics.median(v) for k, v in samples.items()}
    ms = t["main"]
    tf = c.flops() / (ms * 1e-3) / 1e12
    out = {"workload": f"query-split causal attention, P={c.P}, seq {c.seq}, {c.heads} heads, head_dim "
                       f"{c.head_dim}", "order": f"{order}, causal-pruned K/V forwarding", "ms": round(ms, 4),
           "tflops": round(tf, 2),
           "frac_of_bf16_peak": round(tf / pk["bf16_burst"], 4), "flop": c.flops(),
           "flop_counting": "causal triangle only (QK^T and PV)",
           "timing": f"medians of 5 interleaved rounds of {iters} calls per variant"}
    if baselines:
        ctx.qsplit_attn(Q, K, V, O, heads=c.heads, head_dim=c.head_dim, order="serial", causal_prune=True)
        torch.cuda.synchronize()
        ring_ms, kernel_ms = ctx.phase_ms()
        full_ms, t_serial, t_c, t_serial_c = t["full"], t["serial"], t["main_c"], t["serial_c"]
        out.update({"full_ring_ms": round(full_ms, 4),
                    "serial_ms": round(t_serial, 4), "serial_phases_ms": {"ring": round(ring_ms, 4),
                                                                           "kernel": round(kernel_ms, 4)},
                    "compute_only_ms": round(t_c, 4), "serial_compute_only_ms": round(t_serial_c, 4),
                    "exposed_copy_ms": round(ms - t_c, 4),
                    "exposed_frac": round((ms - t_c) / ms, 4),
                    "full_ring_exposed_frac": round((full_ms - t_c) / full_ms, 4),
                    "serial_exposed_ms": round(t_serial - t_serial_c, 4),
                    "definition": "T_order - T_compute_only(order) (the same kernel, flags published, no copy)"})
    return out


def run_tail_rs(args, world, device, pk):
    """Small-batch tail-dominated GEMM-RS (P=8, tokens 512, in-features 28672, out 8192):
    rank-adaptive kept-slice-last order against the naive ring order and the baselines."""
    import torch
    import overlapped_tensor_gemm_gb300 as fo
    c = wl.TAIL_RS
    inp = wl.rs_inputs(c.P, c.tokens, c.n_out, c.k_row, c.seed, integer=False)

    def dev(bits):
        return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).cuda()

    X = [dev(x) for x in inp["X"]]
    W = [dev(w) for w in inp["W_row"]]
    Y = [torch.empty((c.m, c.n_out), dtype=torch.bfloat16, device="cuda") for _ in range(c.P)]
    ctx = fo.Context(device)
    stream = torch.cuda.current_stream()

    def timed(order):
        for _ in range(max(args.warmup, 3)):
            ctx.gemm_rs(X, W, Y, order=order)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(args.steps):
            ctx.gemm_rs(X, W, Y, order=order)
        b.record(stream)
        torch.cuda.synchronize()
        ctx.poll()
        return a.elapsed_time(b) / args.steps

    with ClockSampler(device) as clk:
        t = {o: timed(o) for o in ("flash", "naive", "serial", "slicing")}
    ctx.gemm_rs(X, W, Y, order="serial")
    torch.cuda.synchronize()
    ring_ms, gemm_ms = ctx.phase_ms()
    ctx.close()
    tf = c.flops() / (t["flash"] * 1e-3) / 1e12
    return {"metric": METRIC, "value": round(tf, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(t["flash"], 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"tail-dominated GEMM-RS, P={c.P}, tokens {c.tokens}, in {c.k_total}, out "
                                   f"{c.n_out}"},
            "pct_of_peak": round(100 * tf / pk["bf16_burst"], 2), "clocks": clk.summary(),
            "orders_ms": {k: round(v, 4) for k, v in t.items()},
            "serial_phases_ms": {"gemm": round(gemm_ms, 4), "ring_reduce": round(ring_ms, 4)},
            "exposed_ms": {k: round(v - gemm_ms, 4) for k, v in t.items()}}


def run_attn_layer(args, world, device, pk):
    """Attention block (Flash-AG QKV projection -> per-rank causal attention of the rank's
    heads -> Flash-RS output projection), Llama-3-8B-shaped, against its serial and
    data-slicing baselines."""
    import torch
    import overlapped_tensor_gemm_gb300 as fo
    c = wl.ATTN_LAYER
    g = torch.Generator(device="cuda")
    g.manual_seed(c.seed)
    hd = c.heads * c.head_dim
    X = [torch.randn((c.m, c.hidden), generator=g, device="cuda").to(torch.bfloat16) for _ in range(c.P)]
    Wq = [(torch.randn((3 * hd, c.hidden), generator=g, device="cuda") * wl.W_STD).to(torch.bfloat16)
          for _ in range(c.P)]
    Wo = [(torch.randn((c.hidden, hd), generator=g, device="cuda") * wl.W_STD).to(torch.bfloat16)
          for _ in range(c.P)]
    Z = [torch.empty((c.m, c.hidden), dtype=torch.bfloat16, device="cuda") for _ in range(c.P)]
    ctx = fo.Context(device)
    stream = torch.cuda.current_stream()

    def timed(order, iters):
        for _ in range(max(args.warmup, 1)):
            ctx.attn_layer(X, Wq, Wo, Z, heads=c.heads, order=order)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(iters):
            ctx.attn_layer(X, Wq, Wo, Z, heads=c.heads, order=order)
        b.record(stream)
        torch.cuda.synchronize()
        ctx.poll()
        return a.elapsed_time(b) / iters

    with ClockSampler(device) as clk:
        ms = timed("flash", args.steps)
    clocks = clk.summary()
    fl = c.flops()
    tf = fl["total"] / (ms * 1e-3) / 1e12
    res = {"metric": "attention block TFLOP/s (Flash-AG QKV, attention, Flash-RS out-projection)",
           "value": round(tf, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) activations, N(0,0.02) weights)",
           "config": {"workload": f"attention block, P={c.P}, tokens {c.tokens}, hidden {c.hidden}, "
                                  f"{c.heads * c.P} heads of {c.head_dim} ({c.heads} per rank)",
                      "l2": "inputs larger than L2 (no flush)"},
           "pct_of_peak": round(100 * tf / pk["bf16_burst"], 2), "clocks": clocks,
           "flop": fl}
    if not args.no_extras:
        res["baselines_ms"] = {o: round(timed(o, args.steps), 4) for o in ("serial", "slicing", "naive")}
    ctx.close()
    return res


def run_a2a(args, world, device, pk):
    """Flash all-to-all, Ulysses-style: the QKV projection whose output head groups go
    to their ranks (fo_gemm_a2a) and the output projection whose K chunks come from
    every rank (fo_a2a_gemm), against the serial and naive orders."""
    import torch
    import overlapped_tensor_gemm_gb300 as fo
    c = wl.A2A
    P, m, H = c.P, c.m, c.hidden
    g = torch.Generator(device="cuda")
    g.manual_seed(c.seed)
    rnd = lambda shape, sd=1.0: (torch.randn(shape, generator=g, device="cuda") * sd).to(torch.bfloat16)  # noqa: E731
    X = [rnd((m, H)) for _ in range(P)]
    Wqkv = [rnd((3 * H, H), wl.W_STD) for _ in range(P)]
    Yq = [torch.empty((P * m, 3 * H // P), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    C = [rnd((P * m, H // P)) for _ in range(P)]
    Wo = [rnd((H, H), wl.W_STD) for _ in range(P)]
    Z = [torch.empty((m, H), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    ctx = fo.Context(device)
    stream = torch.cuda.current_stream()

    def timed(fn, iters):
        for _ in range(max(args.warmup, 1)):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(iters):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        ctx.poll()
        return a.elapsed_time(b) / iters

    prod = lambda o: (lambda: ctx.gemm_a2a(X, Wqkv, Yq, order=o))  # noqa: E731
    cons = lambda o: (lambda: ctx.a2a_gemm(C, Wo, Z, order=o))  # noqa: E731
    with ClockSampler(device) as clk:
        t_prod = timed(prod("flash"), args.steps)
        t_cons = timed(cons("flash"), args.steps)
    fl = c.flops()
    ms = t_prod + t_cons
    tf = (fl["gemm_a2a"] + fl["a2a_gemm"]) / (ms * 1e-3) / 1e12
    res = {"metric": "Flash all-to-all projections TFLOP/s (QKV -> A2A, A2A -> output projection)",
           "value": round(tf, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": "bf16", "data": "synthetic (seeded N(0,1) activations, N(0,0.02) weights)",
           "config": {"workload": f"Ulysses projections, P={P}, tokens {c.tokens}, hidden {H}",
                      "l2": "inputs larger than L2 (no flush)"},
           "pct_of_peak": round(100 * tf / pk["bf16_burst"], 2), "clocks": clk.summary(),
           "gemm_a2a": {"ms": round(t_prod, 4), "tflops": round(fl["gemm_a2a"] / (t_prod * 1e-3) / 1e12, 2)},
           "a2a_gemm": {"ms": round(t_cons, 4), "tflops": round(fl["a2a_gemm"] / (t_cons * 1e-3) / 1e12, 2)}}
    if not args.no_extras:
        for name, fn in (("gemm_a2a", prod), ("a2a_gemm", cons)):
            for o in ("serial", "naive"):
                res[name][f"{o}_ms"] = round(timed(fn(o), args.steps), 4)
            fn("serial")()
            torch.cuda.synchronize()
            coll, gemm_ms = ctx.phase_ms()
            res[name]["serial_phases_ms"] = {"collective": round(coll, 4), "gemm": round(gemm_ms, 4)}
            res[name]["exposed_ms"] = round(res[name]["ms"] - gemm_ms, 4)
    ctx.close()
    return res


def run_mlp_backward(args, world, device, pk):
    """Training backward of the Llama-3-8B MLP's two projections (P=4): the down
    projection (row-parallel: dH by Flash-AG, dW local) and the gate/up projection
    (column-parallel: dX by Flash-RS, dW local), against the serial order."""
    import torch
    import overlapped_tensor_gemm_gb300 as fo
    cfg = wl.LLAMA8B
    P, m, Hd, F = cfg.P, cfg.m, cfg.hidden, cfg.ffn // cfg.P
    M = P * m
    g = torch.Generator(device="cuda")
    g.manual_seed(cfg.seed + 100)
    rnd = lambda shape, sd=1.0: (torch.randn(shape, generator=g, device="cuda") * sd).to(torch.bfloat16)  # noqa: E731
    X = [rnd((m, Hd)) for _ in range(P)]
    Wc = [rnd((2 * F, Hd), wl.W_STD) for _ in range(P)]
    dY = [rnd((M, 2 * F)) for _ in range(P)]
    dX = [torch.empty((m, Hd), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    dWc = [torch.empty((2 * F, Hd), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    H = [rnd((M, F)) for _ in range(P)]
    Wr = [rnd((Hd, F), wl.W_STD) for _ in range(P)]
    dZ = [rnd((m, Hd)) for _ in range(P)]
    dH = [torch.empty((M, F), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    dWr = [torch.empty((Hd, F), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    ctx = fo.Context(device)
    stream = torch.cuda.current_stream()

    def step(order):
        ctx.row_linear_backward(H, Wr, dZ, dH, dWr, order=order)
        ctx.col_linear_backward(X, Wc, dY, dX, dWc, order=order)

    def timed(order, iters):
        for _ in range(max(args.warmup, 1)):
            step(order)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(iters):
            step(order)
        b.record(stream)
        torch.cuda.synchronize()
        ctx.poll()
        return a.elapsed_time(b) / iters

    with ClockSampler(device) as clk:
        ms = timed("flash", args.steps)
    flop = 2 * (2 * M * Hd * F * P) + 2 * (2 * M * 2 * F * Hd * P)  # dH + dWr, dX + dWc
    tf = flop / (ms * 1e-3) / 1e12
    res = {"metric": "MLP backward TFLOP/s (dH by Flash-AG, dX by Flash-RS, local dW)", "value": round(tf, 2),
           "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": "bf16", "data": "synthetic (seeded N(0,1) activations and gradients, N(0,0.02) weights)",
           "config": {"workload": f"llama8b MLP backward, P={P}, tokens {M}, hidden {Hd}, ffn {cfg.ffn}",
                      "l2": "inputs larger than L2 (no flush)"},
           "pct_of_peak": round(100 * tf / pk["bf16_burst"], 2), "clocks": clk.summary(), "flop": flop}
    if not args.no_extras:
        res["serial_ms"] = round(timed("serial", args.steps), 4)
    ctx.close()
    return res


def run_attention_only(args, rank, world, device, pk, barrier, max_over_ranks):
    import overlapped_tensor_gemm_gb300 as fo
    ctx = fo.Context(device)
    c = wl.ATTN if args.workload == "attn" else wl.attn_sweep(int(args.workload[4:-1]) * 1024)
    res = attention_bench(ctx, pk, args.steps, args.attn_order, baselines=not args.no_extras, c=c)
    ctx.close()
    return {"metric": "query-split attention TFLOP/s", "value": res["tflops"], "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["ms"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": {"workload": res["workload"]}, "attention": res}


# --------------------------------------------------------------------------
# reference arm: the CPU oracle on a bounded sample
# --------------------------------------------------------------------------

def run_reference(args):
    cfg = mlp_config(args.workload if not (args.workload.startswith("attn") or args.workload in ("a2a", "mlp_bwd"))
                     else "llama8b")
    inp = wl.mlp_inputs(cfg)
    inp_f64 = decode_inputs(inp)
    per_step = max(2.0, min(20.0, 60.0 / max(1, args.steps + args.warmup)))
    rows = calibrate_rows(cfg, inp_f64, per_step)
    for i in range(args.warmup):
        oracle_mlp_sample(cfg, inp_f64, rows, 100 + i)
    times, flop = [], 0
    for i in range(args.steps):
        dt, flop = oracle_mlp_sample(cfg, inp_f64, rows, 200 + i)
        times.append(dt)
    ms = 1e3 * sum(times) / len(times)
    value = flop / (ms * 1e-3) / 1e12
    sample = f"{rows} token rows per slice x {cfg.P} slices of the {cfg.name} layer per step"
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{cfg.name}: MLP layer, P={cfg.P}, tokens {cfg.tokens}, hidden {cfg.hidden}, "
                                   f"ffn {cfg.ffn}"},
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args)), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    out = run_ours(args, rank, world, local)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
