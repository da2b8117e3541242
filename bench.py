"""Benchmark of the block-sparse FlexAttention forward on one GB300.

A step is one pass of the hot path over the workload already resident in
HBM: the BlockMask build (flex_block_mask_create) and the attention forward
(flex_attention_fwd), both through the C-ABI.  The metric is forward TFLOP/s
counted over unmasked blocks only (4 * 128 * 128 * D per full or partial
tile), also given as a fraction of the dense bf16 tensor peak.

Prints ONE JSON line (rank 0).  `--impl reference` times the float64 CPU
oracle on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from block_sparse_masked_blockmask_gb300 import workloads as W  # noqa: E402

METRIC = "flex-attn fwd TFLOP/s (unmasked blocks) and % of GB300 bf16 tensor peak"
UNIT = "TFLOP/s"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0
# NVIDIA's published dense bf16 tensor rate of one GB300 GPU: 36 PFLOP/s for an
# 8-GPU HGX B300 board is quoted with 2:4 sparsity, i.e. 2.25 PFLOP/s dense each.
SPEC_BF16_TFLOPS = 2250.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "attn_bf16_traffic.txt")
KERNEL_SOURCES = ["attn_bf16_kernel.cuh", "attn_bf16_launch.cuh", "attn_bf16.cu", "attn_bf16_d64.cu",
                  "attn_bf16_d128.cu", "ptx.cuh", "flex_internal.h", "tilelist.cuh"]


def workload_by_name(name: str) -> W.Workload:
    for w in W.CONFIGS:
        if w.name == name:
            return w
    raise SystemExit(f"unknown workload {name}; choose from {[w.name for w in W.CONFIGS]}")


def tile_counts(bm: dict) -> np.ndarray:
    """Computed tiles (full + partial) per (b, h, q block)."""
    return bm["kv_num_blocks"].astype(np.int64) + bm["full_kv_num_blocks"].astype(np.int64)


def unmasked_block_flops(w: W.Workload, bm: dict) -> float:
    return float(tile_counts(bm).sum()) * 4.0 * 128 * 128 * w.D


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"bf16": float(d["bf16_tflops"]), "bf16_sustained": float(d.get("bf16_tflops_sustained", 0.0)),
                "hbm": float(d["hbm_gbs"]), "source": "measured"}
    return {"bf16": FALLBACK_BF16_TFLOPS, "bf16_sustained": 0.0, "hbm": FALLBACK_HBM_GBS, "source": "fallback"}


def kernel_sources_digest() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "block_sparse_masked_blockmask_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it matches the current kernel sources."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    rec = {}
    with open(TRAFFIC_FILE) as f:
        for line in f:
            if "=" in line and not line.startswith("#"):
                k, v = line.strip().split("=", 1)
                rec[k.strip()] = v.strip()
    if rec.get("workload") != workload or rec.get("sources_sha256_16") != kernel_sources_digest():
        return None
    try:
        return float(rec["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.device_index = device_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.device_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        time.sleep(0.15)
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self) -> dict:
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = max(mx, float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": mx or None,
                "reasons": sorted(reasons), "samples": len(sm)}


def oracle_rows_baseline(w: W.Workload, q, k, v, docs, bm: dict, budget_s: float) -> dict:
    """The float64 oracle timed on a bounded sample of the workload's rows (host cores)."""
    import oracle
    tiles = tile_counts(bm)  # [B, H, NQB]
    total_rows = w.B * w.H * w.S
    rng = np.random.default_rng(5)

    def run(n):
        rows = np.sort(rng.choice(total_rows, size=min(n, total_rows), replace=False)).astype(np.int64)
        t0 = time.perf_counter()
        oracle.workload_attention(w, q, k, v, docs, rows=rows)
        dt = time.perf_counter() - t0
        i = rows % w.S
        bh = rows // w.S
        flops = float((tiles.reshape(-1, tiles.shape[-1])[bh, i // 128] * 4.0 * 128 * w.D).sum())
        return rows.size, dt, flops

    n0, t0, _ = run(256)
    n = int(min(total_rows, max(256, n0 * budget_s / max(t0, 1e-3))))
    n, dt, flops = run(n)
    return {"value": flops / dt / 1e12, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{n} of {total_rows} query rows of {w.name} (all keys of each row, float64), "
                      f"{dt:.1f} s; TFLOP/s credits each row its share of unmasked-block FLOPs"}


def run_reference(args, w: W.Workload) -> None:
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    q, k, v, docs = W.workload_inputs(w)
    import oracle
    bm = oracle.workload_block_mask(w, docs)
    # each step is a bounded sample; the whole run stays within a few minutes
    per_step = args.ref_seconds if args.ref_seconds > 0 else min(6.0, 150.0 / (args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_rows_baseline(w, q, k, v, docs, bm, budget_s=min(per_step, 0.5))
    vals, secs = [], []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        r = oracle_rows_baseline(w, q, k, v, docs, bm, budget_s=per_step)
        secs.append(time.perf_counter() - t0)
        vals.append(r["value"])
    value = float(np.median(vals))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * float(np.median(secs)),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_dict(w),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": r["cores"], "kind": "oracle",
                             "sample": r["sample"]},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def config_dict(w: W.Workload) -> dict:
    c = {"workload": w.name, "B": w.B, "H": w.H, "S": w.S, "D": w.D, "block": 128,
         "mask": W.MASK_NAMES[w.mask], "score": W.SCORE_NAMES[w.score], "scale": w.scale,
         "input_dtype": w.dtype}
    if w.mask == W.MASK_SLIDING_WINDOW:
        c["window"] = w.window
    if w.mask == W.MASK_CAUSAL_PREFIX:
        c["prefix"] = w.prefix
    if w.score == W.SCORE_SOFTCAP:
        c["softcap"] = w.softcap
    qkv_bytes = 3 * w.B * w.H * w.S * w.D * (2 if w.dtype == "bf16" else 4)
    c["l2"] = (f"inputs larger than L2 ({qkv_bytes / 2**20:.0f} MiB of Q/K/V vs 129 MiB), no flush"
               if qkv_bytes > L2_BYTES else "L2 flushed between steps (256 MiB write)")
    return c


def max_over_ranks(ms: float, dist=None, device="cuda") -> float:
    """The largest of the ranks' times (every rank gets it); `ms` itself on one process."""
    if dist is None:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(flops_per_rank: float, ms: float, world: int) -> float:
    """TFLOP/s of all ranks together: each rank did flops_per_rank (weak scaling) in at most ms."""
    return world * flops_per_rank / (ms * 1e-3) / 1e12


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=W.BF16_CAUSAL_ALIBI_S16384.name)
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="oracle sample budget (cpu_baseline)")
    ap.add_argument("--ref-seconds", type=float, default=0.0,
                    help="oracle sample budget per reference step (0: fit the run in ~150 s)")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--e2e-chunks", type=int, default=16,
                    help="(b, h) chunks of flex_attention_fwd_host, whose copies overlap the work")
    ap.add_argument("--option-steps", type=int, default=20,
                    help="launches per kernel-option variant (OUTPUT_MAX, PRESCALE_QK, ...); 0 skips them")
    ap.add_argument("--backward-steps", type=int, default=5,
                    help="timed flex_attention_bwd launches on the same workload; 0 skips them")
    ap.add_argument("--config-steps", type=int, default=50,
                    help="timed attention launches on each of the five synthetic configurations; 0 skips them")
    ap.add_argument("--fp32-steps", type=int, default=10,
                    help="timed float32 launches at B1 H16 S4096 (D = 64, 128); 0 skips them")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=None, help="override B (profiling a smaller case)")
    ap.add_argument("--heads", type=int, default=None, help="override H (profiling a smaller case)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    w = workload_by_name(args.workload)
    if args.batch or args.heads:
        w = W.scaled(w, B=args.batch or w.B, H=args.heads or w.H, name=w.name + "_profiling_subset")
    if args.impl == "reference":
        run_reference(args, w)
        return
    run_ours(args, w)


def prepare_device_inputs(torch, w: W.Workload):
    """The workload's seeded inputs on the device (the same bits the oracle sees)."""
    q, k, v, docs = W.workload_inputs(w)

    def to_dev(x):
        if w.dtype == "bf16":
            return torch.from_numpy(W.bf16_bits(x).view(np.int16)).cuda().view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(x)).cuda()

    dd = torch.from_numpy(docs).cuda() if docs is not None else None
    return (q, k, v, docs), (to_dev(q), to_dev(k), to_dev(v), dd)


def config_timings(fa, torch, device_index: int, steps: int, peaks: dict) -> dict | None:
    """Attention-kernel throughput on every synthetic configuration (outside the headline's timed region).

    Per configuration: the BlockMask is built once, 10 untimed launches, then
    `steps` attention launches are timed one by one with CUDA events on the
    launching stream, L2 flushed before each launch when the inputs fit in L2,
    clocks sampled while they run.  TFLOP/s counts unmasked-block FLOPs over
    the median launch time (the mean is reported beside it).
    """
    if steps <= 0:
        return None
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 * 2**20, dtype=torch.uint8, device="cuda")
    res = {}
    for w in W.CONFIGS:
        _, (dq, dk, dv, dd) = prepare_device_inputs(torch, w)
        out = torch.empty_like(dq)
        lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device="cuda")
        bm = fa.flex_block_mask_create(w.mask, w.B, w.H, w.S, w.S, 128, window=w.window, prefix=w.prefix,
                                       doc_ids=dd, stream=stream)
        flops = unmasked_block_flops(w, bm.as_numpy())
        small = 3 * dq.numel() * dq.element_size() <= L2_BYTES

        def launch():
            fa.flex_attention_fwd(dq, dk, dv, bm, w.score, w.score_param, w.scale, out=out, lse=lse, stream=stream)

        for _ in range(10):
            launch()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        with ClockSampler(device_index) as clocks:
            for a, b in ev:
                if small:
                    flush.zero_()
                a.record(stream)
                launch()
                b.record(stream)
            torch.cuda.synchronize()
        if fa.flex_device_status() != fa.FLEX_OK:
            raise RuntimeError(f"device status reported a timeout on {w.name}")
        ms = [a.elapsed_time(b) for a, b in ev]
        mean, median = float(np.mean(ms)), float(np.median(ms))
        tflops = flops / (median * 1e-3) / 1e12
        res[w.name] = {"dtype": w.dtype, "unmasked_block_flops": flops, "attn_ms_mean": mean,
                       "attn_ms_median": median, "tflops": tflops, "tflops_of_mean": flops / (mean * 1e-3) / 1e12,
                       "frac_of_measured_bf16_peak": tflops / peaks["bf16"],
                       "frac_of_spec_bf16_peak": tflops / SPEC_BF16_TFLOPS,
                       "kernel": "attn_bf16_kernel" if w.dtype == "bf16" else "attn_fp32_kernel (three-way bf16 split, tcgen05)",
                       "l2": "flushed before each launch" if small else "inputs larger than L2",
                       "launches": steps, "clocks": clocks.summary()}
        del dq, dk, dv, dd, out, lse, bm
        torch.cuda.empty_cache()
    return res


def kernel_option_timings(fa, torch, w, dq, dk, dv, bm, out, lse, stream, flush, flops, steps):
    """Attention launches under each kernel option (outside the headline's timed region).

    The variants run interleaved, one launch each per round, on the same
    BlockMask and inputs, so clock drift falls on all of them alike.
    """
    if steps <= 0:
        return None
    row_max = torch.empty_like(lse)
    variants = {
        "default": {},
        "output_max": {"max_scores": row_max},
        "prescale_qk": {"prescale_qk": True},
        "rows_guaranteed_safe": {"rows_guaranteed_safe": True},
        "all": {"max_scores": row_max, "prescale_qk": True, "rows_guaranteed_safe": True},
    }

    def launch(opts):
        fa.flex_attention_fwd_opts(dq, dk, dv, bm, w.score, w.score_param, w.scale, out=out, lse=lse,
                                   stream=stream, **opts)

    for opts in variants.values():
        launch(opts)
    torch.cuda.synchronize()
    ev = {name: [] for name in variants}
    for _ in range(steps):
        for name, opts in variants.items():
            if flush is not None:
                flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            launch(opts)
            b.record(stream)
            ev[name].append((a, b))
    torch.cuda.synchronize()
    if fa.flex_device_status() != fa.FLEX_OK:
        raise SystemExit("device status reported a timeout during the kernel-option launches")
    ms = {name: float(np.mean([a.elapsed_time(b) for a, b in pairs])) for name, pairs in ev.items()}
    return {"api": "flex_attention_fwd_opts", "launches_each": steps, "ms_per_launch": ms,
            "tflops": {name: flops / (t * 1e-3) / 1e12 for name, t in ms.items()}}


# bf16 MMA FLOPs the float32 path executes per product FLOP (three-way split, six products)
FP32_SPLIT_PRODUCTS = 6


def fp32_bwd_executed(D):
    """Product FLOPs the fp32 backward executes per algorithmic FLOP (10 D per
    computed pair): S and dP are recomputed by the dK/dV and the dQ kernels
    (14 D), and at D = 128 by both 64-column halves of dK/dV (18 D)."""
    return 1.4 if D == 64 else 1.8


def fp32_bwd_kernels(D):
    if D == 64:
        return "attn_bwd_delta (CUDA cores) + bwdf32::dkdv_kernel + bwdf32::dq_kernel (tcgen05)"
    return "attn_bwd_delta (CUDA cores) + bwdf32::dkdv128_kernel + bwdf32::dq128_kernel (tcgen05)"


def fp32_scale_timings(fa, torch, device_index: int, steps: int, peaks: dict) -> dict | None:
    """The float32 path (three-way bf16 split on tcgen05) at a size where it is throughput-bound.

    The five synthetic configurations hold one float32 case, small enough for
    the oracle; this one is the same kind (causal, identity score) at
    B1 H16 S4096, D = 64 and 128.  Each product takes six bf16 MMAs, so the
    tensor cores execute 6x the algorithmic FLOPs; the ceiling of the
    algorithmic rate is the measured bf16 burst / 6.  The float32 backward
    is timed on the same inputs: at D = 64 on the tensor cores (the same
    split, against the same ceiling); at D = 128 dK/dV run on the CUDA cores
    and dQ on the tensor cores, reported against the CUDA cores' fp32 FMA
    rate.
    """
    if steps <= 0:
        return None
    stream = torch.cuda.current_stream()
    ceiling = peaks["bf16"] / FP32_SPLIT_PRODUCTS
    res = {"kernel": "attn_fp32_kernel (three-way bf16 split, tcgen05)", "ceiling_tflops": ceiling,
           "ceiling_source": f"{peaks['source']} bf16 burst / {FP32_SPLIT_PRODUCTS} (bf16 MMA FLOPs per FLOP)"}
    for D in (64, 128):
        w = W.scaled(W.FP32_CAUSAL_S256, name=f"fp32_causal_b1h16s4096d{D}", H=16, S=4096, D=D)
        _, (dq, dk, dv, _) = prepare_device_inputs(torch, w)
        out = torch.empty_like(dq)
        lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device="cuda")
        bm = fa.flex_block_mask_create(w.mask, w.B, w.H, w.S, w.S, 128, stream=stream)
        flops = unmasked_block_flops(w, bm.as_numpy())

        def launch():
            fa.flex_attention_fwd(dq, dk, dv, bm, w.score, w.score_param, w.scale, out=out, lse=lse, stream=stream)

        for _ in range(3):
            launch()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        with ClockSampler(device_index) as clocks:
            for a, b in ev:
                a.record(stream)
                launch()
                b.record(stream)
            torch.cuda.synchronize()
        if fa.flex_device_status() != fa.FLEX_OK:
            raise RuntimeError(f"device status reported a timeout on {w.name}")
        ms = float(np.mean([a.elapsed_time(b) for a, b in ev]))
        achieved = flops / (ms * 1e-3) / 1e12
        # backward: 2.5x the forward's algorithmic FLOPs (see backward_timings)
        gen = torch.Generator(device=dq.device).manual_seed(1)
        dout = torch.randn(out.shape, generator=gen, device=dq.device, dtype=torch.float32)
        bq = fa.flex_block_mask_transpose(bm, stream=stream)
        gq, gk, gv = torch.empty_like(dq), torch.empty_like(dk), torch.empty_like(dv)

        def launch_bwd():
            fa.flex_attention_bwd(dq, dk, dv, out, lse, dout, bm, bq, w.score, w.score_param, w.scale, dq=gq,
                                  dk=gk, dv=gv, stream=stream)

        launch_bwd()
        torch.cuda.synchronize()
        evb = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(2)]
        for a, b in evb:
            a.record(stream)
            launch_bwd()
            b.record(stream)
        torch.cuda.synchronize()
        if fa.flex_device_status() != fa.FLEX_OK:
            raise RuntimeError(f"device status reported a timeout in the backward on {w.name}")
        ms_b = float(np.mean([a.elapsed_time(b) for a, b in evb]))
        bwd_tflops = 2.5 * flops / (ms_b * 1e-3) / 1e12
        bwd_roof = {"bound": "tensor", "peak": ceiling, "frac": bwd_tflops / ceiling,
                    "peak_source": "measured bf16 burst / 6",
                    "executed_bf16_mma_tflops": bwd_tflops * fp32_bwd_executed(D) * FP32_SPLIT_PRODUCTS,
                    "kernels": fp32_bwd_kernels(D)}
        res[w.name] = {"ms_per_launch": ms, "unmasked_block_flops": flops, "tflops": achieved,
                       "executed_bf16_mma_tflops": FP32_SPLIT_PRODUCTS * achieved,
                       "frac_of_ceiling": achieved / ceiling,
                       "l2": "K and V (64 MB at D = 128) stay in L2 across launches", "launches": steps,
                       "clocks": clocks.summary(),
                       "backward": {"ms_per_launch": ms_b, "launches": len(evb), "tflops": bwd_tflops, **bwd_roof}}
        del dq, dk, dv, out, lse, bm, bq, dout, gq, gk, gv
        torch.cuda.empty_cache()
    return res


def backward_timings(fa, torch, w, dq, dk, dv, bm, out, lse, stream, flops_fwd, steps, peaks):
    """flex_attention_bwd on the bench workload (outside the headline's timed region).

    Algorithmic FLOPs: per computed pair, the recomputed score and dP dots and
    the dV, dK, dQ updates, 10 D, i.e. 2.5 x the forward's 4 D.  The bf16
    kernels execute 14 D per pair (the dQ kernel recomputes the score and dP
    dots instead of accumulating dQ across CTAs); the roofline counts the
    algorithmic 10 D.
    """
    if steps <= 0:
        return None
    gen = torch.Generator(device=dq.device).manual_seed(1)
    dout = torch.randn(out.shape, generator=gen, device=dq.device, dtype=torch.float32).to(out.dtype)
    bq = fa.flex_block_mask_transpose(bm, stream=stream)
    gq, gk, gv = torch.empty_like(dq), torch.empty_like(dk), torch.empty_like(dv)
    delta = torch.empty_like(lse)

    def launch():
        fa.flex_attention_bwd(dq, dk, dv, out, lse, dout, bm, bq, w.score, w.score_param, w.scale, dq=gq, dk=gk,
                              dv=gv, delta=delta, stream=stream)

    launch()
    torch.cuda.synchronize()
    ev = []
    for _ in range(steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        launch()
        b.record(stream)
        ev.append((a, b))
    torch.cuda.synchronize()
    if fa.flex_device_status() != fa.FLEX_OK:
        raise RuntimeError("device status reported a timeout during the backward launches")
    if not (torch.isfinite(gq).all() and torch.isfinite(gk).all() and torch.isfinite(gv).all()):
        raise RuntimeError("non-finite gradients")
    ms = float(np.mean([a.elapsed_time(b) for a, b in ev]))
    flops = 2.5 * flops_fwd
    achieved = flops / (ms * 1e-3) / 1e12
    if w.dtype == "bf16":
        roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16"],
                "frac_of_sustained": achieved / peaks["bf16_sustained"] if peaks["bf16_sustained"] else None,
                "peak_source": f"{peaks['source']} bf16 burst (dense cuBLAS); frac_of_sustained: the seconds-long figure",
                "executed_mma_flops": 3.5 * flops_fwd,
                "kernels": "attn_bwd_delta (CUDA cores) + attn_bwd_tc<dK,dV> + attn_bwd_tc<dQ> (tcgen05)"}
    else:
        ceiling = peaks["bf16"] / FP32_SPLIT_PRODUCTS
        roof = {"bound": "tensor", "achieved": achieved, "peak": ceiling, "unit": "TFLOP/s",
                "frac": achieved / ceiling, "peak_source": f"{peaks['source']} bf16 burst / 6",
                "executed_bf16_mma_flops": fp32_bwd_executed(w.D) * FP32_SPLIT_PRODUCTS * flops,
                "kernels": fp32_bwd_kernels(w.D)}
    return {"api": "flex_attention_bwd", "launches": steps, "ms_per_launch": ms, "algorithmic_flops": flops,
            "roofline": roof}


def run_ours(args, w: W.Workload) -> None:
    import torch
    from block_sparse_masked_blockmask_gb300 import flexattn as fa

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    (q, k, v, docs), (dq, dk, dv, dd) = prepare_device_inputs(torch, w)
    out = torch.empty_like(dq)
    lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    flush = None
    if 3 * dq.numel() * dq.element_size() <= L2_BYTES:
        flush = torch.empty(256 * 2**20, dtype=torch.uint8, device="cuda")

    def step():
        bm = fa.flex_block_mask_create(w.mask, w.B, w.H, w.S, w.S, 128, window=w.window, prefix=w.prefix,
                                       doc_ids=dd, stream=stream)
        fa.flex_attention_fwd(dq, dk, dv, bm, w.score, w.score_param, w.scale, out=out, lse=lse, stream=stream)
        return bm

    bm = None
    for _ in range(args.warmup):
        bm = step()
    torch.cuda.synchronize()
    if fa.flex_device_status() != fa.FLEX_OK:
        raise SystemExit("device status reported a timeout during warm-up")
    bm_host = bm.as_numpy()
    flops = unmasked_block_flops(w, bm_host)

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        for i in range(args.steps):
            if flush is not None:
                flush.zero_()
            e0, e1, e2 = ev[i]
            e0.record(stream)
            bmi = fa.flex_block_mask_create(w.mask, w.B, w.H, w.S, w.S, 128, window=w.window, prefix=w.prefix,
                                            doc_ids=dd, stream=stream)
            e1.record(stream)
            fa.flex_attention_fwd(dq, dk, dv, bmi, w.score, w.score_param, w.scale, out=out, lse=lse,
                                  stream=stream)
            e2.record(stream)
        torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    if fa.flex_device_status() != fa.FLEX_OK:
        raise SystemExit("device status reported a timeout during the timed region")
    step_ms = [a.elapsed_time(c) for a, _, c in ev]
    attn_ms = [b.elapsed_time(c) for _, b, c in ev]
    total_ms = max_over_ranks(float(np.sum(step_ms)), dist)
    ms_per_step = total_ms / args.steps
    value = whole_job_rate(flops, ms_per_step, world)

    # end to end through the public API: host inputs in, host outputs back, every step
    hq, hk, hv = (x.cpu().pin_memory() for x in (dq, dk, dv))
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    hlse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    hdoc = torch.from_numpy(docs).pin_memory() if docs is not None else None
    h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv)) + (hdoc.numel() * 4 if hdoc is not None else 0)
    d2h = hout.numel() * hout.element_size() + hlse.numel() * 4

    # flex_attention_fwd_host: the copies of chunk c + 1 (of the (b, h) pairs)
    # overlap the BlockMask-driven attention of chunk c and the copy back of c - 1
    bufs = fa.DeviceBuffers(w.B, w.H, w.S, w.S, w.D, dq.dtype, document=docs is not None)

    def e2e_step():
        fa.flex_attention_fwd_host(hq, hk, hv, bufs, w.mask, hout, hlse, window=w.window, prefix=w.prefix,
                                   doc_ids=hdoc, score_kind=w.score, score_param=w.score_param, scale=w.scale,
                                   chunks=args.e2e_chunks, stream=stream)

    e2e = None
    if args.e2e_steps > 0:
        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(args.e2e_steps):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(a.elapsed_time(b) / args.e2e_steps, dist)
        # the host result is the device path's result
        if not (torch.equal(hout[0, 0].float(), out[0, 0].float().cpu()) and torch.equal(hlse[-1, -1], lse[-1, -1].cpu())):
            raise SystemExit("flex_attention_fwd_host result differs from flex_attention_fwd")
        e2e = {"value": whole_job_rate(flops, e2e_ms, world), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "ms_per_step": e2e_ms, "api": "flex_attention_fwd_host",
               "chunks": args.e2e_chunks}

    options = kernel_option_timings(fa, torch, w, dq, dk, dv, bm, out, lse, stream, flush, flops,
                                    args.option_steps)

    if rank != 0:
        return
    peaks = measured_peaks()
    attn_mean_ms = float(np.mean(attn_ms))
    achieved = flops / (attn_mean_ms * 1e-3) / 1e12
    traffic = recorded_traffic(w.name)
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16"], "traffic": traffic,
                "kernel": "attn_bf16_kernel" if w.dtype == "bf16" else "attn_fp32_kernel",
                "peak_source": f"{peaks['source']} bf16 burst (dense cuBLAS)",
                "achieved_hbm_gbs": None if traffic is None else traffic / (attn_mean_ms * 1e-3) / 1e9,
                "algorithmic_flops_per_launch": flops, "mean_launch_ms": attn_mean_ms}
    configs = None
    try:
        configs = config_timings(fa, torch, local, args.config_steps, peaks)
    except Exception as exc:  # noqa: BLE001
        configs = {"error": f"{type(exc).__name__}: {exc}"}
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = oracle_rows_baseline(w, q, k, v, docs, bm_host, budget_s=args.cpu_seconds)
    # the backward pass last: an error there is reported in its own field
    # and leaves the forward's numbers above as measured
    fp32_scale = None
    try:
        fp32_scale = fp32_scale_timings(fa, torch, local, args.fp32_steps, peaks)
    except Exception as exc:  # noqa: BLE001
        fp32_scale = {"error": f"{type(exc).__name__}: {exc}"}
    backward = None
    try:
        backward = backward_timings(fa, torch, w, dq, dk, dv, bm, out, lse, stream, flops, args.backward_steps,
                                    peaks)
    except Exception as exc:  # noqa: BLE001
        backward = {"error": f"{type(exc).__name__}: {exc}"}
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
            "config": config_dict(w), "pct_of_bf16_peak": 100.0 * value / peaks["bf16"],
            "pct_of_spec_bf16_peak": 100.0 * value / SPEC_BF16_TFLOPS,
            "spec_bf16_peak": {"value": SPEC_BF16_TFLOPS, "unit": "TFLOP/s",
                               "source": "NVIDIA HGX B300: 36 PFLOP/s bf16 per 8 GPUs with 2:4 sparsity, "
                                         "i.e. 2.25 PFLOP/s dense per GPU"},
            "roofline": roofline, "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": 2 * args.steps, "clocks": clocks.summary(),
            "attn_ms_per_launch": {"mean": attn_mean_ms, "median": float(np.median(attn_ms)),
                                   "min": float(np.min(attn_ms))},
            "block_mask_ms_per_launch": float(np.mean(np.asarray(step_ms) - np.asarray(attn_ms))),
            "kernel_options": options, "backward": backward, "configs": configs,
            "fp32_at_scale": fp32_scale}
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
