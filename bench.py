#!/usr/bin/env python3
"""Benchmark of the fused QK-prep path on one GB300 (or N independent
replicas under torchrun).

Workload: the untiled 544x960 latent grid, T32 x H34 x W60 = 65,280 tokens,
24 heads x 128 channels, rotary 96 split 32/32/32 over (t, h, w), BF16 packed
QKV ~N(0,1) with 0.1 % x50 outlier columns, seeded and synthetic.  One step
prepares that tile twice, as the workload specifies: BF16 head-major Q/K/V,
then e4m3 codes with dynamic per-tensor scales (amax pass + cast pass).

Metric: algorithmic HBM bytes per second (16-bit: 12*H*D bytes per token;
e4m3 dynamic: 15*H*D, the input read twice), with tokens/s and the fraction
of the measured HBM copy peak beside it.  Inputs (1.2 GB) are larger than
L2 (129 MB), so steps do not reuse each other's data in L2.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

``--impl reference`` times the CPU oracle (test infrastructure, plain C) on
the host cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from video_vae_decoder_qkv_gb300 import workloads as W  # noqa: E402

METRIC = "fused QK-prep HBM GB/s and % of GB300 peak; tokens/s at 65k-token tile"
SPEC16 = W.LATENT_65K
SPEC8 = W.LATENT_65K_E4M3
KERNEL_FILES = ["video_vae_decoder_qkv_gb300/csrc/h3qk_kernels.cuh",
                "video_vae_decoder_qkv_gb300/csrc/h3qk_launch.cuh"]
WORKLOAD = ("latent_65k: 544x960 latent grid T32xH34xW60 = 65,280 tokens, 24 heads x 128, "
            "rotary 96 (32/32/32 over t,h,w), BF16 packed QKV ~N(0,1) with 0.1% x50 outlier "
            "columns; each step: BF16 head-major out, then e4m3 out with dynamic scales")


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tokens", type=int, default=0,
                    help="profiling only: run the first N tokens of the tile (not a bench line)")
    return ap.parse_args(argv)


# --------------------------------------------------------------------------
# ranks
# --------------------------------------------------------------------------

def rank_info():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def init_dist(world: int, backend: str):
    if world <= 1:
        return None
    import torch.distributed as dist

    if not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def barrier(dist, device=None):
    if dist is not None:
        if device is not None:
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def reduce_max_sum(dist, elapsed_s: float, units: float, device=None):
    """Max of the ranks' elapsed times and sum of their units (the whole-job
    aggregate: value = units of all ranks / slowest rank's time)."""
    if dist is None:
        return elapsed_s, units
    import torch

    dev = device if device is not None else torch.device("cpu")
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


# --------------------------------------------------------------------------
# clocks during the timed region
# --------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        # samples arrive on a pipe (no file is written)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            text, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            text, _ = self.proc.communicate()
        rows = []
        for line in (text or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        power = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(power) if power else None}


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "MEASURED_PEAKS.json hbm_gbs (measured copy)"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback 6.8 TB/s (no MEASURED_PEAKS.json)"


def kernel_sha() -> str:
    h = hashlib.sha256()
    for f in KERNEL_FILES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def recorded_traffic(key: str = "out16_latent65k"):
    """DRAM bytes (read + write) per launch of one kernel on one workload from
    the committed ncu record (profiles/traffic.json), or None when the kernel
    source changed since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("kernel_source_sha256") != kernel_sha():
        return None
    k = rec.get("kernels", {}).get(key)
    return k.get("dram_bytes_per_launch") if k else None


# --------------------------------------------------------------------------
# CPU oracle timings (baseline / reference arm)
# --------------------------------------------------------------------------

def oracle_rows(inp, rows: int, threads: int) -> tuple[float, int]:
    """Time the oracle on the first `rows` tokens of the workload, in both
    output modes; returns (seconds, algorithmic bytes)."""
    import oracle

    def pb_of(spec):
        return oracle.Problem(batch=1, seq=rows, heads=spec.heads, head_dim=spec.head_dim,
                              rotary_dim=spec.rotary_dim, n_axes=spec.n_axes,
                              axis_dims=tuple(spec.axis_dims), in_dtype=spec.in_dtype,
                              out_kind=spec.out_kind, scale_mode=spec.scale_mode, eps=spec.eps,
                              theta=spec.theta)

    qkv, pos = inp.qkv[:rows], inp.pos[:rows]
    t0 = time.perf_counter()
    oracle.prepare(pb_of(SPEC16), qkv, inp.wq, inp.wk, pos, threads=threads)
    oracle.prepare(pb_of(SPEC8), qkv, inp.wq, inp.wk, pos, threads=threads)
    dt = time.perf_counter() - t0
    hd = SPEC16.hd
    return dt, rows * hd * (12 + 15)


def cpu_threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def run_reference(args):
    rank, world, _ = rank_info()
    if rank != 0:
        return 0
    import oracle

    oracle.build()
    inp = W.generate(SPEC16)
    threads = cpu_threads()
    # size each step so the whole run stays within a few minutes
    cal_s, _ = oracle_rows(inp, 256, threads)
    rate = 256 / max(cal_s, 1e-6)
    budget = min(20.0, 150.0 / max(1, args.steps + args.warmup))
    rows = int(max(64, min(SPEC16.rows, rate * budget)))
    for _ in range(args.warmup):
        oracle_rows(inp, rows, threads)
    total_s, total_b = 0.0, 0
    for _ in range(args.steps):
        s, b = oracle_rows(inp, rows, threads)
        total_s += s
        total_b += b
    gbs = total_b / total_s / 1e9
    sample = f"first {rows} of 65,280 tokens per step, BF16 out then e4m3 dynamic"
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded)",
        "tokens_per_s": rows * args.steps / total_s,
        "config": {"workload": WORKLOAD, "sample_tokens_per_step": rows},
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------
# the CUDA path
# --------------------------------------------------------------------------

def adjacent_ops(dev, stream, iters: int = 20):
    """The decoder block's two streaming neighbours of the path, timed after
    the main region at 8x the B300 table's shapes (inputs above L2): SwiGLU on
    [14376, 2 x 8192] fp16 and the scaled residual on [28752, 2048]."""
    import torch

    from video_vae_decoder_qkv_gb300 import scaled_residual, silu_and_mul

    g = torch.Generator(device=dev).manual_seed(0)
    x = torch.randn((14376, 16384), generator=g, device=dev).to(torch.float16)
    y = torch.empty((14376, 8192), dtype=torch.float16, device=dev)
    res = torch.randn((28752, 2048), generator=g, device=dev)
    br = torch.randn((28752, 2048), generator=g, device=dev).to(torch.float16)
    sc = torch.rand(2048, generator=g, device=dev)
    out = torch.empty_like(res)
    rows = {}
    for name, fn, nbytes in (
            ("silu_and_mul", lambda: silu_and_mul(x, out=y, stream=stream), x.numel() * 2 + y.numel() * 2),
            ("scaled_residual", lambda: scaled_residual(res, br, sc, out=out, stream=stream),
             res.numel() * 4 + br.numel() * 2 + out.numel() * 4)):
        for _ in range(3):
            fn()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        a.record(stream)
        for _ in range(iters):
            fn()
        b.record(stream)
        torch.cuda.synchronize(dev)
        ms = a.elapsed_time(b) / iters
        rows[name] = {"ms": ms, "GB/s": nbytes / (ms / 1e3) / 1e9, "bytes": nbytes}
    rows["silu_and_mul"]["shape"] = [14376, 16384]
    rows["scaled_residual"]["shape"] = [28752, 2048]
    del x, y, res, br, sc, out
    torch.cuda.empty_cache()
    return rows


def variant_ops(dev, stream, qkv, wq, wk, pos, common, spec, iters: int = 20):
    """Other output forms of the path on the same tile, timed after the main
    region the way `large_configs` times its calls: the sage outputs (float32
    Q, float32 K * kv_scale, float16 V * kv_scale; 6 bytes read + 10 written
    per element) and the e4m3 cast with a static scale table (6 read + 3
    written).  CUDA events around each call on its stream, median of `iters`
    after 3 warm-ups, L2 flushed before each call by a 256 MB write."""
    import torch

    from video_vae_decoder_qkv_gb300 import prepare, prepare_sage

    N, H, D = spec.rows, spec.heads, spec.head_dim
    shape = (1, H, N, D)
    n = spec.valid_rows() * spec.hd
    rows = {}
    qs = torch.empty(shape, dtype=torch.float32, device=dev)
    ks = torch.empty(shape, dtype=torch.float32, device=dev)
    vs = torch.empty(shape, dtype=torch.float16, device=dev)
    out8 = tuple(torch.empty(shape, dtype=torch.float8_e4m3fn, device=dev) for _ in range(3))
    sc = torch.empty(3, dtype=torch.float32, device=dev)
    table = torch.tensor([0.02, 0.02, 0.01], dtype=torch.float32, device=dev)
    scratch = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for name, fn, nbytes in (
            ("sage_f32q_f32k_f16v", lambda: prepare_sage(qkv, wq, wk, pos, kv_scale=0.5, out=(qs, ks, vs),
                                                         stream=stream, **common), 16 * n),
            ("e4m3_static", lambda: prepare(qkv, wq, wk, pos, scale_mode="static", static_scales=table,
                                            out=out8, out_scales=sc, stream=stream, **common), 9 * n)):
        ts = []
        for i in range(3 + iters):
            scratch.fill_(i & 0xFF)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            if i >= 3:
                ts.append(a.elapsed_time(b))
        ms = statistics.median(ts)
        rows[name] = {"ms": ms, "GB/s": nbytes / (ms / 1e3) / 1e9, "bytes": nbytes,
                      "l2": "flushed before each call (256 MB write)"}
    del qs, ks, vs, out8, scratch
    torch.cuda.empty_cache()
    return rows


def small_calls(dev, calls: int = 50):
    """The decoder tile (4,896 tokens, 16 x 64, fp16 out) and the batch of 8
    such tiles (e4m3 dynamic): per-call GPU time from `calls` calls captured
    in one CUDA graph and replayed, which leaves out the Python and launch
    overhead that dominates an event pair around one call this small."""
    import numpy as np
    import torch

    from video_vae_decoder_qkv_gb300 import prepare

    rows = {}
    for spec in (W.DECODER_TILE, W.BATCHED_FP8):
        inp = W.generate(spec)
        dt = torch.float16 if spec.in_dtype == W.FP16 else torch.bfloat16
        qkv = torch.from_numpy(inp.qkv.view(np.int16)).to(dev).view(dt)
        wq, wk, pos = (torch.from_numpy(a).to(dev) for a in (inp.wq, inp.wk, inp.pos))
        mode = {W.SCALE_NONE: "none", W.SCALE_DYNAMIC: "dynamic", W.SCALE_STATIC: "static"}[spec.scale_mode]
        shape = (spec.batch, spec.heads, spec.seq, spec.head_dim)
        odt = torch.float8_e4m3fn if spec.out_kind == W.OUT_E4M3 else dt
        out = tuple(torch.empty(shape, dtype=odt, device=dev) for _ in range(3))
        sc = torch.empty(3, device=dev)
        ws = torch.zeros(4, dtype=torch.int32, device=dev)
        side = torch.cuda.Stream(dev)
        kw = dict(heads=spec.heads, head_dim=spec.head_dim, rotary_dim=spec.rotary_dim, batch=spec.batch,
                  valid_len=spec.valid_len, scale_mode=mode, n_axes=spec.n_axes, axis_dims=spec.axis_dims,
                  out=out, out_scales=sc, workspace=ws, stream=side)
        try:
            with torch.cuda.stream(side):
                for _ in range(3):
                    prepare(qkv, wq, wk, pos, **kw)
            torch.cuda.synchronize(dev)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                for _ in range(calls):
                    prepare(qkv, wq, wk, pos, **kw)
            ts = []
            for _ in range(10):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                g.replay()
                b.record()
                b.synchronize()
                ts.append(a.elapsed_time(b) / calls)
            ms = statistics.median(ts)
            rows[spec.name] = {"us_per_call": 1e3 * ms, "GB/s": spec.algorithmic_bytes() / (ms / 1e3) / 1e9,
                               "bytes": spec.algorithmic_bytes(), "tokens": spec.rows,
                               "mode": "fp16 out" if mode == "none" else f"e4m3 {mode}"}
            del g
        except Exception as e:  # noqa: BLE001 - report, do not fail the bench line
            rows[spec.name] = {"error": str(e)[:200]}
        del qkv, out
        torch.cuda.empty_cache()
    return rows


def large_configs(dev, peak: float, iters: int = 20):
    """The 104,080-row prefix workload (40 heads x 128, rotary 128 on 1-D
    positions, valid prefix 104,076, 0.05 % x50 outlier columns) cast to
    e4m3 under a static table and under dynamic scales: per-call GPU time by
    CUDA events on the call's stream, median of `iters` calls after 3
    warm-ups, with L2 flushed before each call by a 256 MB scratch write."""
    import numpy as np
    import torch

    from video_vae_decoder_qkv_gb300 import prepare

    rows = {}
    spec = W.PREFIX_104K_STATIC
    inp = W.generate(spec)
    qkv = torch.from_numpy(inp.qkv.view(np.int16)).to(dev).view(torch.bfloat16)
    wq, wk, pos = (torch.from_numpy(a).to(dev) for a in (inp.wq, inp.wk, inp.pos))
    table = torch.from_numpy(inp.static_scales).to(dev)
    shape = (spec.batch, spec.heads, spec.seq, spec.head_dim)
    out = tuple(torch.empty(shape, dtype=torch.float8_e4m3fn, device=dev) for _ in range(3))
    sc = torch.empty(3, device=dev)
    ws = torch.zeros(4, dtype=torch.int32, device=dev)
    scratch = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    side = torch.cuda.Stream(dev)
    kw = dict(heads=spec.heads, head_dim=spec.head_dim, rotary_dim=spec.rotary_dim, valid_len=spec.valid_len,
              n_axes=spec.n_axes, axis_dims=spec.axis_dims, out=out, out_scales=sc, workspace=ws, stream=side)
    try:
        for cfg in (W.PREFIX_104K_STATIC, W.PREFIX_104K_DYNAMIC):
            mode = "static" if cfg.scale_mode == W.SCALE_STATIC else "dynamic"
            st = table if mode == "static" else None
            ts = []
            with torch.cuda.stream(side):
                for i in range(3 + iters):
                    scratch.fill_(i & 0xFF)
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(side)
                    prepare(qkv, wq, wk, pos, scale_mode=mode, static_scales=st, **kw)
                    b.record(side)
                    b.synchronize()
                    if i >= 3:
                        ts.append(a.elapsed_time(b))
            ms = statistics.median(ts)
            gbs = cfg.algorithmic_bytes() / (ms / 1e3) / 1e9
            rows[cfg.name] = {"ms": ms, "GB/s": gbs, "pct_of_peak": 100.0 * gbs / peak,
                              "pct_of_nominal_8tbs": gbs / 80.0,
                              "bytes": cfg.algorithmic_bytes(), "valid_tokens": cfg.valid_rows(),
                              "mode": f"e4m3 {mode}", "l2": "flushed before each call (256 MB write)"}
    except Exception as e:  # noqa: BLE001 - report, do not fail the bench line
        rows["error"] = str(e)[:200]
    del qkv, out, scratch
    torch.cuda.empty_cache()
    return rows


def pass_rooflines(dev, peak: float, iters: int = 20):
    """The two passes of the dynamic e4m3 call, each timed alone through the
    split entry points (h3qk_amax, then h3qk_cast with that amax): the
    65,280-token latent tile and the 104,080-row prefix, plus the prefix's
    static-table cast.  CUDA events on the launching stream around each
    launch, median of `iters` after 3 warm-ups, L2 flushed before each by a
    256 MB write.  Algorithmic bytes per launch: amax reads 6*H*D per valid
    token; cast reads 6*H*D and writes 3*H*D."""
    import numpy as np
    import torch

    from video_vae_decoder_qkv_gb300 import amax as amax_pass
    from video_vae_decoder_qkv_gb300 import cast as cast_pass
    from video_vae_decoder_qkv_gb300 import prepare

    rows = {}
    scratch = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    side = torch.cuda.Stream(dev)
    for spec in (W.LATENT_65K_E4M3, W.PREFIX_104K_DYNAMIC):
        inp = W.generate(spec)
        qkv = torch.from_numpy(inp.qkv.view(np.int16)).to(dev).view(torch.bfloat16)
        wq, wk, pos = (torch.from_numpy(a).to(dev) for a in (inp.wq, inp.wk, inp.pos))
        table = torch.from_numpy(inp.static_scales).to(dev)
        shape = (spec.batch, spec.heads, spec.seq, spec.head_dim)
        out = tuple(torch.empty(shape, dtype=torch.float8_e4m3fn, device=dev) for _ in range(3))
        sc = torch.empty(3, device=dev)
        am = torch.empty(3, device=dev)
        kw = dict(heads=spec.heads, head_dim=spec.head_dim, rotary_dim=spec.rotary_dim, valid_len=spec.valid_len,
                  n_axes=spec.n_axes, axis_dims=spec.axis_dims, stream=side)
        n = spec.valid_rows() * spec.hd
        calls = (("amax", lambda: amax_pass(qkv, wq, wk, pos, out=am, **kw), 6 * n),
                 ("cast", lambda: cast_pass(qkv, wq, wk, pos, am, out=out, out_scales=sc, **kw), 9 * n))
        if spec.name.startswith("prefix"):
            calls += (("static_cast", lambda: prepare(qkv, wq, wk, pos, scale_mode="static", static_scales=table,
                                                      out=out, out_scales=sc, **kw), 9 * n),)
        try:
            for name, fn, nbytes in calls:
                ts = []
                with torch.cuda.stream(side):
                    for i in range(3 + iters):
                        scratch.fill_(i & 0xFF)
                        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                        a.record(side)
                        fn()
                        b.record(side)
                        b.synchronize()
                        if i >= 3:
                            ts.append(a.elapsed_time(b))
                ms = statistics.median(ts)
                gbs = nbytes / (ms / 1e3) / 1e9
                tag = spec.name.split("_")[0]
                key = {"latent": "latent65k", "prefix": "prefix104k"}[tag]
                rows[f"{tag}_{name}"] = {
                    "kernel": f"qkprep_kernel<bf16, LPR=8, CH=2, {'amax' if name == 'amax' else 'cast'}>",
                    "ms": ms, "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                    "algorithmic_bytes_per_launch": nbytes,
                    "traffic": recorded_traffic(f"{name}_{key}")}
        except Exception as e:  # noqa: BLE001 - report, do not fail the bench line
            rows[f"{spec.name}_error"] = str(e)[:200]
        del qkv, out
        torch.cuda.empty_cache()
    del scratch
    torch.cuda.empty_cache()
    return rows


def run_ours(args):
    import numpy as np
    import torch

    from video_vae_decoder_qkv_gb300 import h3qk, prepare

    rank, world, local = rank_info()
    if world != args.gpus and world > 1:
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE {world}", file=sys.stderr)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    h3qk.lib()   # fail loudly now if the library is missing

    spec16, spec8 = SPEC16, SPEC8
    if args.tokens:
        spec16 = SPEC16.with_(seq=args.tokens, grid=None)
        spec8 = SPEC8.with_(seq=args.tokens, grid=None)
    inp = W.generate(spec16)      # each rank: its own replica of the tile
    N, H, D = spec16.rows, spec16.heads, spec16.head_dim
    qkv_h = torch.from_numpy(inp.qkv.view(np.int16)).view(torch.bfloat16)
    qkv = qkv_h.to(dev)
    wq = torch.from_numpy(inp.wq).to(dev)
    wk = torch.from_numpy(inp.wk).to(dev)
    pos = torch.from_numpy(inp.pos).to(dev)
    shape = (1, H, N, D)
    out16 = tuple(torch.empty(shape, dtype=torch.bfloat16, device=dev) for _ in range(3))
    out8 = tuple(torch.empty(shape, dtype=torch.float8_e4m3fn, device=dev) for _ in range(3))
    scales = torch.empty(3, dtype=torch.float32, device=dev)
    ws = torch.zeros(4, dtype=torch.int32, device=dev)
    common = dict(heads=H, head_dim=D, rotary_dim=spec16.rotary_dim, n_axes=3,
                  axis_dims=spec16.axis_dims, theta=spec16.theta, eps=spec16.eps)
    stream = torch.cuda.current_stream(dev)

    def call16():
        prepare(qkv, wq, wk, pos, out=out16, stream=stream, **common)

    def call8():
        prepare(qkv, wq, wk, pos, scale_mode="dynamic", out=out8, out_scales=scales, workspace=ws,
                stream=stream, **common)

    for _ in range(max(3, args.warmup)):
        call16()
        call8()
    torch.cuda.synchronize(dev)

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    sampler.start()
    barrier(dist, dev)
    torch.cuda.synchronize(dev)
    h3qk.launch_count_reset()
    start.record(stream)
    for i in range(K):
        ev[i][0].record(stream)
        call16()
        ev[i][1].record(stream)
        call8()
        ev[i][2].record(stream)
    end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(dist, dev)
    launches = h3qk.launch_count()
    clocks = sampler.stop()
    elapsed_s = start.elapsed_time(end) / 1e3
    t16 = statistics.fmean(e[0].elapsed_time(e[1]) for e in ev) / 1e3
    t8 = statistics.fmean(e[1].elapsed_time(e[2]) for e in ev) / 1e3

    bytes16 = spec16.algorithmic_bytes()
    bytes8 = spec8.algorithmic_bytes()
    step_bytes = bytes16 + bytes8
    t_max, total_bytes = reduce_max_sum(dist, elapsed_s, step_bytes * K, dev)

    # end to end through the C-ABI call on host buffers (h3qk_prepare_host):
    # each of the step's two calls copies its inputs from pinned host memory,
    # computes in overlapping chunks and copies its outputs back
    from video_vae_decoder_qkv_gb300 import h3qk as _h, prepare_host

    E = max(1, min(args.e2e_steps, K))
    qkv_pin = qkv_h.pin_memory()
    wq_pin, wk_pin, pos_pin = (t.cpu().pin_memory() for t in (wq, wk, pos))
    host16 = tuple(torch.empty(shape, dtype=torch.bfloat16).pin_memory() for _ in range(3))
    host8 = tuple(torch.empty(shape, dtype=torch.uint8).pin_memory() for _ in range(3))
    host_sc = torch.empty(3, dtype=torch.float32).pin_memory()
    o = _h.default_opts()
    o.in_dtype, o.n_axes = _h.BF16, 3
    ws_bytes = max(_h.host_workspace_bytes(N, H, D, _h.BF16, _h.SCALE_NONE, o),
                   _h.host_workspace_bytes(N, H, D, _h.E4M3, _h.SCALE_DYNAMIC, o))
    host_ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    in_bytes = sum(t.numel() * t.element_size() for t in (qkv_pin, wq_pin, wk_pin, pos_pin))
    h2d = 2 * in_bytes
    d2h = sum(t.numel() * t.element_size() for t in (*host16, *host8, host_sc))

    def e2e_step():
        prepare_host(qkv_pin, wq_pin, wk_pin, pos_pin, out=host16, workspace=host_ws, stream=stream, **common)
        prepare_host(qkv_pin, wq_pin, wk_pin, pos_pin, scale_mode="dynamic", out=host8, out_scales=host_sc,
                     workspace=host_ws, stream=stream, **common)

    e2e_step()
    torch.cuda.synchronize(dev)
    barrier(dist, dev)
    es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    es.record(stream)
    for _ in range(E):
        e2e_step()
    ee.record(stream)
    torch.cuda.synchronize(dev)
    e2e_s = es.elapsed_time(ee) / 1e3
    e2e_max, e2e_bytes = reduce_max_sum(dist, e2e_s, step_bytes * E, dev)

    large = large_configs(dev, measured_peak()[0]) if not args.tokens else None
    passes = pass_rooflines(dev, measured_peak()[0]) if not args.tokens else None
    variants = variant_ops(dev, stream, qkv, wq, wk, pos, common, spec16)
    extra = adjacent_ops(dev, stream) if not args.tokens else None
    small = small_calls(dev) if not args.tokens else None

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.tokens:
        rows = N
        threads = cpu_threads()
        s, b = oracle_rows(inp, rows, threads)
        cpu = {"value": b / s / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
               "sample": f"all {rows} tokens of the tile once, BF16 out then e4m3 dynamic, {threads} threads",
               "seconds": s}
        # the same oracle on one thread (row ranges do not change its bytes)
        rows1 = min(N, 4096)
        s1, b1 = oracle_rows(inp, rows1, 1)
        cpu["single_thread"] = {"value": b1 / s1 / 1e9, "unit": "GB/s", "cores": 1, "seconds": s1,
                                "sample": f"first {rows1} tokens of the tile, BF16 out then e4m3 dynamic"}

    if rank == 0:
        peak, peak_src = measured_peak()
        value = total_bytes / t_max / 1e9
        ach16 = bytes16 / t16 / 1e9
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K,
            "warmup": max(3, args.warmup), "ms_per_step": 1e3 * t_max / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "io_dtype": "bf16 in; bf16 and e4m3 out",
            "data": "synthetic (seeded numpy draws; random weights)",
            "pct_of_peak": 100.0 * value / peak,
            "pct_of_nominal_8tbs": 100.0 * value / 8000.0,
            "tokens_per_s": N * K * world / t_max,
            "config": {"workload": WORKLOAD if not args.tokens else
                       f"profiling case: first {N} tokens of the 65k tile (not a bench line)",
                       "tokens": N, "heads": H, "head_dim": D, "rotary_dim": spec16.rotary_dim, "global_batch": world,
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "l2": "inputs larger than L2 (1.20 GB packed QKV per pass)"},
            "kernels": {
                "norm_rope_permute_bf16": {"ms": 1e3 * t16, "GB/s": ach16, "bytes": bytes16,
                                           "tokens_per_s": N / t16},
                "e4m3_dynamic_amax_plus_cast": {"ms": 1e3 * t8, "GB/s": bytes8 / t8 / 1e9,
                                                "bytes": bytes8, "tokens_per_s": N / t8},
            },
            "roofline": {"bound": "hbm", "kernel": "qkprep_kernel<bf16, LPR=8, CH=2, out16> (one launch)",
                         "achieved": ach16, "peak": peak, "unit": "GB/s", "frac": ach16 / peak,
                         "traffic": recorded_traffic(), "peak_source": peak_src,
                         "algorithmic_bytes_per_launch": bytes16},
            "pass_rooflines": passes,
            "e2e": {"value": e2e_bytes / e2e_max / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": E, "api": "h3qk_prepare_host (host buffers, chunked copies overlapped with the kernels), both calls of the step"},
            "gpu_launches": launches,
            "variants": variants,
            "small_calls": small,
            "large_configs": large,
            "adjacent_ops": extra,
            "clocks": clocks,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
