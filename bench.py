#!/usr/bin/env python3
"""Benchmark of the tile-partitioned dense GEMM D = alpha*A*B + beta*C on GB300.

One step = one gemm_run (a single kernel launch: the whole hot path, tile
schedule + TMA ring + tcgen05 MMA + epilogue) on one batch of synthetic input
resident in HBM. The default workload is the square 4096^3 bf16 GEMM; the QKV
projection, the MLP down-projection with residual and the M=16 decode shape are
measured the same way and reported under "per_config".

L2: every step reads its own copy of the inputs, drawn from rotating device
buffer sets whose total size exceeds 3x the L2 cache, so no launch finds its
operands already in L2 (no flush kernel runs inside the timed region).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun (N > 1) every rank runs its own independent GEMM (weak scaling,
no data-path collective); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
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

METRIC = "bf16 GEMM TFLOP/s (% of GB300 dense BF16 peak); decode-shape HBM GB/s (% peak)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_NAMES = {"tiled": "tpg::tiled::gemm_tiled_kernel", "stream": "tpg::stream::gemm_stream_kernel"}
# Dense bf16 tensor-core work per SM per SM clock cycle, measured on GB300 with a
# standalone tcgen05.mma loop (no loads, no epilogue, all SMs): a CTA pair runs
# a 256 x 256 x 64 block (four 256 x 256 x 16 MMAs) in 512 cycles, i.e.
# 2 * 256 * 256 * 64 / 2 SMs / 512 = 8192 flop per SM per cycle.
MMA_FLOP_PER_SM_CYCLE = 8192
SUSTAINED_SECONDS = 2.0
REPS = 21


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="square")
    ap.add_argument("--no-extra", action="store_true", help="skip the per_config measurements")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="budget of the oracle sample")
    ap.add_argument("--no-sustained", action="store_true", help="skip the repetitions and the sustained regions")
    ap.add_argument("--only-mx", action="store_true", help="of the per_config rows, measure the block-scaled (MXFP8, FP4) ones only")
    ap.add_argument("--only-rows", default=None,
                    help="comma-separated names of the block-scaled rows to measure (implies --only-mx)")
    return ap.parse_args()


# ----------------------------------------------------------------------------- environment

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(values, world: int, device=None):
    """Element-wise maximum of `values` over all ranks: the slowest rank's
    times, which bound the whole job. Needs an initialised process group when
    world > 1 (NCCL with CUDA tensors in the bench; gloo on CPU in the tests)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def job_throughput(world: int, steps: int, work_per_step: float, span_ms: float, scale: float) -> float:
    """Whole-job rate: the work of all ranks (each ran `steps` steps of
    `work_per_step` units) over the slowest rank's time span_ms, in units of
    `scale` per second (1e12 for TFLOP/s, 1e9 for GB/s)."""
    return world * steps * work_per_step / (span_ms * 1e-3) / scale


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_sha() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "tile_partitioned_dense_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh")):
            with open(os.path.join(csrc, f), "rb") as fh:
                h.update(fh.read())
    return h.hexdigest()[:16]


def profile_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary of this kernel on
    this workload, or None when there is none or the kernel changed since."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    sha = re.search(r"kernel_source_sha:\s*([0-9a-f]+)", text)
    dram = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not sha or not dram or sha.group(1) != kernel_source_sha():
        return None
    return float(dram.group(1))


class ClockSampler:
    """nvidia-smi samples (every 100 ms) of SM clock and throttle reasons."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r.split(", ") for r in self.file.read().strip().splitlines() if r.strip()]
        os.unlink(self.file.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[0]))
                mx.append(float(r[1]))
                for name, v in zip(names, r[4:8]):
                    if v.strip() == "Active":
                        reasons.add(name)
            except (ValueError, IndexError):
                continue
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- our arm

class Workload:
    """Device copies of one config's inputs, replicated into rotating sets."""

    def __init__(self, cfg, torch, l2_bytes: int, pinned: bool):
        from workloads import make_inputs
        self.cfg = cfg
        A, B, C = make_inputs(cfg)
        self.host = {"A": A, "B": B, "C": C}
        out = torch.float32 if cfg.out_dtype == "f32" else torch.bfloat16
        self.out_dtype = out
        self.out_code = 1 if out == torch.float32 else 0
        per_set = A.numel() * 2 + B.numel() * 2 + (cfg.M * cfg.N * (4 if out == torch.float32 else 2)) * (
            2 if C is not None else 1)
        self.nsets = max(2, -(-3 * l2_bytes // per_set) + 1)
        dev = torch.device("cuda")
        self.sets = []
        for _ in range(self.nsets):
            s = {"A": A.to(dev), "B": B.to(dev), "C": C.to(dev) if C is not None else None,
                 "D": torch.empty((cfg.M, cfg.N), dtype=out, device=dev)}
            self.sets.append(s)
        if pinned:
            self.pin = {k: (v.pin_memory() if v is not None else None) for k, v in self.host.items()}
            self.pin["D"] = torch.empty((cfg.M, cfg.N), dtype=out).pin_memory()
        self.bytes_A = A.numel() * 2
        self.bytes_B = B.numel() * 2
        self.bytes_C = C.numel() * C.element_size() if C is not None else 0
        self.bytes_D = cfg.M * cfg.N * (4 if out == torch.float32 else 2)

    def run(self, tpd, h, i, stream):
        s = self.sets[i % self.nsets]
        c = self.cfg
        C = s["C"]
        return tpd.gemm_run(h, c.M, c.N, c.K, s["A"].data_ptr(), c.K, s["B"].data_ptr(), c.N,
                            C.data_ptr() if C is not None else None, c.N, s["D"].data_ptr(), c.N,
                            c.alpha, c.beta, self.out_code, stream)


class TorchMatmul:
    """The same workload through torch.matmul (cuBLAS), on the same rotating
    device buffers: the comparison row of the measurement (not our path)."""

    def __init__(self, wl):
        self.wl = wl

    def run(self, tpd, h, i, stream):
        import torch
        s = self.wl.sets[i % self.wl.nsets]
        c = self.wl.cfg
        if s["C"] is not None and c.beta != 0.0:
            torch.addmm(s["C"], s["A"], s["B"], beta=c.beta, alpha=c.alpha, out=s["D"])
        elif c.alpha == 1.0:
            torch.mm(s["A"], s["B"], out=s["D"])
        else:
            torch.addmm(s["D"], s["A"], s["B"], beta=0.0, alpha=c.alpha, out=s["D"])
        return 0


def torch_matmul_entry(torch, tpd, h, wl, steps, ours_ms, barrier):
    span, _ = time_launches(torch, tpd, h, TorchMatmul(wl), steps, 5, barrier)
    ms = span / steps
    c = wl.cfg
    if c.name == "decode":
        value, unit = c.K * c.N * 2 / (ms * 1e-3) / 1e9, "GB/s"
    else:
        value, unit = c.flops / (ms * 1e-3) / 1e12, "TFLOP/s"
    return {"value": round(value, 2), "unit": unit, "ms_per_step": round(ms, 5), "steps": steps,
            "ours_over_torch": round(ms / ours_ms, 3)}


class MultiWorkload:
    """Batched (bmm) or grouped (mixture-of-experts) GEMM through
    gemm_run_batched / gemm_run_grouped, with rotating device copies."""

    def __init__(self, torch, l2_bytes, kind, M, N, K, count, group_rows=None):
        g = torch.Generator().manual_seed(77)
        self.kind, self.M, self.N, self.K, self.count = kind, M, N, K, count
        self.group_rows = group_rows
        rows = M * count if kind == "bmm" else sum(group_rows)
        self.rows = rows
        a = (torch.randn(rows, K, generator=g)).to(torch.bfloat16)
        b = (torch.randn(count, K, N, generator=g) * 0.02).to(torch.bfloat16)
        per_set = a.numel() * 2 + b.numel() * 2 + rows * N * 2
        self.nsets = max(2, -(-3 * l2_bytes // per_set) + 1)
        self.sets = [{"A": a.cuda(), "B": b.cuda(), "D": torch.empty(rows, N, dtype=torch.bfloat16, device="cuda")}
                     for _ in range(self.nsets)]
        self.flops = 2 * rows * N * K

    def run(self, tpd, h, i, stream):
        s = self.sets[i % self.nsets]
        if self.kind == "bmm":
            return tpd.gemm_run_batched(h, self.count, self.M, self.N, self.K, s["A"].data_ptr(), self.K,
                                        self.M * self.K, s["B"].data_ptr(), self.N, self.K * self.N, None, self.N, 0,
                                        s["D"].data_ptr(), self.N, self.M * self.N, 1.0, 0.0, 0, stream)
        return tpd.gemm_run_grouped(h, self.group_rows, self.N, self.K, s["A"].data_ptr(), self.K, s["B"].data_ptr(),
                                    self.N, self.K * self.N, None, self.N, s["D"].data_ptr(), self.N, 1.0, 0.0, 0,
                                    stream)


class MxWorkload:
    """A block-scaled (MXFP8) workload through gemm_run_mx: E4M3 A and B's
    transpose, E8M0 scales in the blocked layout, bf16 D, rotating device copies."""

    def __init__(self, cfg, torch, l2_bytes):
        from workloads import make_mx_inputs, mx_blocked_scales
        self.cfg = cfg
        A, SA, Bt, SB = make_mx_inputs(cfg.M, cfg.N, cfg.K, seed=cfg.seed)
        self.host = (A, SA, Bt, SB)
        sa = torch.from_numpy(mx_blocked_scales(SA.numpy()))
        sb = torch.from_numpy(mx_blocked_scales(SB.numpy()))
        per_set = A.numel() + Bt.numel() + sa.numel() + sb.numel() + cfg.M * cfg.N * 2
        self.nsets = max(2, -(-3 * l2_bytes // per_set) + 1)
        self.sets = [{"A": A.cuda(), "B": Bt.cuda(), "SA": sa.cuda(), "SB": sb.cuda(),
                      "D": torch.empty((cfg.M, cfg.N), dtype=torch.bfloat16, device="cuda")}
                     for _ in range(self.nsets)]
        self.b_bytes = Bt.numel() + sb.numel()

    def run(self, tpd, h, i, stream):
        s = self.sets[i % self.nsets]
        c = self.cfg
        return tpd.gemm_run_mx(h, c.M, c.N, c.K, s["A"].data_ptr(), c.K, tpd.FP8_E4M3, s["SA"].data_ptr(),
                               s["B"].data_ptr(), c.K, tpd.FP8_E4M3, s["SB"].data_ptr(), None, c.N,
                               s["D"].data_ptr(), c.N, 1.0, 0.0, tpd.OUT_BF16, stream)


class TorchScaledMM:
    """The same MXFP8 workload through torch._scaled_mm (NVIDIA's library
    kernel), on the same buffers: a comparison row, not this library's path."""

    def __init__(self, wl, torch):
        self.wl = wl
        self.torch = torch

    def run(self, tpd, h, i, stream):
        torch = self.torch
        s = self.wl.sets[i % self.wl.nsets]
        a = s["A"].view(torch.float8_e4m3fn)
        b = s["B"].view(torch.float8_e4m3fn).t()
        torch._scaled_mm(a, b, s["SA"].view(torch.float8_e8m0fnu), s["SB"].view(torch.float8_e8m0fnu),
                         out_dtype=torch.bfloat16, out=s["D"])
        return 0


class Fp4Workload:
    """A block-scaled FP4 workload through gemm_run_fp4: packed E2M1 A and B's
    transpose (N(0,1) data quantised per block), scales in the blocked layout,
    bf16 D, rotating device copies."""

    def __init__(self, cfg, torch, l2_bytes):
        from workloads import E4M3_ONE, FP4_NV, make_fp4_inputs, mx_blocked_scales
        self.cfg = cfg
        A, SA, Bt, SB = make_fp4_inputs(cfg.M, cfg.N, cfg.K, seed=cfg.seed, fmt=cfg.fmt)
        self.host = (A, SA, Bt, SB)
        pad = E4M3_ONE if cfg.fmt == FP4_NV else 127
        sa = torch.from_numpy(mx_blocked_scales(SA.numpy(), pad=pad))
        sb = torch.from_numpy(mx_blocked_scales(SB.numpy(), pad=pad))
        per_set = A.numel() + Bt.numel() + sa.numel() + sb.numel() + cfg.M * cfg.N * 2
        self.nsets = max(2, -(-3 * l2_bytes // per_set) + 1)
        self.sets = [{"A": A.cuda(), "B": Bt.cuda(), "SA": sa.cuda(), "SB": sb.cuda(),
                      "D": torch.empty((cfg.M, cfg.N), dtype=torch.bfloat16, device="cuda")}
                     for _ in range(self.nsets)]
        self.b_bytes = Bt.numel() + sb.numel()

    def run(self, tpd, h, i, stream):
        s = self.sets[i % self.nsets]
        c = self.cfg
        return tpd.gemm_run_fp4(h, c.M, c.N, c.K, c.fmt, s["A"].data_ptr(), c.K // 2, s["SA"].data_ptr(),
                                s["B"].data_ptr(), c.K // 2, s["SB"].data_ptr(), None, c.N, s["D"].data_ptr(), c.N,
                                1.0, 0.0, tpd.OUT_BF16, stream)


class TorchScaledMMFp4:
    """The same FP4 workload through torch._scaled_mm (NVIDIA's library
    kernel), on the same buffers: a comparison row, not this library's path.
    NVFP4 scales are E4M3, MXFP4 scales E8M0."""

    def __init__(self, wl, torch):
        self.wl = wl
        self.torch = torch

    def run(self, tpd, h, i, stream):
        from workloads import FP4_NV
        torch = self.torch
        s = self.wl.sets[i % self.wl.nsets]
        a = s["A"].view(torch.float4_e2m1fn_x2)
        b = s["B"].view(torch.float4_e2m1fn_x2).t()
        sdt = torch.float8_e4m3fn if self.wl.cfg.fmt == FP4_NV else torch.float8_e8m0fnu
        torch._scaled_mm(a, b, s["SA"].view(sdt), s["SB"].view(sdt), out_dtype=torch.bfloat16, out=s["D"])
        return 0


def block_scaled_rows(torch, tpd, h, l2, peaks, local, barrier, args, rows):
    """Bench rows of the block-scaled GEMMs. Each row: TFLOP/s against the
    format's tensor peak (the measured bf16 peak times the nominal ratio:
    FP8 2, FP4 6) or, for the HBM-bound shapes, bytes of B and its scales per
    second against the HBM copy peak; with torch._scaled_mm on the same
    buffers when this torch offers it, and the oracle's CPU baseline."""
    out = {}
    keep = set(args.only_rows.split(",")) if args.only_rows else None
    for r in rows:
        if keep is not None and r["name"] not in keep:
            continue
        name, cfg, wl = r["name"], r["cfg"], r["make"](r["cfg"], torch, l2)
        plan = r["plan"](cfg)
        steps = r["steps"]
        span, eager = time_launches(torch, tpd, h, wl, steps, 10, barrier)
        ms = span / steps
        hbm = r["hbm"]
        tpeak = r["ratio"] * peaks["bf16_tflops"]
        if hbm:
            v, unit, peak, bound = wl.b_bytes / (ms * 1e-3) / 1e9, "GB/s", peaks["hbm_gbs"], "hbm"
        else:
            v, unit, peak, bound = cfg.flops / (ms * 1e-3) / 1e12, "TFLOP/s", tpeak, "tensor"
        e = {"value": round(v, 2), "unit": unit, "ms_per_step": round(ms, 5), "eager_ms_per_step": round(eager / steps, 5),
             "steps": steps, "tflops": round(cfg.flops / (ms * 1e-3) / 1e12, 2),
             "roofline": {"bound": bound, "achieved": round(v, 2), "peak": peak, "unit": unit,
                          "frac": round(v / peak, 4), "kernel": "tpg::mx::gemm_mx_kernel",
                          "peak_source": f"{r['ratio']:g} x MEASURED_PEAKS.json bf16 burst (nominal ratio)" if not hbm
                          else "MEASURED_PEAKS.json hbm_gbs"},
             "config": {"workload": f"{name}: {cfg.description}", "M": cfg.M, "N": cfg.N, "K": cfg.K,
                        "l2": f"inputs larger than L2: {wl.nsets} rotating device copies"},
             "plan": plan}
        if not args.no_sustained:
            work = wl.b_bytes if hbm else cfg.flops
            times = time_reps(torch, tpd, h, wl, REPS)
            med, best = statistics.median(times), min(times)
            sc = 1e9 if hbm else 1e12
            e["reps"] = {"count": REPS, "median_ms": round(med, 5), "best_ms": round(best, 5),
                         "median": round(work / (med * 1e-3) / sc, 2), "best": round(work / (best * 1e-3) / sc, 2),
                         "unit": unit}
            if r.get("sustained"):
                sms, n, secs, clocks = time_sustained(torch, tpd, h, wl, ms, SUSTAINED_SECONDS, local)
                sv = work / (sms * 1e-3) / sc
                speak = r["ratio"] * peaks["bf16_tflops_sustained"]
                e["sustained"] = {"value": round(sv, 2), "unit": unit, "ms_per_launch": round(sms, 5), "launches": n,
                                  "seconds": round(secs, 3), "peak": speak, "frac": round(sv / speak, 4),
                                  "peak_key": f"{r['ratio']:g} x bf16_tflops_sustained", "clocks": clocks}
        if r.get("torch") is not None:
            try:
                tspan, _ = time_launches(torch, tpd, h, r["torch"](wl, torch), min(steps, 100), 3, barrier)
                tms = tspan / min(steps, 100)
                e["torch_scaled_mm"] = {"ms_per_step": round(tms, 5), "ours_over_torch": round(tms / ms, 3)}
            except Exception as exc:  # this torch may not offer the format in scaled_mm
                e["torch_scaled_mm"] = {"unavailable": f"{type(exc).__name__}: {str(exc).splitlines()[0][:160]}"}
                torch.cuda.synchronize()
        if r.get("cpu"):
            e["cpu_baseline"] = r["cpu"](cfg, wl.host, 3.0)
        out[name] = e
        del wl
        torch.cuda.empty_cache()
    return out


def mx_entries(torch, tpd, h, l2, peaks, local, barrier, rank, world, args):
    """The MXFP8 rows (QKV and medium shapes tensor-bound, decode HBM-bound)."""
    from workloads import MX_CONFIGS
    cpu = mx_cpu_baseline if rank == 0 and world == 1 and not args.no_cpu_baseline else None
    plan = lambda c: tpd.gemm_mx_query_plan(h, c.M, c.N, c.K)  # noqa: E731
    rows = [{"name": n, "cfg": MX_CONFIGS[n], "make": MxWorkload, "torch": TorchScaledMM, "plan": plan,
             "ratio": 2.0, "hbm": n == "mx_decode", "steps": 200 if n == "mx_qkv" else 400,
             "sustained": n == "mx_qkv", "cpu": cpu} for n in ["mx_qkv", "mx_medium", "mx_decode"]]
    return block_scaled_rows(torch, tpd, h, l2, peaks, local, barrier, args, rows)


def fp4_entries(torch, tpd, h, l2, peaks, local, barrier, rank, world, args):
    """The FP4 rows: NVFP4 on the decode shape and a 256-row one, HBM-bound
    (bytes of B and its scales per second), and on the QKV shape against the
    FP4 tensor peak (the measured bf16 peak times the nominal FP4 : bf16 ratio
    of 6); MXFP4 on the QKV shape, the same way."""
    from workloads import FP4_CONFIGS
    cpu = fp4_cpu_baseline if rank == 0 and world == 1 and not args.no_cpu_baseline else None
    plan = lambda c: tpd.gemm_fp4_query_plan(h, c.fmt, c.M, c.N, c.K)  # noqa: E731
    rows = [{"name": n, "cfg": FP4_CONFIGS[n], "make": Fp4Workload, "torch": TorchScaledMMFp4, "plan": plan,
             "ratio": 6.0, "hbm": not n.endswith("_qkv"), "steps": 200 if n.endswith("_qkv") else 400,
             "sustained": n == "nvfp4_qkv", "cpu": cpu} for n in ["nvfp4_qkv", "nvfp4_m256", "nvfp4_decode", "mxfp4_qkv"]]
    return block_scaled_rows(torch, tpd, h, l2, peaks, local, barrier, args, rows)


def fp4_cpu_baseline(cfg, host, budget_s):
    """The block-scaled oracle as it stands, on a bounded row sample of the FP4 workload."""
    import oracle
    from workloads import FP4_BLOCK, FP4_NV, sample_rows
    A, SA, Bt, SB = host
    sf = oracle.SCALE_E4M3 if cfg.fmt == FP4_NV else oracle.SCALE_E8M0
    threads = len(os.sched_getaffinity(0))

    def run(rows):
        oracle.bs_gemm_rows(A, SA, Bt, SB, None, 1.0, 0.0, 0, oracle.FP4_E2M1, oracle.FP4_E2M1, sf,
                            FP4_BLOCK[cfg.fmt], rows=rows, nthreads=threads)

    probe = sample_rows(cfg.M, max(1, min(cfg.M, threads)), seed=7)
    t0 = time.perf_counter()
    run(probe)
    per_row = (time.perf_counter() - t0) / len(probe)
    nrows = int(max(len(probe), min(cfg.M, budget_s / max(per_row, 1e-9))))
    rows = sample_rows(cfg.M, nrows, seed=11)
    t0 = time.perf_counter()
    run(rows)
    dt = time.perf_counter() - t0
    return {"value": 2.0 * len(rows) * cfg.N * cfg.K / dt / 1e12, "unit": "TFLOP/s", "cores": threads,
            "kind": "oracle", "sample": f"{len(rows)} of {cfg.M} rows of {cfg.name}, {dt:.1f} s, fp64 C block-scaled "
                                        f"oracle, {threads} threads"}


def mx_cpu_baseline(cfg, host, budget_s):
    """The MX oracle as it stands, on a bounded row sample of the same workload."""
    import oracle
    from workloads import sample_rows
    A, SA, Bt, SB = host
    threads = len(os.sched_getaffinity(0))
    probe = sample_rows(cfg.M, max(1, min(cfg.M, threads)), seed=7)
    t0 = time.perf_counter()
    oracle.mx_gemm_rows(A, SA, Bt, SB, None, 1.0, 0.0, 0, rows=probe, nthreads=threads)
    per_row = (time.perf_counter() - t0) / len(probe)
    nrows = int(max(len(probe), min(cfg.M, budget_s / max(per_row, 1e-9))))
    rows = sample_rows(cfg.M, nrows, seed=11)
    t0 = time.perf_counter()
    oracle.mx_gemm_rows(A, SA, Bt, SB, None, 1.0, 0.0, 0, rows=rows, nthreads=threads)
    dt = time.perf_counter() - t0
    return {"value": 2.0 * len(rows) * cfg.N * cfg.K / dt / 1e12, "unit": "TFLOP/s", "cores": threads,
            "kind": "oracle", "sample": f"{len(rows)} of {cfg.M} rows of {cfg.name}, {dt:.1f} s, fp64 C MX oracle, "
                                        f"{threads} threads"}


class FusedWorkload(Workload):
    """A workload whose epilogue adds a bias row, applies an activation and
    multiplies by an auxiliary [M, N] tensor: fused into gemm_run_epilogue, or
    (unfused) the plain GEMM followed by the same element-wise work in torch."""

    def __init__(self, cfg, torch, l2_bytes, activation, fused):
        super().__init__(cfg, torch, l2_bytes, pinned=False)
        g = torch.Generator().manual_seed(cfg.seed + 100)
        self.torch = torch
        self.act = activation
        self.fused = fused
        bias = (torch.randn(cfg.N, generator=g) * 0.1).to(torch.bfloat16).cuda()
        for st in self.sets:
            st["bias"] = bias
            st["aux"] = torch.rand(cfg.M, cfg.N, generator=g).to(self.out_dtype).cuda()

    def run(self, tpd, h, i, stream):
        if not self.fused:
            st = super().run(tpd, h, i, stream)
            s = self.sets[i % self.nsets]
            torch = self.torch
            f = {1: torch.relu, 2: torch.sigmoid, 3: torch.tanh}[self.act]
            s["D"].copy_(f(s["D"] + s["bias"]) * s["aux"])
            return st
        s = self.sets[i % self.nsets]
        c = self.cfg
        epi = tpd.Epilogue(s["bias"].data_ptr(), tpd.OUT_BF16, self.act, s["aux"].data_ptr(), c.N)
        C = s["C"]
        return tpd.gemm_run_epilogue(h, c.M, c.N, c.K, s["A"].data_ptr(), c.K, s["B"].data_ptr(), c.N,
                                     C.data_ptr() if C is not None else None, c.N, s["D"].data_ptr(), c.N,
                                     c.alpha, c.beta, self.out_code, epi, stream)


def time_launches(torch, tpd, h, wl, steps, warmup, barrier):
    """Time `steps` back-to-back launches, bracketed by barrier + synchronize.

    The launches are captured once into a CUDA graph (gemm_run allocates
    nothing and never synchronises, so it is capture-safe) and the graph is
    replayed inside the timed region, so the number is the GPU's, not the
    Python launch loop's. Returns (span_ms, eager_span_ms): the device time
    from the first launch's start to the last launch's end for the graph
    replay, and the same for an eager loop of the same launches (context).
    """
    stream = torch.cuda.current_stream()
    for i in range(warmup):
        assert wl.run(tpd, h, i, stream.cuda_stream) == 0
    torch.cuda.synchronize()
    # graph of exactly `steps` launches over the rotating buffer sets
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            cap = torch.cuda.current_stream().cuda_stream
            for i in range(steps):
                st = wl.run(tpd, h, i, cap)
                if st != 0:
                    raise RuntimeError(tpd.gemm_status_string(st))
    stream.wait_stream(side)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    graph.replay()
    t1.record(stream)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    span = t0.elapsed_time(t1)
    # eager loop (host issues every launch), after the timed region: context only
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        st = wl.run(tpd, h, warmup + i, stream.cuda_stream)
        if st != 0:
            raise RuntimeError(tpd.gemm_status_string(st))
    e1.record(stream)
    torch.cuda.synchronize()
    eager = e0.elapsed_time(e1)
    st = tpd.gemm_sync_status(h, None)
    if st != 0:
        raise RuntimeError("device status: " + tpd.gemm_status_string(st))
    del graph
    return span, eager


def time_reps(torch, tpd, h, wl, reps, warmup=3):
    """`reps` isolated launches, each timed on its own with CUDA events on the
    launching stream (a short device sleep ahead of each keeps the host's
    launch latency out of the interval), each on the next rotating buffer set
    so that its operands are not in L2. Returns the per-launch times in ms."""
    stream = torch.cuda.current_stream()
    for i in range(warmup):
        if wl.run(tpd, h, i, stream.cuda_stream) != 0:
            raise RuntimeError("warm-up launch failed")
    torch.cuda.synchronize()
    times = []
    for i in range(reps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(100_000)
        e0.record(stream)
        st = wl.run(tpd, h, warmup + i, stream.cuda_stream)
        e1.record(stream)
        if st != 0:
            raise RuntimeError(tpd.gemm_status_string(st))
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    if tpd.gemm_sync_status(h, None) != 0:
        raise RuntimeError("device status after the timed repetitions")
    return times


def time_sustained(torch, tpd, h, wl, est_ms, seconds, gpu_index):
    """Back-to-back launches for at least `seconds`: a CUDA graph of G launches
    (about 25 ms of work) replayed R times between two CUDA events, with
    nvidia-smi sampling the SM clock and throttle reasons meanwhile. Under the
    power cap a dense GEMM settles below its burst clock within a fraction of
    a second, so this is the figure to hold against the sustained peak.
    Returns (ms per launch, launches, seconds, clocks)."""
    g = max(1, min(2000, int(25.0 / max(est_ms, 1e-3))))
    reps = max(1, int(seconds * 1e3 / (g * est_ms)) + 1)
    stream = torch.cuda.current_stream()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            cap = torch.cuda.current_stream().cuda_stream
            for i in range(g):
                st = wl.run(tpd, h, i, cap)
                if st != 0:
                    raise RuntimeError(tpd.gemm_status_string(st))
    stream.wait_stream(side)
    graph.replay()  # warm
    torch.cuda.synchronize()
    sampler = ClockSampler(gpu_index)
    sampler.start()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    ms = e0.elapsed_time(e1)
    if tpd.gemm_sync_status(h, None) != 0:
        raise RuntimeError("device status after the sustained region")
    del graph
    return ms / (g * reps), g * reps, ms / 1e3, clocks


def work_of(cfg):
    """(work per launch, scale, unit) of the config's headline metric: bytes of
    B for the decode shape, flops for the others."""
    if cfg.name == "decode":
        return cfg.K * cfg.N * 2, 1e9, "GB/s"
    return cfg.flops, 1e12, "TFLOP/s"


def measure_extra(torch, tpd, h, wl, cfg, avg_ms, peaks, gpu_index, reps=REPS, seconds=SUSTAINED_SECONDS):
    """Median and best of isolated launches, and the sustained figure with its
    clock record and fraction of the sustained peak."""
    work, scale, unit = work_of(cfg)
    times = time_reps(torch, tpd, h, wl, reps)
    med, best = statistics.median(times), min(times)
    out = {"reps": {"count": reps, "median_ms": round(med, 5), "best_ms": round(best, 5),
                    "median": round(work / (med * 1e-3) / scale, 2), "best": round(work / (best * 1e-3) / scale, 2),
                    "unit": unit, "how": "isolated launches, CUDA events around each, inputs not in L2"}}
    ms, n, secs, clocks = time_sustained(torch, tpd, h, wl, avg_ms, seconds, gpu_index)
    v = work / (ms * 1e-3) / scale
    if cfg.name == "decode":
        peak, pkey = peaks["hbm_gbs"], "hbm_gbs"
    else:
        peak, pkey = peaks["bf16_tflops_sustained"], "bf16_tflops_sustained"
    out["sustained"] = {"value": round(v, 2), "unit": unit, "ms_per_launch": round(ms, 5), "launches": n,
                        "seconds": round(secs, 3), "peak": peak, "peak_key": pkey, "frac": round(v / peak, 4),
                        "clocks": clocks,
                        "how": "a CUDA graph of back-to-back launches replayed for at least "
                               f"{seconds:.0f} s between CUDA events, rotating inputs larger than L2"}
    return out


def theoretical_peak(torch, local, clocks):
    """SMs x SM clock x the measured per-SM tensor rate, at the maximum clock
    and at the median clock sampled under load."""
    sms = torch.cuda.get_device_properties(local).multi_processor_count
    mx = (clocks or {}).get("sm_max_mhz") or 2070.0
    med = (clocks or {}).get("sm_mhz") or mx
    f = lambda mhz: round(sms * mhz * 1e6 * MMA_FLOP_PER_SM_CYCLE / 1e12, 1)
    return {"value": f(mx), "unit": "TFLOP/s", "sms": sms, "sm_mhz": mx, "at_median_clock": f(med),
            "median_sm_mhz": med, "flop_per_sm_cycle": MMA_FLOP_PER_SM_CYCLE,
            "how": "SMs x SM clock x dense bf16 flop per SM per cycle, the last measured with a standalone "
                   "tcgen05.mma loop (256 x 256 x 64 per CTA pair in 512 cycles)"}


def time_e2e(torch, tpd, h, wl, steps):
    """End to end through the public API: per step, copy A, B (and C) from
    pinned host memory, run gemm_run, copy D back to pinned host memory.

    Pipelined as a serving loop would run it: host-to-device copies on one
    stream, gemm_run on a second, device-to-host copies on a third, two device
    buffer sets used in turn, events ordering every reuse (step i's inputs go
    up while step i-1 computes and step i-2's result comes down). Every step
    still copies all of its inputs in and its result out inside the timed
    region. Returns (pipelined ms per step, serial ms per step, bytes in, bytes out)."""
    sets = wl.sets[:2]
    pins_d = [wl.pin["D"], torch.empty_like(wl.pin["D"]).pin_memory()]
    s_in, s_gemm, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    in_done = [ev(), ev()]
    gemm_done = [ev(), ev()]
    out_done = [ev(), ev()]
    used = [False, False]

    def step(i):
        k = i % 2
        s = sets[k]
        with torch.cuda.stream(s_in):
            if used[k]:
                s_in.wait_event(gemm_done[k])  # the set's A, B, C have been read
            s["A"].copy_(wl.pin["A"], non_blocking=True)
            s["B"].copy_(wl.pin["B"], non_blocking=True)
            if s["C"] is not None:
                s["C"].copy_(wl.pin["C"], non_blocking=True)
            in_done[k].record(s_in)
        s_gemm.wait_event(in_done[k])
        if used[k]:
            s_gemm.wait_event(out_done[k])  # the set's D has been copied out
        st = wl.run(tpd, h, k, s_gemm.cuda_stream)
        if st != 0:
            raise RuntimeError(tpd.gemm_status_string(st))
        gemm_done[k].record(s_gemm)
        with torch.cuda.stream(s_out):
            s_out.wait_event(gemm_done[k])
            pins_d[k].copy_(s["D"], non_blocking=True)
            out_done[k].record(s_out)
        used[k] = True

    for i in range(4):
        step(i)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(s_in)
    for i in range(steps):
        step(i)
    t1.record(s_out)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / steps

    # the same steps one after another on one stream, for context
    stream = torch.cuda.current_stream()
    s = sets[0]
    torch.cuda.synchronize()
    u0 = torch.cuda.Event(enable_timing=True)
    u1 = torch.cuda.Event(enable_timing=True)
    u0.record(stream)
    for _ in range(steps):
        s["A"].copy_(wl.pin["A"], non_blocking=True)
        s["B"].copy_(wl.pin["B"], non_blocking=True)
        if s["C"] is not None:
            s["C"].copy_(wl.pin["C"], non_blocking=True)
        if wl.run(tpd, h, 0, stream.cuda_stream) != 0:
            raise RuntimeError("gemm_run failed")
        pins_d[0].copy_(s["D"], non_blocking=True)
    u1.record(stream)
    torch.cuda.synchronize()
    serial_ms = u0.elapsed_time(u1) / steps
    return ms, serial_ms, wl.bytes_A + wl.bytes_B + wl.bytes_C, wl.bytes_D


def chunk_tradeoff(torch, tpd, h, M=1024, N=8192, K=3584, reps=30):
    """The chunk-size tradeoff of the tensor-parallel overlay loop on this GPU:
    gemm_run_chunked on one shard of an MLP down-projection (1024 tokens,
    hidden 8192, K = 28672 / 8), 1/2/4/8 chunks. Reports the median total time
    and the time until chunk 0's rows are done (when a collective could start).
    A device sleep ahead of the timed region keeps the GPU busy while the host
    issues every chunk, so the times are the GPU's, not the launch latency's."""
    g = torch.Generator().manual_seed(9)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16).cuda()
    B = (torch.randn(K, N, generator=g) * 0.02).to(torch.bfloat16).cuda()
    D = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()
    out = {}
    for chunks in (1, 2, 4, 8):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(chunks)]
        for e in evs:
            e.record(stream)
        torch.cuda.synchronize()
        totals, firsts = [], []
        for r in range(reps + 3):
            t0 = torch.cuda.Event(enable_timing=True)
            torch.cuda._sleep(400_000)  # ~0.2 ms: longer than issuing 8 chunks from the host
            t0.record(stream)
            st = tpd.gemm_run_chunked(h, chunks, M, N, K, A.data_ptr(), K, B.data_ptr(), N, None, N, D.data_ptr(),
                                      N, 1.0, 0.0, 0, [e.cuda_event for e in evs], stream.cuda_stream)
            if st != 0:
                raise RuntimeError(tpd.gemm_status_string(st))
            torch.cuda.synchronize()
            if r >= 3:
                totals.append(t0.elapsed_time(evs[-1]))
                firsts.append(t0.elapsed_time(evs[0]))
        tot = statistics.median(totals)
        out[str(chunks)] = {"total_ms": round(tot, 4), "first_chunk_ms": round(statistics.median(firsts), 4),
                            "tflops": round(2 * M * N * K / (tot * 1e-3) / 1e12, 1)}
    return {"unit": "ms", "config": {"workload": f"gemm_run_chunked, M={M} N={N} K={K} bf16, launches queued behind a "
                                                 "device sleep, median of 30"}, "chunks": out}


def roofline_entry(cfg, kernel, avg_ms, peaks, peak_src):
    if cfg.name == "decode":
        b_bytes = cfg.K * cfg.N * 2
        achieved = b_bytes / (avg_ms * 1e-3) / 1e9
        peak = peaks["hbm_gbs"]
        unit, bound = "GB/s", "hbm"
    else:
        achieved = cfg.flops / (avg_ms * 1e-3) / 1e12
        peak = peaks["bf16_tflops"]
        unit, bound = "TFLOP/s", "tensor"
    return {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
            "frac": round(achieved / peak, 4), "peak_source": f"{peak_src} (MEASURED_PEAKS.json burst)"
            if peak_src == "measured" else "fallback", "peak_kind": "burst: the timed region is short",
            "traffic": profile_traffic(kernel, cfg.name), "kernel": KERNEL_NAMES[kernel]}


def config_entry(cfg, wl, nsets):
    return {"workload": f"{cfg.name}: {cfg.description}", "M": cfg.M, "N": cfg.N, "K": cfg.K,
            "alpha": cfg.alpha, "beta": cfg.beta, "out_dtype": cfg.out_dtype,
            "l2": f"inputs larger than L2: {nsets} rotating device copies of A,B(,C),D, one per launch in turn",
            "parallelism": "replicas (independent GEMM per GPU)"}


def cpu_baseline(cfg, budget_s, inputs=None, threads=None):
    """The oracle as it stands, on a bounded row sample of the same workload
    (all rows when they fit the budget), on `threads` host threads (default:
    every core this process may use)."""
    import oracle
    from workloads import make_inputs, sample_rows
    A, B, C = inputs if inputs is not None else make_inputs(cfg)
    if threads is None:
        threads = len(os.sched_getaffinity(0))
    probe = sample_rows(cfg.M, max(1, min(cfg.M, threads)), seed=7)
    t0 = time.perf_counter()
    oracle.gemm_rows(A, B, C, cfg.alpha, cfg.beta, 1 if cfg.out_dtype == "f32" else 0, rows=probe,
                     nthreads=threads)
    per_row = (time.perf_counter() - t0) / len(probe)
    nrows = int(max(len(probe), min(cfg.M, budget_s / max(per_row, 1e-9))))
    rows = sample_rows(cfg.M, nrows, seed=11)
    t0 = time.perf_counter()
    oracle.gemm_rows(A, B, C, cfg.alpha, cfg.beta, 1 if cfg.out_dtype == "f32" else 0, rows=rows,
                     nthreads=threads)
    dt = time.perf_counter() - t0
    flops = 2.0 * len(rows) * cfg.N * cfg.K
    if cfg.name == "decode":
        value, unit = len(rows) / cfg.M * cfg.K * cfg.N * 2 / dt / 1e9, "GB/s"
    else:
        value, unit = flops / dt / 1e12, "TFLOP/s"
    return {"value": value, "unit": unit, "cores": threads, "kind": "oracle",
            "sample": f"{len(rows)} of {cfg.M} rows of {cfg.name} (all N columns, full K), "
                      f"{dt:.1f} s, fp64 C oracle, {threads} threads"}


def run_ours(args):
    import torch
    import torch.distributed as dist
    import tile_partitioned_dense_gb300 as tpd
    from workloads import CONFIGS

    world, rank, local = dist_env()
    if world != args.gpus:
        if world > 1 or args.gpus > 1:
            raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE={world}; launch N>1 with torchrun")
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if world > 1:
            dist.barrier()

    peaks, peak_src = load_peaks()
    props = torch.cuda.get_device_properties(local)
    l2 = int(getattr(props, "L2_cache_size", 0) or 129 * 2 ** 20)
    h = tpd.gemm_create(local)
    # Workspace for the K split of the CTA-pair kernel's last partial round. Every
    # GEMM below runs on one stream at a time (the e2e loop keeps them on one),
    # as a handle with a workspace requires.
    ws_bytes = tpd.gemm_workspace_size(h)
    ws_buf = torch.empty(ws_bytes + 256, dtype=torch.uint8, device=f"cuda:{local}")
    st = tpd.gemm_set_workspace(h, (ws_buf.data_ptr() + 255) // 256 * 256, ws_bytes,
                                torch.cuda.current_stream().cuda_stream)
    if st != 0:
        raise RuntimeError("gemm_set_workspace: " + tpd.gemm_status_string(st))

    cfg = CONFIGS[args.workload]
    wl = Workload(cfg, torch, l2, pinned=not args.no_e2e)
    plan = tpd.gemm_query_plan(h, cfg.M, cfg.N, cfg.K, wl.out_code)
    plan["tail_ksplit"] = tpd.gemm_plan_tail_ksplit(h, cfg.M, cfg.N, cfg.K, wl.out_code)
    kernel = "stream" if plan["variant"] == tpd.VARIANT_STREAM else "tiled"

    sampler = ClockSampler(local)
    sampler.start()
    span, eager = time_launches(torch, tpd, h, wl, args.steps, args.warmup, barrier)
    clocks = sampler.stop()

    # max over ranks of the timed-region time
    span_max, eager_max = max_over_ranks([span, eager], world, device="cuda")
    avg_max = span_max / args.steps  # average launch duration over the timed region
    head_extra = {}
    if not args.no_sustained:
        head_extra = measure_extra(torch, tpd, h, wl, cfg, avg_max, peaks, local)
    if cfg.name == "decode":
        unit = "GB/s"
        value = job_throughput(world, args.steps, cfg.K * cfg.N * 2, span_max, 1e9)
    else:
        unit = "TFLOP/s"
        value = job_throughput(world, args.steps, cfg.flops, span_max, 1e12)

    e2e = None
    if not args.no_e2e:
        e2e_steps = max(3, min(args.steps, 20))
        ms, serial_ms, bi, bo = time_e2e(torch, tpd, h, wl, e2e_steps)
        ms = max_over_ranks([ms], world, device="cuda")[0]
        ev = job_throughput(world, 1, cfg.K * cfg.N * 2, ms, 1e9) if cfg.name == "decode" else \
            job_throughput(world, 1, cfg.flops, ms, 1e12)
        serial_ms = max_over_ranks([serial_ms], world, device="cuda")[0]
        e2e = {"value": round(ev, 3), "unit": unit, "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
               "ms_per_step": round(ms, 4), "steps": e2e_steps, "serial_ms_per_step": round(serial_ms, 4),
               "path": "every step: pinned host -> device copies of A, B (C), gemm_run (C ABI), device -> pinned "
                       "host copy of D; copies in, GEMMs and copies out on three streams over two buffer sets, "
                       "ordered by events (serial_ms_per_step: the same steps on one stream)"}

    per_config = {}
    launches = args.steps
    torch_rows = {}
    if args.only_rows:
        args.only_mx = True
    bf16_extra = not args.no_extra and not args.only_mx
    if bf16_extra:
        if cfg.name != "tiny":
            # the same number of back-to-back launches as the headline's timed region,
            # so that both run as long under the power cap
            torch_rows[cfg.name] = torch_matmul_entry(torch, tpd, h, wl, min(args.steps, 4000), avg_max, barrier)
        for name in ["qkv", "mlp_down", "decode", "square", "tiny"]:
            if name == cfg.name:
                continue
            c2 = CONFIGS[name]
            w2 = Workload(c2, torch, l2, pinned=False)
            p2 = tpd.gemm_query_plan(h, c2.M, c2.N, c2.K, w2.out_code)
            p2["tail_ksplit"] = tpd.gemm_plan_tail_ksplit(h, c2.M, c2.N, c2.K, w2.out_code)
            k2 = "stream" if p2["variant"] == tpd.VARIANT_STREAM else "tiled"
            steps2 = max(20, min(400, int(0.4 / (c2.flops / 1.5e15 if name != "decode" else 40e-6) + 1)))
            span2, eager2 = time_launches(torch, tpd, h, w2, steps2, 10, barrier)
            avg2 = span2 / steps2
            if name == "decode":
                v2 = c2.K * c2.N * 2 / (span2 / steps2 * 1e-3) / 1e9
                u2 = "GB/s"
            else:
                v2 = c2.flops / (span2 / steps2 * 1e-3) / 1e12
                u2 = "TFLOP/s"
            per_config[name] = {"value": round(v2, 2), "unit": u2, "ms_per_step": round(span2 / steps2, 5),
                                "eager_ms_per_step": round(eager2 / steps2, 5),
                                "steps": steps2, "roofline": roofline_entry(c2, k2, avg2, peaks, peak_src),
                                "config": config_entry(c2, w2, w2.nsets), "plan": p2}
            if not args.no_sustained and name != "tiny":
                per_config[name].update(measure_extra(torch, tpd, h, w2, c2, avg2, peaks, local))
            if name != "tiny":  # torch.mm has no bf16 x bf16 -> fp32 output form
                torch_rows[name] = torch_matmul_entry(torch, tpd, h, w2, steps2, avg2, barrier)
            launches += steps2
            if rank == 0 and world == 1 and not args.no_cpu_baseline:
                per_config[name]["cpu_baseline"] = cpu_baseline(c2, 3.0, inputs=(w2.host["A"], w2.host["B"],
                                                                                 w2.host["C"]))
                if name in ("tiny", "decode"):
                    per_config[name]["cpu_baseline_1core"] = cpu_baseline(c2, 60.0, inputs=(
                        w2.host["A"], w2.host["B"], w2.host["C"]), threads=1)
            del w2
            torch.cuda.empty_cache()

    if bf16_extra:
        # fused epilogue (bias + sigmoid + aux multiply) on the QKV shape, against the
        # plain GEMM followed by the same element-wise work in torch
        c2 = CONFIGS["qkv"]
        out = {}
        for fused in (True, False):
            w2 = FusedWorkload(c2, torch, l2, tpd.ACT_SIGMOID, fused)
            span2, _ = time_launches(torch, tpd, h, w2, 200, 5, barrier)
            out[fused] = span2 / 200
            del w2
            torch.cuda.empty_cache()
        per_config["qkv_bias_sigmoid_aux"] = {
            "value": round(c2.flops / (out[True] * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "ms_per_step": round(out[True], 5), "unfused_ms_per_step": round(out[False], 5),
            "speedup_vs_unfused": round(out[False] / out[True], 3),
            "config": {"workload": "qkv shape, D = sigmoid(A*B + bias) * aux, bf16; unfused = gemm_run then "
                                   "torch sigmoid(D + bias) * aux in the same graph", "M": c2.M, "N": c2.N, "K": c2.K}}
        launches += 200
        # batched and grouped GEMM: 8 x 2048^3 and 8 experts of uneven size (8192 rows, 4096 x 4096)
        peak = peaks["bf16_tflops"]
        moe_rows = [512, 1024, 768, 2048, 256, 1536, 1024, 1024]
        for name, wl2, desc in [
                ("bmm_8x2048", MultiWorkload(torch, l2, "bmm", 2048, 2048, 2048, 8), "batched GEMM, 8 x 2048x2048x2048, bf16"),
                ("grouped_moe8", MultiWorkload(torch, l2, "grouped", 0, 4096, 4096, 8, moe_rows),
                 f"grouped GEMM, 8 experts with rows {moe_rows} (8192 total), N = K = 4096, bf16")]:
            span2, eager2 = time_launches(torch, tpd, h, wl2, 100, 5, barrier)
            ms2 = span2 / 100
            v2 = wl2.flops / (ms2 * 1e-3) / 1e12
            per_config[name] = {"value": round(v2, 2), "unit": "TFLOP/s", "ms_per_step": round(ms2, 5),
                                "eager_ms_per_step": round(eager2 / 100, 5),
                                "roofline": {"bound": "tensor", "achieved": round(v2, 2), "peak": peak,
                                             "unit": "TFLOP/s", "frac": round(v2 / peak, 4)},
                                "config": {"workload": desc}}
            launches += 100
            del wl2
            torch.cuda.empty_cache()

    if not args.no_extra:
        bs = mx_entries(torch, tpd, h, l2, peaks, local, barrier, rank, world, args)
        bs.update(fp4_entries(torch, tpd, h, l2, peaks, local, barrier, rank, world, args))
        per_config.update(bs)
        launches += sum(e["steps"] for e in bs.values())

    if bf16_extra:
        per_config["tp_overlay_chunks"] = chunk_tradeoff(torch, tpd, h)
        per_config["torch_matmul"] = {
            "note": "torch.matmul / addmm (cuBLAS) on the same shapes and rotating buffers, timed the same way; "
                    "a comparison row, not this library's path",
            "rows": torch_rows}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(cfg, args.cpu_seconds, inputs=(wl.host["A"], wl.host["B"], wl.host["C"]))

    if rank == 0:
        line = {
            "metric": METRIC,
            "value": round(value, 3),
            "unit": unit,
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(span_max / args.steps, 5),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic (seeded: A,B ~ N(0,1) for square; see workloads.py)",
            "config": config_entry(cfg, wl, wl.nsets),
            "impl": "ours",
            "roofline": roofline_entry(cfg, kernel, avg_max, peaks, peak_src),
            "reps": head_extra.get("reps"),
            "sustained": head_extra.get("sustained"),
            "theoretical_peak": theoretical_peak(torch, local, (head_extra.get("sustained") or {}).get("clocks")
                                                 or clocks) if cfg.name != "decode" else None,
            "cpu_baseline": cpu,
            "e2e": e2e,
            # our kernel launches inside the headline timed region (one per step),
            # and inside every timed region of this run (per_config included)
            "gpu_launches": args.steps,
            "gpu_launches_all_timed_regions": launches,
            "clocks": clocks,
            "plan": plan,
            "kernel_avg_ms": round(avg_max, 5),
            "eager_ms_per_step": round(eager_max / args.steps, 5),
            "timing": "K launches captured once in a CUDA graph, replayed in the timed region; "
                      "CUDA events on the launching stream; eager_ms_per_step: the same launches "
                      "issued one by one from Python",
            "per_config": per_config,
        }
        print(json.dumps(line), flush=True)
    tpd.gemm_destroy(h)
    if world > 1:
        dist.destroy_process_group()


# ----------------------------------------------------------------------------- reference arm

def run_reference(args):
    """The oracle (the plain fp64 CPU definition) timed as the reference arm:
    each step computes a bounded row sample of the same workload."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    from workloads import CONFIGS, make_inputs, sample_rows
    cfg = CONFIGS[args.workload]
    A, B, C = make_inputs(cfg)
    threads = len(os.sched_getaffinity(0))
    out = 1 if cfg.out_dtype == "f32" else 0
    probe = sample_rows(cfg.M, max(1, min(cfg.M, threads)), seed=7)
    t0 = time.perf_counter()
    oracle.gemm_rows(A, B, C, cfg.alpha, cfg.beta, out, rows=probe, nthreads=threads)
    per_row = (time.perf_counter() - t0) / len(probe)
    # keep the whole --steps K --warmup W run within about two minutes
    per_step_s = max(0.2, min(3.0, 120.0 / max(1, args.steps + args.warmup)))
    nrows = int(max(1, min(cfg.M, per_step_s / max(per_row, 1e-9))))
    times = []
    for i in range(args.warmup + args.steps):
        rows = sample_rows(cfg.M, nrows, seed=100 + i)
        t0 = time.perf_counter()
        oracle.gemm_rows(A, B, C, cfg.alpha, cfg.beta, out, rows=rows, nthreads=threads)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    ms = 1e3 * sum(times) / len(times)
    if cfg.name == "decode":
        value, unit = nrows / cfg.M * cfg.K * cfg.N * 2 / (ms * 1e-3) / 1e9, "GB/s"
    else:
        value, unit = 2.0 * nrows * cfg.N * cfg.K / (ms * 1e-3) / 1e12, "TFLOP/s"
    sample = (f"{nrows} of {cfg.M} rows of {cfg.name} per step (all N columns, full K), "
              f"fp64 C oracle, {threads} threads")
    line = {"metric": METRIC, "value": value, "unit": unit, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded, workloads.py)",
            "config": {"workload": f"{cfg.name}: {cfg.description}", "M": cfg.M, "N": cfg.N, "K": cfg.K},
            "impl": "reference",
            "cpu_baseline": {"value": value, "unit": unit, "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
