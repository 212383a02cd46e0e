#!/usr/bin/env python3
"""Benchmark of the differential-attention forward on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
lambda from its four parameter vectors (diffattn_lambda) followed by the
forward O = (A1 - lambda A2) V (diffattn_fwd, reading lambda on the device).
Default workload: B=2, H=16, T=8192, D=64, V width 128, bf16, causal.

Prints one JSON line (rank 0).  Timing: W untimed warm-up steps, then K
timed steps; each step is bracketed by CUDA events on the launch stream, and
the L2 cache is flushed between steps outside the events (a 256 MiB write,
then a 256 MiB read so that the write's dirty lines reach DRAM before the
step rather than during it; --l2-flush write keeps the write alone).
`value` is the algorithmic TFLOP/s of the whole job (unmasked pairs x 12 D,
all ranks).  `e2e` repeats the measurement with inputs copied from pinned
host memory and the output copied back inside the timed region.

--impl reference times the float64 CPU oracle (the only reference
implementation of this operation) on a bounded sample of the same workload.

Multi-GPU: replicas only (each rank runs its own copy of the workload; the
forward has no exchange step), so scaling is weak and value sums the ranks'
work over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "diffattn_fwd TFLOP/s and % of GB300 bf16 tensor peak (B=2,H=16,T=8192,D=64 causal)"
UNIT = "TFLOP/s"
L2_BYTES = 129 * 1000 * 1000
FLUSH_BYTES = 256 * 1024 * 1024


class L2Flush:
    """The L2 flush between timed steps (outside the events): a write of a
    buffer larger than L2 evicts the previous step's lines.  With kind
    "write-read" a read of a second such buffer follows, so that the dirty
    lines the write left are written back to DRAM before the step, not during
    it, and the step starts with L2 holding clean lines of neither its inputs
    nor its outputs."""

    def __init__(self, dev, kind: str):
        import torch
        self.kind = kind
        self.w = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.r = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=dev) if kind == "write-read" else None

    def zero_(self):
        self.w.zero_()
        if self.r is not None:
            self.r.sum()

    def describe(self) -> str:
        return L2Flush.describe_kind(self.kind)

    @staticmethod
    def describe_kind(kind: str) -> str:
        if kind == "write":
            return "flushed between steps (256 MiB write outside the timed events)"
        return ("flushed between steps (256 MiB write, then a 256 MiB read that cleans the "
                "written lines, outside the timed events)")
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "diffattn_fwd_tc_b2h16t8192.md")
KERNEL_SOURCES = ["fwd_tc.cu", "ptx.cuh", "kernels.h", "api.cu"]   # the kernel and its launch plan
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# --------------------------------------------------------------------------
# host logic shared by every rank count (tested on CPU with gloo)
# --------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return world, rank, local


def check_world(gpus: int, world: int) -> None:
    """--gpus N must match the number of ranks the launcher started: one
    process per GPU.  Without a launcher (WORLD_SIZE unset) only N = 1 runs;
    running one replica for N > 1 would report work N GPUs never did."""
    if gpus < 1:
        raise ValueError(f"--gpus must be >= 1, got {gpus}")
    if world == 1 and gpus > 1:
        raise ValueError(f"--gpus {gpus} needs {gpus} processes, one per GPU: launch with "
                         f"python -m torch.distributed.run --nproc-per-node {gpus} "
                         f"--master-addr 127.0.0.1 bench.py --gpus {gpus} ...")
    if world > 1 and gpus != world:
        raise ValueError(f"--gpus {gpus} does not match the {world} ranks the launcher started")


# Dense bf16 tensor-core rate of one SM per clock (tcgen05 kind::f16 with fp32
# accumulation; a microbenchmark of back-to-back 128 x 256 x 16 products on
# this GPU measured 8184).  Times the SM count and the sampled SM clock it
# gives the tensor peak at the clock the kernel actually ran at.
BF16_FLOP_PER_CLK_PER_SM = 8192


def clock_peak(achieved_tflops: float, clocks, num_sms: int):
    """The kernel's fraction of the tensor peak at its own sampled SM clock."""
    if not clocks:
        return None
    mhz = clocks.get("sm_mhz_loaded") or clocks.get("sm_mhz")
    if not mhz:
        return None
    peak = num_sms * mhz * 1e6 * BF16_FLOP_PER_CLK_PER_SM / 1e12
    return {"sm_mhz": mhz, "sms": num_sms, "flop_per_clk_per_sm": BF16_FLOP_PER_CLK_PER_SM,
            "peak": peak, "frac": achieved_tflops / peak,
            "clock": "median SM clock of the samples under load (nvidia-smi, sampled, never set)"}


def reduce_max(value: float, world: int) -> float:
    """Max of a float over all ranks (identity for one rank)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def job_value(flops_per_step: float, steps: int, world: int, max_seconds: float) -> float:
    """Whole-job TFLOP/s: every rank's work over the slowest rank's time."""
    return flops_per_step * steps * world / max_seconds / 1e12


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "differential_attention_fwd_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source for this workload; else None."""
    try:
        text = open(PROFILE_SUMMARY).read()
    except OSError:
        return None
    m_hash = re.search(r"kernel_source_sha256:\s*([0-9a-f]+)", text)
    m_traffic = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    m_work = re.search(r"workload:\s*(\S+)", text)
    if not (m_hash and m_traffic and m_work):
        return None
    if m_hash.group(1) != kernel_source_hash() or m_work.group(1) != workload:
        return None
    return float(m_traffic.group(1))


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.out = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        return self.parse(out)

    @classmethod
    def parse(cls, text: str):
        """Median SM clock, max clock and the throttle reasons seen."""
        rows = []
        for line in text.splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) != len(cls.FIELDS):
                continue
            try:
                power = float(parts[2])
            except ValueError:
                power = float("nan")
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[4:], power))
            except ValueError:
                continue
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r, _ in rows for i, x in enumerate(r) if x.lower() == "active"})
        # samples under load: power above half of the highest power seen
        pmax = max((p for *_, p in rows if p == p), default=float("nan"))
        loaded = [s for s, _, _, p in rows if p == p and p >= 0.5 * pmax]
        return {"sm_mhz": statistics.median(s for s, _, _, _ in rows),
                "sm_mhz_loaded": statistics.median(loaded) if loaded else None,
                "samples_loaded": len(loaded), "power_w_max": pmax if pmax == pmax else None,
                "sm_max_mhz": max(m for _, m, _, _ in rows), "reasons": reasons, "samples": len(rows)}


# --------------------------------------------------------------------------
# CPU oracle timing (the cpu_baseline leg and the reference arm)
# --------------------------------------------------------------------------
def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n and n[0]:
            return int(n[0])
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return os.cpu_count() or 1


def oracle_rows_flops(rows, T, D, causal, Dv=None):
    """Algorithmic FLOPs of the given query rows: 4 D + 4 Dv per unmasked pair
    (12 D for the operation's own value width, Dv = 2D)."""
    pairs = sum((int(r) + 1) if causal else T for r in rows)
    return pairs * (4 * D + 4 * (2 * D if Dv is None else Dv))


def time_oracle(inp, w, lam, rows, head=(0, 0)):
    """Run the oracle on one head for `rows`; returns (seconds, flops)."""
    import oracle
    t0 = time.perf_counter()
    oracle.differential_attention(inp.q1, inp.k1, inp.q2, inp.k2, inp.v, lam, w.causal,
                                  rows=rows, heads=[head])
    return time.perf_counter() - t0, oracle_rows_flops(rows, w.T, w.D, w.causal, w.Dv)


def sample_rows(T, n, seed):
    """n query rows spread evenly over [0, T) (so causal row costs average
    out), shifted by a seed-dependent phase so that steps differ."""
    n = max(1, min(n, T))
    stride = T // n
    start = (seed * 7919) % stride if stride > 1 else 0
    return (start + np.arange(n, dtype=np.int64) * stride).clip(0, T - 1)


def cpu_baseline(inp, w, lam, budget_s=15.0):
    """Time the oracle, as it stands, on a bounded sample of the workload:
    whole heads (every query row) in (b, h) order until about budget_s of
    work is done, or a row sample of head (0, 0) if one head takes longer."""
    n0 = min(w.T, 256)
    t1, _ = time_oracle(inp, w, lam, sample_rows(w.T, n0, 0))
    per_row = max(t1 / n0, 1e-6)
    if per_row * w.T > budget_s:
        n = int(max(8, budget_s / per_row))
        secs, flops = time_oracle(inp, w, lam, sample_rows(w.T, n, 1))
        what = f"head (0,0), {n} query rows spread over T={w.T}"
    else:
        secs, flops, heads = 0.0, 0, 0
        all_rows = np.arange(w.T, dtype=np.int64)
        for b in range(w.B):
            for h in range(w.H):
                s, f = time_oracle(inp, w, lam, all_rows, head=(b, h))
                secs, flops, heads = secs + s, flops + f, heads + 1
                if secs >= budget_s:
                    break
            if secs >= budget_s:
                break
        what = f"{heads} whole heads of {w.B * w.H} (every query row, T={w.T})"
    return {"value": flops / secs / 1e12, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
            "sample": f"float64 NumPy oracle, {what} "
                      f"({'causal' if w.causal else 'full'} rows, {flops / 1e9:.2f} GFLOP "
                      f"algorithmic) in {secs:.1f} s"}


def run_reference(args, w, world, rank):
    if rank != 0:
        return None
    inp = W.draw(w)
    lam = lambda_for(w, inp)
    budget = 150.0 / max(1, args.steps + args.warmup)
    t1, _ = time_oracle(inp, w, lam, sample_rows(w.T, 4, 0))
    rows_per_step = int(max(1, min(w.T, budget / max(t1 / 4, 1e-5))))
    total_s = 0.0
    total_flops = 0
    for step in range(args.warmup + args.steps):
        rows = sample_rows(w.T, rows_per_step, step)
        s, f = time_oracle(inp, w, lam, rows)
        if step >= args.warmup:
            total_s += s
            total_flops += f
    value = total_flops / total_s / 1e12
    cores = blas_threads()
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_of(w, lam, args.l2_flush),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"each step: {rows_per_step} query rows of head (0,0) spread over "
                                   f"T={w.T}, float64 NumPy oracle on the host cores"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def lambda_for(w, inp) -> float:
    import oracle
    if w.lambdas:
        return float(w.lambdas[0])
    return float(np.float32(oracle.differential_lambda(inp.lq1, inp.lk1, inp.lq2, inp.lk2,
                                                       W.lambda_init_for(w))))


def config_of(w, lam, l2_flush: str = "write-read"):
    grouped = {"H_kv": w.Hk, "shared_keys": w.shared_keys} if (w.Hk != w.H or w.shared_keys) else {}
    return {"workload": w.name, "B": w.B, "H": w.H, **grouped, "T": w.T, "D": w.D, "Dv": w.Dv,
            "causal": w.causal, "lambda_init": W.lambda_init_for(w) if not w.lambdas else None,
            "lambda": lam, "gflop_per_step": w.flops / 1e9,
            "l2": f"{L2Flush.describe_kind(l2_flush)}; inputs {input_bytes(w) / 2**20:.0f} MiB",
            "parallelism": "replicas"}


def input_bytes(w):
    """Bytes of Q1, Q2 (H heads) and K1, K2, V (H_kv heads; one key tensor
    when the branches share it)."""
    el = 2 if w.dtype == "bf16" else 4
    k_tensors = 1 if w.shared_keys else 2
    return w.B * w.T * (w.H * 2 * w.D + w.Hk * (k_tensors * w.D + w.Dv)) * el


# --------------------------------------------------------------------------
# the GPU arm
# --------------------------------------------------------------------------
def run_ours(args, w, world, rank, local):
    import torch
    import differential_attention_fwd_gb300 as da
    from differential_attention_fwd_gb300 import _lib
    from differential_attention_fwd_gb300 import build as build_mod

    build_mod.build()
    lib = _lib.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32

    inp = W.draw(w)
    lam_vecs_host = [torch.from_numpy(x) for x in (inp.lq1, inp.lk1, inp.lq2, inp.lk2)]
    lam_init = W.lambda_init_for(w) if not w.lambdas else 0.0
    host = [torch.from_numpy(x).to(tdt) for x in (inp.q1, inp.k1, inp.q2, inp.k2, inp.v)]
    d_in = [h.to(dev) for h in host]
    if w.shared_keys:
        # one key tensor for both branches: the library sees the same pointer
        host[3], d_in[3] = host[1], d_in[1]
    d_lv = [v.to(dev) for v in lam_vecs_host]
    d_lam = torch.empty((), dtype=torch.float32, device=dev)
    d_out = torch.empty((w.B, w.H, w.T, w.Dv), dtype=tdt, device=dev)
    flush = L2Flush(dev, args.l2_flush)
    stream = torch.cuda.current_stream(dev)
    sh = ctypes.c_void_p(stream.cuda_stream)
    desc = da.make_desc(*d_in, d_out)
    ptr_in = [ctypes.c_void_p(t.data_ptr()) for t in d_in]
    ptr_lv = [ctypes.c_void_p(t.data_ptr()) for t in d_lv]
    p_lam, p_out = ctypes.c_void_p(d_lam.data_ptr()), ctypes.c_void_p(d_out.data_ptr())
    nlam = int(d_lv[0].numel())
    kernel = da.select_kernel(*d_in, out=d_out)
    ws = da.workspace_for(dev, stream)
    p_ws, ws_bytes = ctypes.c_void_p(ws.data_ptr()), ctypes.c_size_t(ws.numel() * 4)
    epi = None
    if args.norm != "none":
        # fused per-head norm with affine parameters, then x (1 - lambda_init)
        g = torch.Generator(device="cpu").manual_seed(11)
        nw = (1 + 0.1 * torch.randn(w.H, w.Dv, generator=g)).to(dev)
        nb = (0.1 * torch.randn(w.H, w.Dv, generator=g)).to(dev)
        epi = _lib.DiffattnEpilogue()
        epi.norm = {"rms": _lib.DIFFATTN_NORM_RMS, "group": _lib.DIFFATTN_NORM_GROUP}[args.norm]
        epi.eps, epi.weight, epi.bias = 1e-5, nw.data_ptr(), nb.data_ptr()
        epi.out_scale, epi.reserved = 1.0 - lam_init, 0
    p_epi = ctypes.byref(epi) if epi is not None else None

    def step():
        rc = lib.diffattn_lambda(*ptr_lv, nlam, ctypes.c_double(lam_init), p_lam, sh)
        if rc:
            raise _lib.DiffattnError(rc, "diffattn_lambda")

    def fwd():
        rc = lib.diffattn_fwd_ex(ctypes.byref(desc), *ptr_in, ctypes.c_float(0.0), p_lam,
                                 1 if w.causal else 0, p_epi, p_out, p_ws, ws_bytes, sh)
        if rc:
            raise _lib.DiffattnError(rc, "diffattn_fwd")

    if w.lambdas:   # lambda given directly: no lambda kernel in the step
        d_lam.fill_(float(w.lambdas[0]))
        launches_per_step = 1
    else:
        launches_per_step = 2

    for _ in range(args.warmup):
        flush.zero_()
        if launches_per_step == 2:
            step()
        fwd()
    torch.cuda.synchronize()
    if da.get_device_error() != 0:
        raise RuntimeError("a kernel wait ran out during warm-up")

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    sampler = ClockSampler(local) if (args.clocks and rank == 0) else None
    barrier(world)
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
        time.sleep(0.3)
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        if launches_per_step == 2:
            step()
        ev[i][1].record(stream)
        fwd()
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    barrier(world)
    step_ms = [a.elapsed_time(c) for a, _, c in ev]
    fwd_ms = [b.elapsed_time(c) for _, b, c in ev]
    total_s = sum(step_ms) / 1e3
    max_s = reduce_max(total_s, world)
    if da.get_device_error() != 0:
        raise RuntimeError("a kernel wait ran out during the timed steps")

    value = job_value(w.flops, args.steps, world, max_s)
    peaks, peak_src = load_peaks()
    fwd_avg_s = statistics.mean(fwd_ms) / 1e3
    achieved = w.flops / fwd_avg_s / 1e12
    peak = float(peaks["bf16_tflops"])
    traffic = profiled_traffic(w.name)
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": traffic,
                "peak_source": f"{peak_src} bf16_tflops (burst; kernel timed alone)",
                "frac_of_sustained": achieved / float(peaks["bf16_tflops_sustained"]),
                "fwd_ms_median": statistics.median(fwd_ms), "fwd_ms_min": min(fwd_ms),
                "fwd_ms_max": max(fwd_ms)}

    roofline["at_sampled_clock"] = clock_peak(
        achieved, clocks, torch.cuda.get_device_properties(dev).multi_processor_count)

    e2e = None
    if args.e2e:
        e2e = run_e2e(args, w, lib, da, _lib, host, lam_vecs_host, lam_init, d_in, d_lv, d_lam,
                      d_out, desc, launches_per_step, flush, stream, world, ws)

    result = {
        "metric": METRIC if w.name == W.HEADLINE else
                  f"diffattn_fwd TFLOP/s and % of GB300 bf16 tensor peak ({w.name}: B={w.B},H={w.H},"
                  f"H_kv={w.Hk},T={w.T},D={w.D},Dv={w.Dv} {'causal' if w.causal else 'full'})",
        "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * max_s / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {**config_of(w, float(d_lam.item()), args.l2_flush),
                   **({"epilogue": f"{args.norm} norm + affine + x(1-lambda_init)"} if args.norm != "none" else {})},
        "pct_of_peak": 100.0 * value / world / peak,
        "roofline": roofline, "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "kernel": {1: "tcgen05", 2: "simt"}.get(kernel, str(kernel)),
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and args.cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(inp, w, float(d_lam.item()), args.cpu_budget)
    return result


def run_e2e(args, w, lib, da, _lib, host, lam_vecs_host, lam_init, d_in, d_lv, d_lam, d_out,
            desc, launches_per_step, flush, stream, world, ws):
    """Same metric, inputs from pinned host memory, output back to the host."""
    import torch
    # one copy per distinct device input (a shared key tensor is copied once)
    uniq = []
    for d, h in zip(d_in, host):
        if all(d is not u for u, _ in uniq):
            uniq.append((d, h.pin_memory()))
    pin_lv = [v.pin_memory() for v in lam_vecs_host]
    out_host = torch.empty(d_out.shape, dtype=d_out.dtype).pin_memory()
    steps = max(1, min(args.steps, args.e2e_steps))
    h2d = sum(h.numel() * h.element_size() for _, h in uniq)
    if launches_per_step == 2:
        h2d += sum(t.numel() * t.element_size() for t in pin_lv)
    d2h = out_host.numel() * out_host.element_size()

    # host inputs in the call's order (a shared key tensor is one host buffer)
    pin_of = {id(d): h for d, h in uniq}
    host_ptrs = [ctypes.c_void_p(pin_of[id(d)].data_ptr()) for d in d_in]
    dev_ptrs = [ctypes.c_void_p(t.data_ptr()) for t in d_in]

    def one():
        if launches_per_step == 2:
            for d, h in zip(d_lv, pin_lv):
                d.copy_(h, non_blocking=True)
            lib.diffattn_lambda(*[ctypes.c_void_p(t.data_ptr()) for t in d_lv], int(d_lv[0].numel()),
                                ctypes.c_double(lam_init), ctypes.c_void_p(d_lam.data_ptr()),
                                ctypes.c_void_p(stream.cuda_stream))
        # the library's host-buffer call: copies in, forward, copy out, pipelined
        rc = lib.diffattn_fwd_host(ctypes.byref(desc), *host_ptrs, ctypes.c_float(0.0),
                                   ctypes.c_void_p(d_lam.data_ptr()), 1 if w.causal else 0,
                                   ctypes.c_void_p(out_host.data_ptr()), *dev_ptrs,
                                   ctypes.c_void_p(d_out.data_ptr()), ctypes.c_void_p(ws.data_ptr()),
                                   ctypes.c_size_t(ws.numel() * 4), ctypes.c_void_p(stream.cuda_stream))
        if rc:
            raise _lib.DiffattnError(rc, "diffattn_fwd_host")

    for _ in range(3):
        one()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    barrier(world)
    for a, b in evs:
        flush.zero_()
        a.record(stream)
        one()
        b.record(stream)
    torch.cuda.synchronize()
    secs = sum(a.elapsed_time(b) for a, b in evs) / 1e3
    max_s = reduce_max(secs, world)
    return {"value": job_value(w.flops, steps, world, max_s), "unit": UNIT,
            "call": "diffattn_fwd_host: the inputs copied in and O copied out by the library, "
                    "pipelined over chunks of heads with the forward",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": steps,
            "ms_per_step": 1e3 * max_s / steps}


BWD_FLOPS_PER_PAIR_PER_D = 20   # recompute S_1, S_2 (4D), dP (4D), dV (4D), dQ_1, dQ_2 (4D), dK_1, dK_2 (4D)


def bwd_flops(w) -> int:
    """Algorithmic backward FLOPs: 20 D per unmasked (query, key) pair."""
    return w.B * w.H * w.pairs_per_head * BWD_FLOPS_PER_PAIR_PER_D * w.D


def cpu_baseline_backward(inp, dout, w, lam, budget_s=15.0):
    """The oracle's backward, as it stands, on whole heads until ~budget_s."""
    import oracle
    from oracle import diffattn_oracle as O
    g = w.H // w.Hk
    secs, heads = 0.0, 0
    for b in range(w.B):
        for h in range(w.H):
            hk = h // g
            t0 = time.perf_counter()
            O._head_backward(*(np.asarray(x, dtype=np.float64) for x in
                               (inp.q1[b, h], inp.k1[b, hk], inp.q2[b, h], inp.k2[b, hk],
                                inp.v[b, hk], dout[b, h])), lam, w.causal)
            secs += time.perf_counter() - t0
            heads += 1
            if secs >= budget_s:
                break
        if secs >= budget_s:
            break
    flops = heads * w.pairs_per_head * BWD_FLOPS_PER_PAIR_PER_D * w.D
    return {"value": flops / secs / 1e12, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
            "sample": f"float64 NumPy oracle backward, {heads} whole heads of {w.B * w.H} "
                      f"(T={w.T}, {flops / 1e9:.1f} GFLOP algorithmic) in {secs:.1f} s"}


def run_backward(args, w, world, rank, local):
    """The backward (diffattn_bwd): row statistics, dQ, dK/dV and dlambda."""
    import torch
    import differential_attention_fwd_gb300 as da
    from differential_attention_fwd_gb300 import _lib
    from differential_attention_fwd_gb300 import build as build_mod

    build_mod.build()
    lib = _lib.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    inp = W.draw(w)
    rng = np.random.Generator(np.random.PCG64(w.seed + 1000))
    dout = rng.standard_normal((w.B, w.H, w.T, w.Dv), dtype=np.float32)
    if w.dtype == "bf16":
        dout = W.round_to_bf16(dout)
    lam = lambda_for(w, inp)
    host = [torch.from_numpy(x).to(tdt) for x in (inp.q1, inp.k1, inp.q2, inp.k2, inp.v, dout)]
    d_in = [h.to(dev) for h in host]
    if w.shared_keys:
        host[3], d_in[3] = host[1], d_in[1]
    grads = [torch.empty(t.shape, dtype=tdt, device=dev) for t in d_in[:5]]
    d_lam = torch.empty((), dtype=torch.float32, device=dev)
    flush = L2Flush(dev, args.l2_flush)
    stream = torch.cuda.current_stream(dev)
    desc = da.make_desc(*d_in[:5], d_in[5])
    need = int(lib.diffattn_bwd_workspace_bytes(ctypes.byref(desc)))
    ws = torch.empty(need // 4 + 4, dtype=torch.float32, device=dev)
    ptrs = [ctypes.c_void_p(t.data_ptr()) for t in d_in]
    gptrs = [ctypes.c_void_p(t.data_ptr()) for t in grads]
    # the forward of the training step (outside the timed region) keeps O, A_2 V
    # and the log-sum-exp; the backward starts from them unless asked to recompute
    saved = None
    if not args.bwd_recompute:
        saved = da.differential_attention_train(*d_in[:5], lam, causal=w.causal)
        sptrs = [ctypes.c_void_p(t.data_ptr()) for t in saved]

    def step():
        head = (ctypes.byref(desc), *ptrs[:5], ctypes.c_float(lam), None, 1 if w.causal else 0)
        tail = (ptrs[5], *gptrs, ctypes.c_void_p(d_lam.data_ptr()), ctypes.c_void_p(ws.data_ptr()),
                ctypes.c_size_t(need), ctypes.c_void_p(stream.cuda_stream))
        if saved is not None:
            rc = lib.diffattn_bwd_saved(*head, *sptrs, *tail)
        else:
            rc = lib.diffattn_bwd(*head, *tail)
        if rc:
            raise _lib.DiffattnError(rc, "diffattn_bwd")

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    if da.get_device_error() != 0:
        raise RuntimeError("a kernel wait ran out during warm-up")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    sampler = ClockSampler(local) if (args.clocks and rank == 0) else None
    barrier(world)
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
        time.sleep(0.3)
    for a, b in ev:
        flush.zero_()
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    barrier(world)
    ms = [a.elapsed_time(b) for a, b in ev]
    max_s = reduce_max(sum(ms) / 1e3, world)
    if da.get_device_error() != 0:
        raise RuntimeError("a kernel wait ran out during the timed steps")
    flops = bwd_flops(w)
    peaks, src = load_peaks()
    avg_s = statistics.mean(ms) / 1e3
    achieved = flops / avg_s / 1e12
    peak = float(peaks["bf16_tflops"])

    e2e = None
    if args.e2e:
        pin = []
        for d, h in zip(d_in, host):
            if all(d is not u for u, _ in pin):
                pin.append((d, h.pin_memory()))
        out_host = [torch.empty(g.shape, dtype=g.dtype).pin_memory() for g in grads]
        lam_host = torch.empty((), dtype=torch.float32).pin_memory()
        h2d = sum(h.numel() * h.element_size() for _, h in pin)
        d2h = sum(t.numel() * t.element_size() for t in out_host) + 4
        steps = max(1, min(args.steps, args.e2e_steps))

        def one():
            for d, h in pin:
                d.copy_(h, non_blocking=True)
            step()
            for o, g in zip(out_host, grads):
                o.copy_(g, non_blocking=True)
            lam_host.copy_(d_lam, non_blocking=True)

        for _ in range(3):
            one()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        barrier(world)
        for a, b in evs:
            flush.zero_()
            a.record(stream)
            one()
            b.record(stream)
        torch.cuda.synchronize()
        secs = reduce_max(sum(a.elapsed_time(b) for a, b in evs) / 1e3, world)
        e2e = {"value": job_value(flops, steps, world, secs), "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": steps,
               "ms_per_step": 1e3 * secs / steps}
    result = {
        "metric": f"diffattn_bwd TFLOP/s, algorithmic 20*D per unmasked pair "
                  f"(B={w.B},H={w.H},T={w.T},D={w.D} {'causal' if w.causal else 'full'})",
        "value": job_value(flops, args.steps, world, max_s), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * max_s / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic",
        "config": {**config_of(w, lam, args.l2_flush), "gflop_per_step": flops / 1e9,
                   # dQ kernel 12 D + dK/dV kernel 16 D per pair, plus 12 D when the
                   # forward is recomputed for the row statistics
                   "executed_gflop_per_step": flops * (28 if saved is not None else 40) / 20 / 1e9,
                   "pass": ("backward from the saved forward results: statistics pass over dO, O "
                            "and A_2 V, dQ kernel, dK/dV kernel, dlambda reduction in two launches "
                            "(5 launches per step)") if saved is not None else
                           ("backward with the forward recomputed: forward kernel in "
                            "row-statistics mode, dQ kernel, dK/dV kernel, dlambda reduction in "
                            "two launches (5 launches per step)")},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": None,
                     "peak_source": f"{src} bf16_tflops (burst)",
                     "scope": "the whole diffattn_bwd call (5 launches); per-kernel shares in profiles/"},
        "e2e": e2e, "gpu_launches": 5 * args.steps, "clocks": clocks,
    }
    if rank == 0 and world == 1 and args.cpu_baseline:
        result["cpu_baseline"] = cpu_baseline_backward(inp, dout, w, lam, args.cpu_budget)
    return result


def run_decode(args, world, rank, local):
    """Decode (Tq queries over a Tk-key cache): HBM-bound, so the metric is
    algorithmic GB/s (K1, K2, V read once; Q read and O written once)."""
    import torch
    import differential_attention_fwd_gb300 as da
    from differential_attention_fwd_gb300 import _lib
    from differential_attention_fwd_gb300 import build as build_mod

    build_mod.build()
    lib = _lib.load()
    prefill = args.mode == "prefill"
    w = W.PREFILL_WORKLOADS[args.prefill_workload] if prefill else W.DECODE_WORKLOADS[args.decode_workload]
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    inp = W.draw_kv(w)
    d_in = [torch.from_numpy(x).to(dev, tdt) for x in (inp.q1, inp.k1, inp.q2, inp.k2, inp.v)]
    if getattr(w, "shared_keys", False):
        d_in[3] = d_in[1]
    d_out = torch.empty((w.B, w.H, w.Tq, w.Dv), dtype=tdt, device=dev)
    flush = L2Flush(dev, args.l2_flush)
    stream = torch.cuda.current_stream(dev)
    desc = da.make_kv_desc(*d_in, d_out)
    need = int(lib.diffattn_decode_workspace_bytes(ctypes.byref(desc)))
    ws = torch.empty(need // 4 + 4, dtype=torch.float32, device=dev)
    ptrs = [ctypes.c_void_p(t.data_ptr()) for t in d_in]

    def step():
        rc = lib.diffattn_decode(ctypes.byref(desc), *ptrs, ctypes.c_float(w.lambda_value), None,
                                 1 if w.causal else 0, None, ctypes.c_void_p(d_out.data_ptr()),
                                 ctypes.c_void_p(ws.data_ptr()), ctypes.c_size_t(need),
                                 ctypes.c_void_p(stream.cuda_stream))
        if rc:
            raise _lib.DiffattnError(rc, "diffattn_decode")

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    sampler = ClockSampler(local) if (args.clocks and rank == 0) else None
    barrier(world)
    if sampler:
        sampler.start()
        time.sleep(0.3)
    for a, b in ev:
        flush.zero_()
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    ms = [a.elapsed_time(b) for a, b in ev]
    max_s = reduce_max(sum(ms) / 1e3, world)
    peaks, src = load_peaks()
    gbs = w.bytes / statistics.mean(ms) * 1e3 / 1e9
    hk = f",H_kv={w.Hk}" if w.Hk != w.H else ""
    config = {"workload": w.name, "B": w.B, "H": w.H, "H_kv": w.Hk, "Tq": w.Tq, "Tk": w.Tk, "D": w.D,
              "Dv": w.Dv, "causal": w.causal, "lambda": w.lambda_value,
              "gbytes_per_step": w.bytes / 1e9, "l2": flush.describe(), "parallelism": "replicas"}
    if prefill:
        # a chunk of queries over the cache: one forward launch, compute-bound
        tflops = w.flops / statistics.mean(ms) * 1e3 / 1e12
        peak = float(peaks["bf16_tflops"])
        roofline = {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s",
                    "frac": tflops / peak, "traffic": None,
                    "peak_source": f"{src} bf16_tflops (burst; kernel timed alone)",
                    "at_sampled_clock": clock_peak(
                        tflops, clocks, torch.cuda.get_device_properties(dev).multi_processor_count)}
        return {
            "metric": f"diffattn_decode (queries over a cache) TFLOP/s (B={w.B},H={w.H}{hk},"
                      f"Tq={w.Tq},Tk={w.Tk},D={w.D},Dv={w.Dv})",
            "value": w.flops * args.steps * world / max_s / 1e12, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * max_s / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
            "data": "synthetic", "config": {**config, "gflop_per_step": w.flops / 1e9},
            "roofline": roofline, "gpu_launches": args.steps, "clocks": clocks,
        }
    return {
        "metric": f"diffattn_decode HBM GB/s (B={w.B},H={w.H}{hk},Tq={w.Tq},Tk={w.Tk},D={w.D})",
        "value": w.bytes * args.steps * world / max_s / 1e9, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * max_s / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "H_kv": w.Hk, "Tq": w.Tq, "Tk": w.Tk, "D": w.D,
                   "causal": w.causal, "lambda": w.lambda_value, "gbytes_per_step": w.bytes / 1e9,
                   "l2": flush.describe(),
                   "parallelism": "replicas"},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": float(peaks["hbm_gbs"]), "unit": "GB/s",
                     "frac": gbs / float(peaks["hbm_gbs"]), "traffic": None,
                     "peak_source": f"{src} hbm_gbs (copy bandwidth)"},
        # two launches (the key-range splits, then their combination), or one
        # when the call runs on the forward kernels (16 bytes of workspace)
        "gpu_launches": (1 if need == 16 else 2) * args.steps, "clocks": clocks,
        "path": "forward kernels (queries at the end of the key sequence)" if need == 16
                else "split-key decode",
    }


WAIT_ROLES = ("producer", "mma_issuers", "softmax_warps")
WAIT_KINDS = ("total_cycles", "q_load", "k_load", "v_load", "item_start", "tensor", "epilogue", "peer",
              "k_lead_sum", "k_lead_count", "k_late_sum", "k_late_count", "k_floor_sum",
              "first_tile_busy", "tile_busy", "epilogue_busy", "tile_count", "item_count",
              "epilogue_o_load", "epilogue_l_exchange", "epilogue_math", "epilogue_stage_wait",
              "epilogue_store")
WAIT_SPAN_CTAS = 1024
WAIT_SHARES = 8     # kinds 1..7 are shares of the role's cycles; the rest are key-tile counters


def wait_profile_summary(raw, spans=None):
    """Shares of each role's cycles spent waiting, by what completes the
    barrier (the counters of the wait-profile build: [role][kind]), and the
    spread of the CTAs' start and end times (spans: [cta][start, end] in ns,
    zero for CTAs that did not run)."""
    out = {}
    n = len(WAIT_KINDS)
    for r, role in enumerate(WAIT_ROLES):
        tot = raw[n * r]
        out[role] = {"cycles": tot, **{k: (raw[n * r + i] / tot if tot else None)
                                        for i, k in enumerate(WAIT_KINDS[:WAIT_SHARES]) if i}}
    mma = out["mma_issuers"]
    base = n * WAIT_ROLES.index("mma_issuers")
    lead_n, late_n = raw[base + 9], raw[base + 11]
    floor = raw[base + 12] / lead_n if lead_n else None
    mean_wait = raw[base + 2] / lead_n if lead_n else None
    mma["key_tiles"] = {
        "waits": lead_n,
        "mean_lead_cycles": raw[base + 8] / lead_n if lead_n else None,
        "mean_wait_cycles": mean_wait,
        "mean_wait_floor_cycles": floor,
        "late_waits": late_n,
        "mean_issue_to_landing_cycles_of_late": raw[base + 10] / late_n if late_n else None}
    # the part of the key-tile waits beyond the floor of a wait whose data is
    # already there, as a share of the MMA threads' cycles
    k_beyond = (max(0.0, (mean_wait - floor)) * lead_n / mma["cycles"]) if (lead_n and mma["cycles"]) else None
    sm = n * WAIT_ROLES.index("softmax_warps")
    tiles, items = raw[sm + 16], raw[sm + 17]
    if tiles and items:
        # per warp: first tiles are one per item, the rest are tiles - items
        out["softmax_warps"]["per_warp_cycles"] = {
            "first_tile": raw[sm + 13] / items,
            "other_tile": raw[sm + 14] / max(1, tiles - items),
            "epilogue": raw[sm + 15] / items,
            "epilogue_o_load": raw[sm + 18] / items,
            "epilogue_l_exchange": raw[sm + 19] / items,
            "epilogue_math": raw[sm + 20] / items,
            "epilogue_stage_wait": raw[sm + 21] / items,
            "epilogue_store": raw[sm + 22] / items}
    span = None
    if spans:
        pairs = [(spans[2 * i], spans[2 * i + 1]) for i in range(len(spans) // 2)
                 if spans[2 * i] and spans[2 * i + 1]]
        if pairs:
            t0 = min(a for a, _ in pairs)
            ends = sorted(b - t0 for _, b in pairs)
            span = {"ctas": len(pairs), "first_end_us": ends[0] / 1e3,
                    "median_end_us": ends[len(ends) // 2] / 1e3, "last_end_us": ends[-1] / 1e3,
                    "last_start_us": (max(a for a, _ in pairs) - t0) / 1e3}
    return {
        "build": "libdiffattn_waitprof.so: the same sources with -DDIFFATTN_WAIT_PROFILE (clock64 "
                 "around every mbarrier wait of the forward kernel; timings of this run are not "
                 "bench values)",
        "roles": out,
        # the MMA-issuing threads are the consumers of the TMA loads: the share
        # of their time spent waiting for Q/K/V tiles to land
        "tma_stall_share": (mma["q_load"] or 0) + (mma["k_load"] or 0) + (mma["v_load"] or 0),
        "k_wait_share_beyond_floor": k_beyond,
        "cta_span_last_launch": span,
        "tensor_wait_share_softmax": sum(out["softmax_warps"][k] or 0
                                         for k in ("item_start", "tensor", "epilogue")),
    }


BWD_WAIT_ROLES = ("producer", "mma_issuer", "elementwise_warps")
BWD_WAIT_KINDS = ("total_cycles", "kv_slot_free", "query_stage_free", "kv_load", "scores_read_out",
                  "query_stage_load", "operands_ready", "accumulators_read_out", "scores_ready",
                  "row_statistics", "scores_tmem_read", "math", "previous_products_done",
                  "operand_stores", "accumulators_ready", "epilogue", "tile_count", "item_count")
BWD_WAIT_SHARES = 16   # kinds 1..15 are shares of the role's cycles; the last two are counts


DQ_WAIT_ROLES = ("producer", "mma_issuer", "elementwise_warps")
DQ_WAIT_KINDS = ("total_cycles", "q_slot_free", "k_slot_free", "v_slot_free", "q_load", "k_load",
                 "v_load", "ds_ready", "dq_read_out", "scores_ready", "tmem_read", "math", "ds_store",
                 "dq_ready", "epilogue", "tile_count", "item_count")
DQ_WAIT_SHARES = 15   # kinds 1..14 are shares of the role's cycles; the last two are counts


def dq_wait_profile_summary(raw):
    """The dQ kernel's wait profile ([role][kind] counters of the wait-profile
    build), as bwd_wait_profile_summary for the dK/dV kernel."""
    n = len(DQ_WAIT_KINDS)
    out = {}
    for r, role in enumerate(DQ_WAIT_ROLES):
        tot = raw[n * r]
        out[role] = {"cycles": tot}
        for i, k in enumerate(DQ_WAIT_KINDS[1:DQ_WAIT_SHARES], start=1):
            if raw[n * r + i]:
                out[role][k] = raw[n * r + i] / tot if tot else None
    ew = n * DQ_WAIT_ROLES.index("elementwise_warps")
    tiles, items = raw[ew + 15], raw[ew + 16]
    if tiles:
        out["elementwise_warps"]["per_tile_cycles"] = {
            k: raw[ew + i] / tiles for i, k in enumerate(DQ_WAIT_KINDS) if 9 <= i <= 12}
        out["elementwise_warps"]["per_tile_cycles"]["all"] = raw[ew] / tiles
    if items:
        out["elementwise_warps"]["per_item_epilogue_cycles"] = raw[ew + 14] / items
    return {"kernel": "dq::diffattn_bwd_dq_kernel", "roles": out}


def bwd_wait_profile_summary(raw):
    """The dK/dV kernel's wait profile ([role][kind] counters of the
    wait-profile build): each role's cycles by what it waits for or works on,
    as shares of the role's cycles, and per query tile for the elementwise
    warps."""
    n = len(BWD_WAIT_KINDS)
    out = {}
    for r, role in enumerate(BWD_WAIT_ROLES):
        tot = raw[n * r]
        out[role] = {"cycles": tot}
        for i, k in enumerate(BWD_WAIT_KINDS[1:BWD_WAIT_SHARES], start=1):
            if raw[n * r + i]:
                out[role][k] = raw[n * r + i] / tot if tot else None
    ew = n * BWD_WAIT_ROLES.index("elementwise_warps")
    tiles, items = raw[ew + 16], raw[ew + 17]
    if tiles:
        out["elementwise_warps"]["per_tile_cycles"] = {
            k: raw[ew + i] / tiles for i, k in enumerate(BWD_WAIT_KINDS) if 8 <= i <= 13}
        out["elementwise_warps"]["per_tile_cycles"]["all"] = raw[ew] / tiles
    if items:
        out["elementwise_warps"]["per_item_epilogue_cycles"] = raw[ew + 15] / items
    return {"build": "libdiffattn_waitprof.so: the same sources with -DDIFFATTN_WAIT_PROFILE "
                     "(clock64 around the dK/dV kernel's barrier waits and work; timings of this "
                     "run are not bench values)",
            "kernel": "dkdv::diffattn_bwd_dkdv_kernel", "roles": out}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=W.HEADLINE, choices=sorted(W.ALL_WORKLOADS))
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work")
    ap.add_argument("--no-e2e", dest="e2e", action="store_false")
    ap.add_argument("--e2e-steps", type=int, default=100)
    ap.add_argument("--no-clocks", dest="clocks", action="store_false")
    ap.add_argument("--l2-flush", choices=["write", "write-read"], default="write-read",
                    help="the L2 flush between timed steps")
    ap.add_argument("--mode", choices=["forward", "backward", "decode", "prefill"], default="forward")
    ap.add_argument("--decode-workload", default="decode_b16h16q1k8192", choices=sorted(W.DECODE_WORKLOADS))
    ap.add_argument("--prefill-workload", default="prefill_b4h16q1024k8192",
                    choices=sorted(W.PREFILL_WORKLOADS))
    ap.add_argument("--bwd-recompute", action="store_true",
                    help="backward mode: recompute the forward instead of starting from the "
                         "training forward's saved results")
    ap.add_argument("--norm", choices=["none", "rms", "group"], default="none",
                    help="fuse a per-head norm and the (1 - lambda_init) multiplier")
    ap.add_argument("--wait-profile", action="store_true",
                    help="forward or backward mode: run the wait-profile build of the library and "
                         "report each warp role's barrier-wait shares (of the forward kernel, or of "
                         "the dK/dV kernel; a measurement run, not a bench value)")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        ap.error("at least 3 warm-up steps")

    world, rank, local = dist_env()
    try:
        check_world(args.gpus, world)
    except ValueError as e:
        ap.error(str(e))
    if world > 1 and args.impl == "ours":
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    w = W.ALL_WORKLOADS[args.workload]
    if args.mode in ("decode", "prefill") and args.impl == "ours":
        res = run_decode(args, world, rank, local)
        if rank == 0:
            print(json.dumps(res), flush=True)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    if args.impl == "reference":
        res = run_reference(args, w, world, rank)
    elif args.mode == "backward" and args.wait_profile:
        import ctypes as C
        from differential_attention_fwd_gb300 import _lib
        from differential_attention_fwd_gb300 import build as build_mod
        lib = _lib.load(build_mod.build(variant="waitprof"))
        lib.diffattn_bwd_wait_profile.argtypes = [C.POINTER(C.c_ulonglong), C.c_int]
        lib.diffattn_bwd_wait_profile.restype = C.c_int
        nk = 3 * len(BWD_WAIT_KINDS)
        nq = 3 * len(DQ_WAIT_KINDS)
        clear = (C.c_ulonglong * (nk + nq))()
        lib.diffattn_bwd_wait_profile(clear, len(clear))
        res = run_backward(args, w, world, rank, local)
        raw = (C.c_ulonglong * (nk + nq))()
        if lib.diffattn_bwd_wait_profile(raw, len(raw)) != 0:
            raise RuntimeError("diffattn_bwd_wait_profile failed")
        res = {"wait_profile": bwd_wait_profile_summary(list(raw)[:nk]),
               "wait_profile_dq": dq_wait_profile_summary(list(raw)[nk:]), "workload": w.name,
               "steps": args.steps, "warmup": args.warmup,
               "instrumented_backward_ms": res.get("ms_per_step")}
    elif args.mode == "backward":
        res = run_backward(args, w, world, rank, local)
    elif args.wait_profile:
        import ctypes as C
        from differential_attention_fwd_gb300 import _lib
        from differential_attention_fwd_gb300 import build as build_mod
        lib = _lib.load(build_mod.build(variant="waitprof"))
        lib.diffattn_wait_profile.argtypes = [C.POINTER(C.c_ulonglong), C.c_int]
        lib.diffattn_wait_profile.restype = C.c_int
        res = run_ours(args, w, world, rank, local)
        n = 3 * len(WAIT_KINDS)
        raw = (C.c_ulonglong * (n + 2 * WAIT_SPAN_CTAS))()
        if lib.diffattn_wait_profile(raw, n + 2 * WAIT_SPAN_CTAS) != 0:
            raise RuntimeError("diffattn_wait_profile failed")
        res = {"wait_profile": wait_profile_summary(list(raw)[:n], list(raw)[n:]), "workload": w.name,
               "steps": args.steps, "warmup": args.warmup,
               "instrumented_kernel_ms_median": res["roofline"]["fwd_ms_median"]}
    else:
        res = run_ours(args, w, world, rank, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
