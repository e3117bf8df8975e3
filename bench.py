"""Benchmark: fused top-K KL loss, forward + backward, on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step is one pass of the whole loss path over one batch: kd_fused_kl_fwd
(teacher prep, logits GEMM with the online log-sum-exp and id gather in its
epilogue, merge) and then kd_fused_kl_bwd (recompute GEMM with the dz
epilogue, dH and dW GEMMs), chunk group by chunk group. The headline workload
is the long-context projection (T=262144, d=2880, V=201088, K=100,
chunk=4096), the largest of the loss workloads, with synthetic inputs and a
teacher cache built by kd_topk_cache from a perturbed-W teacher. The other
two loss workloads (Llama-3.2-3B- and GPT-OSS-20B-shaped) are timed in the
same run and reported under "other_configs". The offline cache extraction is
timed separately on its own workload ([8192, 201088] bf16 logits) and
reported under "topk_extraction".

Prints one JSON line (rank 0). Under torchrun each rank runs an independent
replica on its own GPU (no collective on the data path); the barrier and the
max over ranks use torch.distributed.
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
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import top_kl_loss_tcgen05_b300 as kd  # noqa: E402
from top_kl_loss_tcgen05_b300 import _native, synth  # noqa: E402

METRIC = "fused top-K KL fwd+bwd tokens/s and TFLOP/s (% BF16 tensor peak); peak GiB"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


# ----------------------------------------------------------------------------- helpers


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def _code_only(src: str) -> str:
    """C/CUDA source without comments, trailing blanks and empty lines, so
    that an edit to comments alone keeps the hash."""
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    lines = (re.sub(r"//.*$", "", ln).rstrip() for ln in src.splitlines())
    return "\n".join(ln for ln in lines if ln)


def kernel_src_hash(files=None) -> str:
    """Identifies CUDA sources (code, not comments) that an ncu traffic record
    was taken on: the listed files of the package's csrc/, else all of them."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "top_kl_loss_tcgen05_b300", "csrc")
    names = sorted(files) if files else sorted(f for f in os.listdir(csrc) if f.endswith((".cu", ".cuh", ".h")))
    for f in names:
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update(f.encode() + b"\0" + _code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def gemm_tiles_desc() -> str:
    """The GEMM tile shapes this process runs (the library's test switches,
    kd_test_set_gemm_tiles, override the per-kernel defaults)."""
    cta2, wide = _native.get_gemm_tiles()
    if cta2 == 0:
        return "128x256 per CTA"
    if wide in (0, 1):
        return "%s per CTA pair (tcgen05 cta_group::2), every GEMM" % ("256x512" if wide == 1 else "256x256")
    return "256x512 per CTA pair (tcgen05 cta_group::2), every GEMM"


def default_group(chunk: int) -> int:
    """Chunks per GEMM launch under the library's default rule (kd.h: G =
    clamp(4096 / chunk, 1, 4), integer division)."""
    return max(1, min(4, 4096 // chunk))


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources and this workload; else None."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
    except Exception:
        return None
    e = d.get(kernel, {}).get(workload)
    if not e or e.get("src_sha") != kernel_src_hash(e.get("src_files")):
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, dev: torch.device):
        self.uuid = None
        try:
            self.uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
        except Exception:
            pass
        self.proc = None
        self.lines = []

    def start(self):
        cmd = ["nvidia-smi", "--query-gpu=" + self.Q, "--format=csv,noheader,nounits", "-lms", "200"]
        if self.uuid:
            cmd += ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=5)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info

        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return len(os.sched_getaffinity(0))


# ----------------------------------------------------------------------------- workload


def make_workload(name: str, dev: torch.device, rows: int | None = None):
    c = synth.CONFIGS[name]
    T, d, V, K, chunk, seed = c["T"], c["d"], c["V"], c["K"], c["chunk"], c["seed"]
    if rows:
        T = min(T, int(rows))
    H, W = synth.student(T, d, V, seed, device=dev)
    # teacher cache: perturbed-W teacher logits (fp32, chunk by chunk) -> kd_topk_cache
    Wt = synth.teacher_weight(W, seed)
    ids = torch.empty(T, K, dtype=torch.int32, device=dev)
    logp = torch.empty(T, K, dtype=torch.float32, device=dev)
    step = max(1, min(T, (1 << 30) // (4 * V)))
    for t0 in range(0, T, step):
        t1 = min(T, t0 + step)
        tl = synth.teacher_logits_from(H[t0:t1], Wt)
        i, lp = kd.topk_cache(tl, K)
        ids[t0:t1] = i
        logp[t0:t1] = lp
        del tl
    del Wt
    torch.cuda.synchronize(dev)
    return dict(T=T, d=d, V=V, K=K, chunk=chunk, H=H, W=W, ids=ids, logp=logp)


def describe(name: str, rows: int | None = None) -> str:
    c = synth.CONFIGS[name]
    T = min(c["T"], int(rows)) if rows else c["T"]
    out = "%s: T=%d d=%d V=%d K=%d chunk=%d" % (name, T, c["d"], c["V"], c["K"], c["chunk"])
    if T != c["T"]:
        out += " (first %d of its %d positions)" % (T, c["T"])
    return out


# ----------------------------------------------------------------------------- oracle (cpu baseline)


def oracle_sample(wl_cpu, rows: int):
    """Time the fp64 oracle on `rows` positions of the workload (fwd + bwd)."""
    from oracle import kd_oracle as O

    H = wl_cpu["H"][:rows]
    W64 = wl_cpu["W64"]
    ids = wl_cpu["ids"][:rows]
    logp = wl_cpu["logp"][:rows]
    t0 = time.perf_counter()
    O.fused_kl_forward(H, W64, ids, logp)
    O.fused_kl_backward(H, W64, ids, logp, 1.0 / wl_cpu["T"])
    return time.perf_counter() - t0


def cpu_workload(wl):
    return dict(T=wl["T"], H=wl["H"][:4096].float().cpu().numpy().astype(np.float64),
                W64=wl["W"].float().cpu().numpy().astype(np.float64), ids=wl["ids"][:4096].cpu().numpy(),
                logp=wl["logp"][:4096].cpu().numpy())


def size_sample(cw, budget_s: float) -> int:
    """Rows of oracle work that take at most about budget_s. Rows double from
    4 until one call takes a third of the budget (or all rows are in), then
    scale to the budget from that last measurement. With time(r) = a + b r
    and a >= 0 (a per-call cost, e.g. allocating the fp64 dW), scaling the
    rows by budget / time(r) cannot overshoot the budget."""
    cap = len(cw["ids"])
    oracle_sample(cw, 2)  # warm-up
    r = min(4, cap)
    t = oracle_sample(cw, r)
    while t < budget_s / 3.0 and r < cap:
        r = min(cap, 2 * r)
        t = oracle_sample(cw, r)
    return int(max(2, min(cap, r * budget_s / max(t, 1e-6))))


def cpu_baseline(wl, budget_s: float = 15.0):
    cw = cpu_workload(wl)
    rows = size_sample(cw, budget_s)
    t = oracle_sample(cw, rows)
    if t < 0.4 * budget_s and rows < len(cw["ids"]):  # the fit underestimated the per-row cost
        rows = int(min(len(cw["ids"]), rows * min(4.0, budget_s / max(t, 1e-3))))
        t = oracle_sample(cw, rows)
    return {"value": rows / t, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
            "sample": "fp64 numpy oracle, forward + backward (loss, lse, dH, dW contribution) of the first %d "
                      "positions of the workload at full d and V; %.1f s" % (rows, t)}


# ----------------------------------------------------------------------------- top-K extraction


def bench_topk(dev, peaks, iters=5, rows=None):
    c = dict(synth.CONFIGS["topk"])
    if rows:
        c["T"] = int(rows)
    x = synth.topk_logits(c["T"], c["V"], c["seed"], device=dev)
    ws = kd.workspace(256, dev)
    for _ in range(2):
        kd.topk_cache(x, c["K"], ws=ws)
    torch.cuda.synchronize(dev)
    _native.profile_begin()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(iters):
        kd.topk_cache(x, c["K"], ws=ws)
    e.record()
    torch.cuda.synchronize(dev)
    prof = _native.profile_end()
    ms = s.elapsed_time(e) / iters
    launches, kms = prof.get("topk_cache", (iters, ms * iters))
    kernel_ms = kms / max(1, launches)
    nbytes = 2 * c["T"] * c["V"] + 8 * c["T"] * c["K"]
    achieved = nbytes / (kernel_ms * 1e-3) / 1e9
    peak = float(peaks["hbm_gbs"])
    fallback_rows = int(ws[4:8].view(torch.int32).item())
    del x
    return {
        "workload": "topk: logits [%d, %d] bf16 (N(0,2) + Zipf-like bias), K=%d" % (c["T"], c["V"], c["K"]),
        "ms": kernel_ms, "rows_per_s": c["T"] / (kernel_ms * 1e-3),
        "rows_on_radix_path": fallback_rows // (iters + 2),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": ncu_traffic("topk_cache", "topk"), "algorithmic_bytes_per_launch": nbytes},
    }


def bench_teacher(dev, peaks, iters=5):
    """Teacher-side cache (kd_teacher_topk_cache) on a Llama-3.1-8B-shaped LM
    head: the projection GEMM with its LSE epilogue, and the tile-pruned
    top-K selection. Timed alone, so the GEMM roofline uses the burst peak."""
    c = synth.CONFIGS["teacher"]
    T, d, V, K, chunk = c["T"], c["d"], c["V"], c["K"], c["chunk"]
    H, W = synth.teacher_head(T, d, V, c["seed"], device=dev)
    ws = kd.workspace(_native.lib().kd_teacher_topk_workspace_size(d, V, K, chunk), dev)
    for _ in range(2):
        kd.teacher_topk_cache(H, W, K, chunk=chunk, ws=ws)
    torch.cuda.synchronize(dev)
    _native.profile_begin()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(iters):
        kd.teacher_topk_cache(H, W, K, chunk=chunk, ws=ws)
    e.record()
    torch.cuda.synchronize(dev)
    prof = _native.profile_end()
    ms = s.elapsed_time(e) / iters
    gn, gms = prof.get("teacher_logits_gemm", (1, float("nan")))
    sn, sms = prof.get("teacher_tile_topk", (1, float("nan")))
    flops_launch = 2.0 * T * d * V * iters / gn
    achieved = flops_launch / (gms / gn * 1e-3) / 1e12
    peak = float(peaks["bf16_tflops"])
    exact_rows = int(ws[4:8].view(torch.int32).item())
    del H, W, ws
    return {
        "workload": "teacher: H [%d, %d] x W [%d, %d] bf16 (Llama-3.1-8B-shaped LM head), K=%d, chunk=%d"
                    % (T, d, V, d, K, chunk),
        "ms": ms, "rows_per_s": T / (ms * 1e-3), "tflops": 2.0 * T * d * V / (ms * 1e-3) / 1e12,
        "gemm_ms": gms / iters, "select_ms": sms / iters, "rows_on_radix_path": exact_rows // (iters + 2),
        "workspace_gib": ws_bytes_gib(d, V, K, chunk),
        "roofline": {"bound": "tensor", "kernel": "teacher_logits_gemm", "achieved": achieved, "peak": peak,
                     "unit": "TFLOP/s", "frac": achieved / peak, "traffic": None,
                     "peak_kind": "bf16_tflops burst (measured)", "algorithmic_flops_per_launch": flops_launch},
    }


def ws_bytes_gib(d, V, K, chunk):
    return _native.lib().kd_teacher_topk_workspace_size(d, V, K, chunk) / 2**30


# ----------------------------------------------------------------------------- main


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_reference(args, world, rank):
    """The reference arm: the fp64 oracle, as it stands, on the host cores."""
    if rank != 0:
        return
    dev = torch.device("cuda", 0) if torch.cuda.is_available() else torch.device("cpu")
    name = args.workload
    c = synth.CONFIGS[name]
    # inputs of the GPU arm's shapes and distributions, drawn on the host for
    # the first (at most 4096) positions; a synthetic cache of the same shape
    # stands in for the teacher's, so this arm runs without the GPU path
    H, W = synth.student(min(c["T"], 4096), c["d"], c["V"], c["seed"], device="cpu")
    ids, logp = synth.synthetic_cache(min(c["T"], 4096), c["V"], c["K"], c["seed"])
    cw = dict(T=c["T"], H=H.float().numpy().astype(np.float64), W64=W.float().numpy().astype(np.float64),
              ids=ids.numpy(), logp=logp.numpy())
    # each step a bounded sample, sized so the whole run takes about 2.5 min
    per_step = max(1.0, min(8.0, 150.0 / max(1, args.steps + args.warmup)))
    rows = size_sample(cw, per_step)
    for _ in range(args.warmup):
        oracle_sample(cw, rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_sample(cw, rows)
    el = time.perf_counter() - t0
    value = rows * args.steps / el
    cores = blas_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": describe(name), "sample_rows_per_step": rows},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": "fp64 numpy oracle fwd+bwd of %d positions per step at full d and V" % rows},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def fused_roofline(prof, steps, T, d, V, peaks, peaks_src, clk, workload):
    """Roofline of the dominant kernel of a fused-loss step: algorithmic flops
    per launch (the kernel's per-step flops / its launches per step) over its
    mean CUDA-event launch time. Reported against the sustained bf16 peak (the
    kernel runs inside a long step), against the burst peak, and
    clock-normalised: against the sustained peak scaled from the SM clock it
    was measured at to this run's median SM clock."""
    flops_per_step = {"logits_fwd_lse_gather": 2.0 * T * d * V, "logits_dz": 2.0 * T * d * V,
                      "grad_dH_dW": 4.0 * T * d * V}
    flops_per_launch = {k: f * steps / prof[k][0] for k, f in flops_per_step.items() if k in prof}
    total_kernel_ms = sum(v[1] for v in prof.values())
    kernels = {k: {"launches": n, "ms_per_step": t / steps, "share": t / total_kernel_ms if total_kernel_ms else 0.0}
               for k, (n, t) in prof.items()}
    for k in kernels:
        if k in flops_per_launch:
            n, t = prof[k]
            kernels[k]["tflops"] = flops_per_launch[k] / (t / n * 1e-3) / 1e12
    dom = max(prof.items(), key=lambda kv: kv[1][1])[0] if prof else None
    roof = None
    if dom in flops_per_launch:
        n, t = prof[dom]
        achieved = flops_per_launch[dom] / (t / n * 1e-3) / 1e12
        peak_tf = float(peaks["bf16_tflops_sustained"])
        peak_burst = float(peaks["bf16_tflops"])
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak_tf, "unit": "TFLOP/s",
                "frac": achieved / peak_tf, "traffic": ncu_traffic(dom, workload), "kernel": dom,
                "peak_kind": "bf16_tflops_sustained (%s)" % peaks_src,
                "algorithmic_flops_per_launch": flops_per_launch[dom],
                "peak_burst": peak_burst, "frac_burst": achieved / peak_burst}
        peak_mhz = (peaks.get("clocks_under_load") or {}).get("sm_mhz_median")
        if clk and clk.get("sm_mhz") and peak_mhz:
            roof.update({"sm_mhz": clk["sm_mhz"], "peak_sustained_sm_mhz": peak_mhz,
                         "frac_clock_normalised": achieved / (peak_tf * clk["sm_mhz"] / peak_mhz),
                         "clock_note": "frac_clock_normalised = achieved / (peak x this run's median SM MHz / "
                                       "the median SM MHz the sustained peak was measured at)"})
    return roof, kernels, sum(n for n, _ in prof.values())


class FusedRun:
    """Device buffers and the fused-loss step (kd_fused_kl_fwd then
    kd_fused_kl_bwd, through the C ABI) of one workload."""

    def __init__(self, name, dev, rows=None):
        self.name = name
        self.rows = rows
        self.dev = dev
        wl = make_workload(name, dev, rows)
        self.wl = wl
        self.T, self.d, self.V, self.K, self.chunk = wl["T"], wl["d"], wl["V"], wl["K"], wl["chunk"]
        self.H, self.W, self.ids, self.logp = wl["H"], wl["W"], wl["ids"], wl["logp"]
        self.ws = kd.fused_kl_workspace(self.d, self.V, self.K, self.chunk, dev)
        self.lse = torch.empty(self.T, dtype=torch.float32, device=dev)
        self.loss = torch.empty((), dtype=torch.float32, device=dev)
        self.dH = torch.empty(self.T, self.d, dtype=torch.float32, device=dev)
        self.dW = torch.empty(self.V, self.d, dtype=torch.float32, device=dev)
        self.L = _native.lib()
        self.stream = torch.cuda.current_stream(dev).cuda_stream

    def fwd(self, Hx=None, idsx=None, logpx=None):
        Hx = self.H if Hx is None else Hx
        idsx = self.ids if idsx is None else idsx
        logpx = self.logp if logpx is None else logpx
        _native.check("kd_fused_kl_fwd", self.L.kd_fused_kl_fwd(
            Hx.data_ptr(), self.W.data_ptr(), idsx.data_ptr(), logpx.data_ptr(), self.T, self.d, self.V, self.K,
            self.chunk, self.loss.data_ptr(), self.lse.data_ptr(), None, self.ws.data_ptr(), self.ws.numel(),
            self.stream))

    def bwd(self, Hx=None, idsx=None, logpx=None):
        Hx = self.H if Hx is None else Hx
        idsx = self.ids if idsx is None else idsx
        logpx = self.logp if logpx is None else logpx
        _native.check("kd_fused_kl_bwd", self.L.kd_fused_kl_bwd(
            Hx.data_ptr(), self.W.data_ptr(), idsx.data_ptr(), logpx.data_ptr(), self.lse.data_ptr(), self.T,
            self.d, self.V, self.K, self.chunk, 1.0 / self.T, None, self.dH.data_ptr(), self.dW.data_ptr(), 0,
            self.ws.data_ptr(), self.ws.numel(), self.stream))

    def step(self, Hx=None, idsx=None, logpx=None):
        self.fwd(Hx, idsx, logpx)
        self.bwd(Hx, idsx, logpx)

    def fwdbwd(self):
        _native.check("kd_fused_kl_fwdbwd", self.L.kd_fused_kl_fwdbwd(
            self.H.data_ptr(), self.W.data_ptr(), self.ids.data_ptr(), self.logp.data_ptr(), self.T, self.d, self.V,
            self.K, self.chunk, 1.0 / self.T, None, self.loss.data_ptr(), self.lse.data_ptr(), None,
            self.dH.data_ptr(), self.dW.data_ptr(), 0, self.ws.data_ptr(), self.ws.numel(), self.stream))

    def io_gib(self):
        ts = (self.H, self.W, self.ids, self.logp, self.lse, self.loss, self.dH, self.dW)
        return sum(t.numel() * t.element_size() for t in ts) / 2**30

    def check_status(self, where):
        st = kd.read_device_status(self.ws)
        if st != 0:
            raise RuntimeError("device status %s %s" % (_native.status_string(st), where))

    def peak_step(self):
        """Peak device memory of one step (everything is allocated through torch)."""
        torch.cuda.synchronize(self.dev)
        torch.cuda.reset_peak_memory_stats(self.dev)
        self.step()
        torch.cuda.synchronize(self.dev)
        return torch.cuda.max_memory_allocated(self.dev) / 2**30

    def timed(self, steps, world):
        """(elapsed ms max over ranks, per-kernel profile, clocks) of `steps`
        back-to-back steps, bracketed by a barrier and synchronisations."""
        clocks = ClockSampler(self.dev)
        barrier(world)
        torch.cuda.synchronize(self.dev)
        clocks.start()
        time.sleep(0.3)
        _native.profile_begin()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record()
        for _ in range(steps):
            self.step()
        ev1.record()
        torch.cuda.synchronize(self.dev)
        prof = _native.profile_end()
        barrier(world)
        clk = clocks.stop()
        return max_over_ranks(ev0.elapsed_time(ev1), world), prof, clk


def config_desc(run: FusedRun) -> dict:
    G = default_group(run.chunk)
    return {"workload": describe(run.name, run.rows), "group": G, "rows_per_gemm_launch": G * run.chunk,
            "group_note": "each GEMM launch covers a group of G chunks (the library's default group rule); the "
                          "workspace holds one group's bf16 dz"}


def measure_other(name, args, dev, peaks, peaks_src, world):
    """tokens/s, TFLOP/s, % of the bf16 peaks, roofline and peak memory of one
    more loss workload, timed like the headline (K steps after W warm-up)."""
    run = FusedRun(name, dev)
    peak_gib = run.peak_step()
    for _ in range(args.warmup - 1):
        run.step()
    run.check_status("during warm-up (%s)" % name)
    el_ms, prof, clk = run.timed(args.steps, world)
    run.check_status("in the timed region (%s)" % name)
    T, d, V = run.T, run.d, run.V
    tflops = 8.0 * T * d * V * args.steps * world / (el_ms * 1e-3) / 1e12
    roof, kernels, launches = fused_roofline(prof, args.steps, T, d, V, peaks, peaks_src, clk, name)
    out = {"value": T * args.steps * world / (el_ms * 1e-3), "unit": "tokens/s", "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": el_ms / args.steps, "tflops": tflops,
           "pct_bf16_peak": tflops / float(peaks["bf16_tflops_sustained"]),
           "pct_bf16_peak_burst": tflops / float(peaks["bf16_tflops"]),
           "peak_gib": peak_gib, "workspace_gib": run.ws.numel() / 2**30, "io_gib": run.io_gib(),
           "config": config_desc(run), "roofline": roof, "gpu_launches": launches, "clocks": clk,
           "kernels": kernels}
    del run
    torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="long", choices=["tiny", "llama3b", "gptoss20b", "long"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-topk", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-fwdbwd", action="store_true", help="skip timing the single-call forward + backward")
    ap.add_argument("--no-teacher", action="store_true", help="skip timing the teacher-side cache")
    ap.add_argument("--no-others", action="store_true", help="skip timing the other loss workloads")
    ap.add_argument("--topk-rows", type=int, default=None, help="rows of the top-K workload (default 8192)")
    ap.add_argument("--rows", type=int, default=None,
                    help="positions of the loss workload (default: all of it). A truncated run keeps d, V, K and the "
                         "chunk, so each GEMM launch does the same work as in the full run: for small profiling "
                         "captures, not for bench lines")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    dev = torch.device("cuda", local)
    peaks, peaks_src = load_peaks()
    _native.load()

    run = FusedRun(args.workload, dev, args.rows)
    T, d, V, K, chunk = run.T, run.d, run.V, run.K, run.chunk
    H, W, ids, logp = run.H, run.W, run.ids, run.logp
    peak_gib = run.peak_step()
    ws_gib = run.ws.numel() / 2**30
    io_gib = run.io_gib()
    for _ in range(args.warmup - 1):
        run.step()
    torch.cuda.synchronize(dev)
    run.check_status("during warm-up")

    # ---- timed region (device-resident inputs)
    el_ms, prof, clk = run.timed(args.steps, world)
    ms_step = el_ms / args.steps
    tokens_s = T * args.steps * world / (el_ms * 1e-3)
    tflops = 8.0 * T * d * V * args.steps * world / (el_ms * 1e-3) / 1e12
    peak_tf = float(peaks["bf16_tflops_sustained"])
    run.check_status("in the timed region")
    roof, kernels, gpu_launches = fused_roofline(prof, args.steps, T, d, V, peaks, peaks_src, clk, args.workload)

    # forward and backward separately (same calls, events between them)
    n_ph = min(args.steps, 5)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n_ph)]
    for e in evs:
        e[0].record()
        run.fwd()
        e[1].record()
        run.bwd()
        e[2].record()
    torch.cuda.synchronize(dev)
    fwd_ms = sorted(e[0].elapsed_time(e[1]) for e in evs)[len(evs) // 2]
    bwd_ms = sorted(e[1].elapsed_time(e[2]) for e in evs)[len(evs) // 2]
    phases = {"fwd_ms": fwd_ms, "bwd_ms": bwd_ms, "fwd_tflops": 2.0 * T * d * V / (fwd_ms * 1e-3) / 1e12,
              "bwd_tflops": 6.0 * T * d * V / (bwd_ms * 1e-3) / 1e12, "stat": "median over %d steps" % len(evs)}

    # ---- single-call forward + backward (kd_fused_kl_fwdbwd: each chunk's
    # logits computed once, 6 T d V projection flops). Reported beside the
    # headline, which is the recompute path (8 T d V).
    fwdbwd = None
    if not args.no_fwdbwd:
        n_fb = min(args.steps, 10)
        for _ in range(args.warmup):
            run.fwdbwd()
        torch.cuda.synchronize(dev)
        barrier(world)
        _native.profile_begin()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record()
        for _ in range(n_fb):
            run.fwdbwd()
        f1.record()
        torch.cuda.synchronize(dev)
        fprof = _native.profile_end()
        fb_ms = max_over_ranks(f0.elapsed_time(f1), world) / n_fb
        run.check_status("in kd_fused_kl_fwdbwd")
        fb_tot = sum(v[1] for v in fprof.values())
        fwdbwd = {"value": T * world / (fb_ms * 1e-3), "unit": "tokens/s", "ms_per_step": fb_ms, "steps": n_fb,
                  "tflops_executed": 6.0 * T * d * V * world / (fb_ms * 1e-3) / 1e12,
                  "pct_bf16_peak_executed": 6.0 * T * d * V / (fb_ms * 1e-3) / 1e12 / peak_tf,
                  "flops_basis": "6*T*d*V: the projection is computed once per chunk, no recompute",
                  "gpu_launches": sum(n for n, _ in fprof.values()),
                  "kernels": {k: {"launches": n, "ms_per_step": t / n_fb, "share": t / fb_tot if fb_tot else 0.0}
                              for k, (n, t) in fprof.items()}}

    # ---- end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        Hh = H.cpu().pin_memory()
        ih = ids.cpu().pin_memory()
        lh = logp.cpu().pin_memory()
        bufs = [(torch.empty_like(H), torch.empty_like(ids), torch.empty_like(logp)) for _ in range(2)]
        out = torch.empty((), dtype=torch.float32).pin_memory()
        cur = torch.cuda.current_stream(dev)
        side = torch.cuda.Stream(dev)
        bi = Hh.numel() * Hh.element_size() + ih.numel() * 4 + lh.numel() * 4

        def h2d(b, stream):
            with torch.cuda.stream(stream):
                for dst, src in zip(bufs[b], (Hh, ih, lh)):
                    dst.copy_(src, non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(stream)
            return ev

        def serial_step():
            h2d(0, cur)
            run.step(*bufs[0])
            out.copy_(run.loss, non_blocking=True)
            cur.synchronize()
            return float(out)

        def run_pipelined(n):
            # the copy of step i + 1's inputs runs on a side stream during step
            # i; every step still waits for its own loss on the host
            ready = h2d(0, side)
            for i in range(n):
                b = i & 1
                cur.wait_event(ready)
                run.step(*bufs[b])
                out.copy_(run.loss, non_blocking=True)
                if i + 1 < n:
                    ready = h2d(b ^ 1, side)  # buffer b ^ 1 was last read by step i - 1, which has finished
                cur.synchronize()
                float(out)

        for _ in range(2):
            serial_step()
        run_pipelined(2)
        torch.cuda.synchronize(dev)
        n_e2e = max(3, min(8, args.steps // 2))
        barrier(world)
        t0 = time.perf_counter()
        run_pipelined(n_e2e)
        el = max_over_ranks(time.perf_counter() - t0, world)
        barrier(world)
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            serial_step()
        el_serial = max_over_ranks(time.perf_counter() - t0, world)
        e2e = {"value": T * n_e2e * world / el, "unit": "tokens/s", "h2d_bytes_per_step": bi,
               "d2h_bytes_per_step": 4, "steps": n_e2e, "serial_value": T * n_e2e * world / el_serial,
               "note": "host clock around n steps; every step copies H, teacher ids and logp from pinned host "
                       "memory and reads its loss back to the host. value: the next step's inputs are copied on "
                       "a side stream while the current step runs (a prefetching loader). serial_value: copy, "
                       "step and read-back one after another. W (LM-head parameter), dH and dW stay on the "
                       "device"}
        del bufs, Hh, ih, lh

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:  # a reported baseline at N=1 only
        cpu = cpu_baseline(run.wl)
    cfg = config_desc(run)
    cfg.update({"parallelism": "replicas" if world > 1 else "1 gpu",
                "l2": "inputs larger than L2 (W alone is %.0f MB)" % (V * d * 2 / 1e6),
                "teacher_cache": "kd_topk_cache of fp32 perturbed-W teacher logits",
                "gemm_tiles": gemm_tiles_desc()})
    del run, H, W, ids, logp
    torch.cuda.empty_cache()

    # ---- the other loss workloads, each timed like the headline
    others = {}
    if not args.no_others:
        for name in ("llama3b", "gptoss20b", "long"):
            if name != args.workload:
                others[name] = measure_other(name, args, dev, peaks, peaks_src, world)

    topk = None if args.no_topk else bench_topk(dev, peaks, rows=args.topk_rows)
    teacher = None if args.no_teacher else bench_teacher(dev, peaks)

    if rank == 0:
        line = {
            "metric": METRIC, "value": tokens_s, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "tflops": tflops, "pct_bf16_peak": tflops / peak_tf,
            "pct_bf16_peak_burst": tflops / float(peaks["bf16_tflops"]),
            "pct_bf16_peak_basis": "8*T*d*V flops per step vs bf16_tflops_sustained and bf16_tflops (burst) "
                                   "(%s)" % peaks_src,
            "peak_gib": peak_gib, "workspace_gib": ws_gib, "io_gib": io_gib, "phases": phases,
            "config": cfg,
            "roofline": roof, "kernels": kernels, "gpu_launches": gpu_launches,
            "clocks": clk, "e2e": e2e, "cpu_baseline": cpu, "other_configs": others or None,
            "topk_extraction": topk, "fused_fwdbwd": fwdbwd, "teacher_topk": teacher,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
