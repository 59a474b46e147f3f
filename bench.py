"""Benchmark of the fused linear cross-entropy hot path (forward + backward) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

One step = flce_forward + flce_backward (every kernel of the path) over one batch of the
workload's synthetic inputs, already resident in HBM. Prints ONE JSON line on rank 0.

* value: whole-job tokens/s (all ranks), from CUDA events over exactly K timed steps bracketed
  by a barrier and a device synchronise on both sides, max over ranks.
* roofline: the dominant tensor-core kernel role (largest summed launch time in the timed
  region), timed per launch with CUDA events on its launch stream through libflce's timing
  hooks; achieved = its algorithmic FLOPs / its launch time, against the measured dense-bf16
  burst peak (the timed region lasts well under a second); the fraction of the sustained
  (seconds-long, power-capped) peak is reported beside it.
* e2e: the same metric with host-resident inputs: each step copies x, weight and target from
  pinned host memory, runs the path, and reads the loss back, all inside the timed region.
* cpu_baseline: the float64 oracle timed on this host's cores on a bounded token sample.
* --impl reference: the reference arm is the float64 oracle (there is no other implementation
  to run): each step is a bounded token sample of the same workload, timed on the host cores.
* context.torch_eager: for comparison only, the unfused PyTorch formulation on the same GPU
  (bf16 matmul through cuBLAS, logits upcast to fp32, cross_entropy, autograd backward), which
  materialises the T x V logits; run when they fit comfortably in device memory.
With N > 1 (torchrun) every rank runs an independent replica of the workload (weak scaling,
no collective on the data path); the path has no exchange step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from lm_head_linear_02_gb300 import roofline  # noqa: E402
from lm_head_linear_02_gb300.inputs import WORKLOADS, make_inputs  # noqa: E402

METRIC = "FLCE fwd+bwd tokens/s and % dense-BF16 tensor peak at T=16384,H=4096,V=128256"
UNIT = "tokens/s"
DEFAULT_WORKLOAD = "llama3_head_t16384"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
CSRC = os.path.join(ROOT, "lm_head_linear_02_gb300", "csrc")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.json")


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# --tune NAME=VALUE: the library's process-wide tuning keys (include/flce.h, FLCE_TUNE_*)
TUNING_KEYS = {"raster_rows": "FLCE_TUNE_RASTER_ROWS", "sm_pairs": "FLCE_TUNE_SM_PAIRS",
               "wide_tiles": "FLCE_TUNE_WIDE_TILES", "raster_vocab": "FLCE_TUNE_RASTER_VOCAB",
               "split_epilogue": "FLCE_TUNE_SPLIT_EPILOGUE", "chunk_bytes": "FLCE_TUNE_CHUNK_BYTES",
               "ordered_drain": "FLCE_TUNE_ORDERED_DRAIN"}


def parse_tuning(items):
    """['raster_vocab=4096', ...] -> {'raster_vocab': 4096, ...} (names checked, values int)."""
    out = {}
    for item in items:
        name, sep, value = item.partition("=")
        if not sep or name not in TUNING_KEYS:
            raise ValueError(f"--tune expects NAME=VALUE with NAME in {sorted(TUNING_KEYS)}")
        out[name] = int(value, 0)
    return out


def max_over_ranks(value: float, dist, device=None) -> float:
    """The largest of each rank's value (a timed region ends when the slowest rank is done).
    Single-process runs (dist None) return the value itself."""
    if dist is None:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, seconds: float) -> float:
    """Units processed by all ranks together per second of the slowest rank."""
    return world * units_per_rank / seconds


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def strip_comments(src: str) -> str:
    """C/C++ source without comments and whitespace (string and character literals kept), so
    that the digest below changes with the code only."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            i = src.find("\n", i)
            i = n if i < 0 else i
        elif src.startswith("/*", i):
            i = src.find("*/", i + 2)
            i = n if i < 0 else i + 2
        else:
            if not c.isspace():
                out.append(c)
            i += 1
    return "".join(out)


def sources_digest(read=None) -> str:
    """SHA-256 over the comment-free kernel sources (the key of the recorded DRAM traffic)."""
    h = hashlib.sha256()
    names = sorted(n for n in os.listdir(CSRC) if n.endswith((".cu", ".cuh", ".h")))
    for name in names:
        if read is None:
            with open(os.path.join(CSRC, name), encoding="utf-8") as f:
                text = f.read()
        else:
            text = read(name)
        h.update(name.encode() + b"\0" + strip_comments(text).encode())
    return h.hexdigest()


def recorded_traffic(role: str, workload: str):
    """DRAM bytes per launch from a committed ncu capture, or None if the kernels changed."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    entry = rec.get("roles", {}).get(role)
    if not entry or rec.get("sources_sha256") != sources_digest():
        return None
    if entry.get("workload") != workload:
        return None
    return entry.get("bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock/throttle sampling during the timed region: samples every 100 ms,
    timestamped, of which those inside the window marked by begin()/end() are kept."""

    # power.draw.instant: power.draw is a one-second average, longer than a short timed region
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw.instant,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.5)  # let the sampler produce its first rows before the timed region
        except OSError:
            self.proc = None

    def begin(self):
        self.t0 = time.time()

    def end(self):
        self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        import datetime
        rows = []
        for r in out.strip().splitlines():
            r = [c.strip() for c in r.split(",")]
            if len(r) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                continue
            try:
                sm, sm_max = float(r[1]), float(r[2])
            except ValueError:
                continue
            try:
                power = float(r[3])
            except ValueError:  # "[N/A]" on boards that do not report it
                power = float("nan")
            rows.append((ts, sm, sm_max, r[5:9], power))
        inside = [r for r in rows
                  if self.t0 is not None and self.t1 is not None and self.t0 <= r[0] <= self.t1]
        use = inside or rows
        if not use:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = {n for r in use for n, v in zip(names, r[3]) if v.lower() == "active"}
        powers = [r[4] for r in use if r[4] == r[4]]
        return {"sm_mhz": statistics.median(r[1] for r in use),
                "sm_max_mhz": max(r[2] for r in use), "reasons": sorted(reasons),
                "power_w": statistics.median(powers) if powers else None,
                "samples": len(use), "in_timed_window": bool(inside)}


# ------------------------------------------------------------------------------ reference arm

def oracle_sample_step(inp, n_tokens: int, step: int):
    """One oracle step on a token sample (different rows each step)."""
    import oracle

    T = inp.workload.T
    start = (step * n_tokens) % max(1, T - n_tokens + 1)
    sl = slice(start, start + n_tokens)
    oracle.flce(inp.x[sl], inp.weight, inp.target[sl], "mean")


def run_reference(args, wl, rank: int, world: int):
    if rank != 0:
        return
    inp = make_inputs(wl)
    n_tok = args.oracle_tokens
    for s in range(args.warmup):
        oracle_sample_step(inp, n_tok, s)
    t0 = time.perf_counter()
    for s in range(args.steps):
        oracle_sample_step(inp, n_tok, args.warmup + s)
    dt = time.perf_counter() - t0
    value = n_tok * args.steps / dt
    cores = os.cpu_count()
    sample = (f"{n_tok} tokens per step of {wl.name} (full H={wl.H}, V={wl.V}), float64 numpy "
              f"oracle forward+backward")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(wl, 0),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def workload_config(wl, n_slabs):
    return {"workload": wl.name, "tokens": wl.T, "hidden": wl.H, "vocab": wl.V,
            "dtype": wl.dtype, "targets": wl.target_dist, "reduction": "mean",
            "backward_vocab_slabs": n_slabs,
            "l2": "inputs larger than L2 (weight alone is %.2f GB > 129 MB)" % (
                wl.V * wl.H * (2 if wl.dtype == "bf16" else 4) / 1e9),
            "parallelism": "replicas"}


# ------------------------------------------------------------------------------ context

def torch_eager_context(x, w, y, steps: int = 3, warmup: int = 2):
    """Time the materialised-logits PyTorch formulation of one fwd+bwd step (context only)."""
    import torch

    T, V = x.shape[0], w.shape[0]
    need = T * V * (x.element_size() + 4 + 4 + 4)  # logits, fp32 copy, its grad, softmax
    free, _ = torch.cuda.mem_get_info()
    if need > 0.5 * free:
        return {"skipped": f"logits need ~{need / 1e9:.1f} GB"}
    xr = x.detach().clone().requires_grad_(True)
    wr = w.detach().clone().requires_grad_(True)

    def step():
        loss = torch.nn.functional.cross_entropy((xr @ wr.T).float(), y, reduction="mean")
        loss.backward()
        xr.grad = None
        wr.grad = None

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    return {"torch_eager_ms_per_step": ms, "torch_eager_tokens_per_s": T / (ms * 1e-3),
            "torch_eager_peak_mem_gb": torch.cuda.max_memory_allocated() / 1e9,
            "what": "bf16 x @ W^T (cuBLAS), fp32 logits, F.cross_entropy, autograd backward"}


# ------------------------------------------------------------------------------ our arm

def cpu_baseline(inp, n_tokens: int, min_seconds: float = 10.0):
    """The float64 oracle, as it stands, on successive samples of n_tokens token rows of the
    workload (from the first row on, wrapping around) until at least min_seconds have passed."""
    import oracle

    T = inp.workload.T
    n = min(n_tokens, T)
    start, done = 0, 0
    t0 = time.perf_counter()
    while True:
        sl = slice(start, start + n)
        oracle.flce(inp.x[sl], inp.weight, inp.target[sl], "mean")
        done += n
        start = start + n if start + 2 * n <= T else 0
        dt = time.perf_counter() - t0
        if dt >= min_seconds:
            break
    return {"value": done / dt, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{done} tokens of {inp.workload.name} in samples of {n} (full H, V), "
                      f"float64 numpy oracle forward+backward, {dt:.1f} s"}


def run_ours(args, wl, rank: int, world: int, dist):
    import torch

    from lm_head_linear_02_gb300 import autograd as A
    from lm_head_linear_02_gb300 import binding as B
    from lm_head_linear_02_gb300 import build as build_mod

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if not build_mod.up_to_date():
        raise RuntimeError("libflce.so is missing or stale: run __graft_entry__.build() first")
    B.lib()
    for name, value in args.tuning.items():
        B.flce_set_tuning(getattr(B, TUNING_KEYS[name]), value)

    t_gen = time.perf_counter()
    inp = make_inputs(wl)
    log(f"[rank {rank}] inputs generated in {time.perf_counter() - t_gen:.1f} s")
    T, H, V = wl.T, wl.H, wl.V
    dt_code = B.dtype_code(wl.dtype)
    tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    if wl.dtype == "bf16":
        hx = torch.from_numpy(inp.x_bits.view(np.int16)).view(torch.bfloat16)
        hw = torch.from_numpy(inp.weight_bits.view(np.int16)).view(torch.bfloat16)
    else:
        hx = torch.from_numpy(inp.x)
        hw = torch.from_numpy(inp.weight)
    hy = torch.from_numpy(inp.target)
    hx, hw, hy = hx.pin_memory(), hw.pin_memory(), hy.pin_memory()
    x = hx.to(dev)
    w = hw.to(dev)
    y = hy.to(dev)
    red = B.FLCE_REDUCTION_MEAN
    fwd_ws = B.flce_forward_workspace_size(T, H, V, dt_code)
    bwd_ws = B.flce_backward_workspace_size(T, H, V, dt_code)
    vc = B.flce_backward_slab_width(T, H, V, dt_code)
    n_slabs = math.ceil(V / vc)
    ws = torch.empty(max(fwd_ws, bwd_ws), dtype=torch.uint8, device=dev)
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    lse = torch.empty(T, dtype=torch.float32, device=dev)
    gl = torch.ones(1, dtype=torch.float32, device=dev)
    gx = torch.empty_like(x)
    gw = torch.empty_like(w)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream

    def step():
        B.flce_forward(x.data_ptr(), w.data_ptr(), y.data_ptr(), T, H, V, dt_code, red,
                       loss.data_ptr(), lse.data_ptr(), ws.data_ptr(), fwd_ws, status.data_ptr(),
                       sp)
        B.flce_backward(x.data_ptr(), w.data_ptr(), y.data_ptr(), lse.data_ptr(), T, H, V,
                        dt_code, red, gl.data_ptr(), gx.data_ptr(), gw.data_ptr(), ws.data_ptr(),
                        bwd_ws, status.data_ptr(), sp)

    def barrier():
        if dist is not None:
            dist.barrier()

    # warm-up
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    A.check_status(status)

    # ---- timed region (device-resident inputs)
    B.flce_timing_read()  # discard warm-up records
    B.flce_timing_enable(True)
    torch.cuda.reset_peak_memory_stats(dev)
    clocks = ClockSampler(local)
    clocks.start()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * args.steps + 1)]
    barrier()
    torch.cuda.synchronize(dev)
    clocks.begin()
    ev[0].record(stream)
    for k in range(args.steps):
        B.flce_forward(x.data_ptr(), w.data_ptr(), y.data_ptr(), T, H, V, dt_code, red,
                       loss.data_ptr(), lse.data_ptr(), ws.data_ptr(), fwd_ws, status.data_ptr(),
                       sp)
        ev[2 * k + 1].record(stream)
        B.flce_backward(x.data_ptr(), w.data_ptr(), y.data_ptr(), lse.data_ptr(), T, H, V,
                        dt_code, red, gl.data_ptr(), gx.data_ptr(), gw.data_ptr(), ws.data_ptr(),
                        bwd_ws, status.data_ptr(), sp)
        ev[2 * k + 2].record(stream)
    torch.cuda.synchronize(dev)
    clocks.end()
    barrier()
    clk = clocks.stop()
    B.flce_timing_enable(False)
    per_role = B.flce_timing_read()
    A.check_status(status)
    total_ms = ev[0].elapsed_time(ev[-1])
    fwd_ms = [ev[2 * k].elapsed_time(ev[2 * k + 1]) for k in range(args.steps)]
    bwd_ms = [ev[2 * k + 1].elapsed_time(ev[2 * k + 2]) for k in range(args.steps)]
    peak_mem = torch.cuda.max_memory_allocated(dev)
    total_ms = max_over_ranks(total_ms, dist, dev)

    # ---- single-call schedule (flce_forward_backward: no logits recompute), same inputs
    single = None
    if wl.dtype == "bf16" and not args.no_single_call:
        fb_ws = B.flce_forward_backward_workspace_size(T, H, V, dt_code)
        del ws  # the single call's peak memory excludes the two-call workspace
        torch.cuda.empty_cache()
        ws_fb = torch.empty(fb_ws, dtype=torch.uint8, device=dev)

        def single_step():
            B.flce_forward_backward(x.data_ptr(), w.data_ptr(), y.data_ptr(), T, H, V, dt_code,
                                    red, gl.data_ptr(), loss.data_ptr(), lse.data_ptr(),
                                    gx.data_ptr(), gw.data_ptr(), ws_fb.data_ptr(), fb_ws,
                                    status.data_ptr(), sp)

        for _ in range(args.warmup):
            single_step()
        torch.cuda.synchronize(dev)
        B.flce_timing_read()
        B.flce_timing_enable(True)
        torch.cuda.reset_peak_memory_stats(dev)
        barrier()
        torch.cuda.synchronize(dev)
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for _ in range(args.steps):
            single_step()
        s1.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
        B.flce_timing_enable(False)
        sroles = B.flce_timing_read()
        A.check_status(status)
        sms_ = s0.elapsed_time(s1)
        sms_ = max_over_ranks(sms_, dist, dev)
        s_ms = sms_ / args.steps
        single = {"ms_per_step": s_ms, "value": whole_job_rate(T, world, s_ms * 1e-3), "unit": UNIT,
                  "chunk_tokens": B.flce_forward_backward_chunk_tokens(T, H, V, dt_code),
                  "flops_per_step": roofline.flops(T, H, V, "model"),
                  "tensor_tflops": roofline.flops(T, H, V, "model") / (s_ms * 1e-3) / 1e12,
                  "roles_ms_per_step": {r: v[1] / args.steps for r, v in sroles.items() if v[0]},
                  "peak_mem_gb": torch.cuda.max_memory_allocated(dev) / 1e9,
                  "workspace_gb": fb_ws / 1e9}
        del ws_fb
        torch.cuda.empty_cache()
        ws = torch.empty(max(fwd_ws, bwd_ws), dtype=torch.uint8, device=dev)

    # ---- end-to-end: host-resident inputs, H2D copies + D2H loss read inside the timed region.
    # Every step copies its x, weight and target from pinned host memory and reads its loss
    # back; the copies of step k+1 run on a second stream into the other of two device input
    # sets while step k computes (the set is reused only after the step that read it is done).
    e2e_steps = max(2, min(args.steps, 20))
    bufs = [(x, w, y), (torch.empty_like(x), torch.empty_like(w), torch.empty_like(y))]
    copy_stream = torch.cuda.Stream(dev)
    h_loss = torch.empty(e2e_steps, dtype=torch.float32).pin_memory()
    copied = [torch.cuda.Event() for _ in range(e2e_steps)]
    done = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
    e2e_start = torch.cuda.Event(enable_timing=True)
    # device-side spans of each step's copies and compute (diagnostics for the e2e line)
    copy_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(e2e_steps)]
    comp_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(e2e_steps)]

    def enqueue_copy(k):
        xb, wb, yb = bufs[k % 2]
        with torch.cuda.stream(copy_stream):
            if k >= 2:
                copy_stream.wait_event(done[k - 2])
            copy_ev[k][0].record(copy_stream)
            xb.copy_(hx, non_blocking=True)
            wb.copy_(hw, non_blocking=True)
            yb.copy_(hy, non_blocking=True)
            copy_ev[k][1].record(copy_stream)
            copied[k].record(copy_stream)

    def run_step(xb, wb, yb):
        B.flce_forward(xb.data_ptr(), wb.data_ptr(), yb.data_ptr(), T, H, V, dt_code, red,
                       loss.data_ptr(), lse.data_ptr(), ws.data_ptr(), fwd_ws, status.data_ptr(),
                       sp)
        B.flce_backward(xb.data_ptr(), wb.data_ptr(), yb.data_ptr(), lse.data_ptr(), T, H, V,
                        dt_code, red, gl.data_ptr(), gx.data_ptr(), gw.data_ptr(), ws.data_ptr(),
                        bwd_ws, status.data_ptr(), sp)

    # untimed warm-up of both input sets (first use of the second set's memory)
    for xb, wb, yb in bufs:
        xb.copy_(hx, non_blocking=True)
        wb.copy_(hw, non_blocking=True)
        yb.copy_(hy, non_blocking=True)
        run_step(xb, wb, yb)
    barrier()
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    e2e_start.record(copy_stream)
    enqueue_copy(0)
    for k in range(e2e_steps):
        if k + 1 < e2e_steps:
            enqueue_copy(k + 1)
        stream.wait_event(copied[k])
        comp_ev[k][0].record(stream)
        run_step(*bufs[k % 2])
        comp_ev[k][1].record(stream)
        h_loss[k].copy_(loss[0], non_blocking=True)
        done[k].record(stream)
    torch.cuda.synchronize(dev)
    e2e_losses = h_loss.tolist()
    e2e_s = time.perf_counter() - t0
    e2e_s = max_over_ranks(e2e_s, dist, dev)
    if len(set(e2e_losses)) != 1:
        raise RuntimeError(f"end-to-end steps disagree: {e2e_losses}")
    # period of each step on the device: from the previous step's end (the start of the first
    # copy for step 0) to the step's end, loss read-back included
    e2e_period_ms = [e2e_start.elapsed_time(done[0])] + [
        done[k - 1].elapsed_time(done[k]) for k in range(1, e2e_steps)]
    e2e_copy_ms = [a.elapsed_time(b) for a, b in copy_ev]
    e2e_comp_ms = [a.elapsed_time(b) for a, b in comp_ev]
    del bufs
    A.check_status(status)
    if rank != 0:
        return

    # ---- roofline of the dominant kernel role
    peaks, peak_kind = load_peaks()
    peak_sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    peak_burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    if wl.dtype == "f32":
        # fp32 inputs run as three TF32 products per algorithmic FLOP (3xTF32): the peak is the
        # measured bf16 one times the nominal dense TF32/bf16 ratio (1.1 / 2.25 PFLOP/s), / 3
        peak_burst *= (1.1 / 2.25) / 3.0
        peak_sus *= (1.1 / 2.25) / 3.0
        peak_kind = peak_kind + ", TF32 = 1.1/2.25 of bf16, / 3 products per FLOP"
    # each role's algorithmic FLOPs per step: one T x H x V contraction, two for the launches
    # that run grad_weight and grad_x together
    role_flops = {r: args.steps * roofline.flops(T, H, V, "fwd") * (2 if r == "backward_grads" else 1)
                  for r in B.TIMING_ROLES}
    dom = max(per_role, key=lambda r: per_role[r][1])
    n_launch, ms_sum = per_role[dom]
    achieved = role_flops[dom] / (ms_sum * 1e-3) / 1e12
    traffic = recorded_traffic(dom, wl.name)
    ms_step = total_ms / args.steps
    step_tflops = roofline.flops(T, H, V, "fwd_bwd") / (ms_step * 1e-3) / 1e12
    # forward: projection kernel + combine + finalize; backward per slab: dz and one launch for
    # both gradients (bf16), or dz, grad_W and grad_x plus 6 TF32 operand splits (fp32).
    # Kernels of the library launched per step, from the contraction launches the timing hooks
    # counted: bf16 - projection, combine, finalize, then per vocab slab dz and one gradient
    # launch; fp32 - the x split, per weight slab a split and a projection, combine, finalize,
    # then two x splits and per vocab slab two weight splits, dz, grad_W and grad_x.
    fwd_launches = per_role["forward"][0] // args.steps
    if wl.dtype == "bf16":
        launches_per_step = fwd_launches + 2 + 2 * n_slabs
    else:
        launches_per_step = 1 + 2 * fwd_launches + 2 + 2 + 5 * n_slabs
    cpu = cpu_baseline(inp, args.oracle_tokens) if world == 1 else None
    context = None
    if world == 1 and not args.no_context:
        del ws
        torch.cuda.empty_cache()
        context = {"torch_eager": torch_eager_context(x, w, y)}
    pair_roles = B.flce_get_tuning(B.FLCE_TUNE_SM_PAIRS) if wl.dtype == "bf16" else 0
    wide_roles = B.flce_get_tuning(B.FLCE_TUNE_WIDE_TILES) & pair_roles
    out = {
        "metric": METRIC, "value": whole_job_rate(T * args.steps, world, total_ms * 1e-3),
        "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
        "data": "synthetic: seeded PCG64, x~N(0,1), weight~N(0,0.02^2), targets %s" % wl.target_dist,
        "config": dict(workload_config(wl, n_slabs),
                       sm_pair_roles=[n for n, b in (("forward", 1), ("dz", 2), ("grads", 4))
                                      if pair_roles & b],
                       wide_tile_roles=[n for n, b in (("forward", 1), ("dz", 2), ("grads", 4))
                                        if wide_roles & b],
                       tuning={name: B.flce_get_tuning(getattr(B, key))
                               for name, key in TUNING_KEYS.items() if name != "sm_pairs"}),
        "fwd_ms": statistics.median(fwd_ms), "bwd_ms": statistics.median(bwd_ms),
        "fwd_tokens_per_s": T / (statistics.median(fwd_ms) * 1e-3),
        "tensor_tflops_step": step_tflops,
        "tensor_frac_of_measured": {"burst": step_tflops / peak_burst,
                                     "sustained": step_tflops / peak_sus,
                                     "peaks_source": peak_kind},
        "flops_per_step": roofline.flops(T, H, V, "fwd_bwd"),
        "roles_ms_per_step": {r: per_role[r][1] / args.steps for r in per_role if per_role[r][0]},
        "roofline": {"bound": "tensor", "kernel": f"k_umma_gemm ({dom})",
                     "achieved": achieved, "peak": peak_burst, "unit": "TFLOP/s",
                     "frac": achieved / peak_burst, "traffic": traffic,
                     "peak_sustained": peak_sus, "frac_sustained": achieved / peak_sus,
                     "algorithmic_flops_per_launch": role_flops[dom] / n_launch,
                     "ms_per_launch": ms_sum / n_launch, "launches": n_launch,
                     "peak_source": f"bf16_tflops (burst) of {peak_kind}; frac_sustained against "
                                    f"bf16_tflops_sustained of {peak_kind}"},
        "cpu_baseline": cpu,
        "e2e": {"value": whole_job_rate(T * e2e_steps, world, e2e_s), "unit": UNIT,
                "steps": e2e_steps, "overlap": "H2D of step k+1 on a copy stream during step k",
                "wall_ms_per_step": e2e_s * 1e3 / e2e_steps,
                "median_wall_ms_per_step": statistics.median(e2e_period_ms),
                "median_value": T / (statistics.median(e2e_period_ms) * 1e-3) * world,
                "period_ms_steps": [round(v, 3) for v in e2e_period_ms],
                "copy_ms_per_step": statistics.median(e2e_copy_ms),
                "compute_ms_per_step": statistics.median(e2e_comp_ms),
                "compute_ms_steps": [round(v, 3) for v in e2e_comp_ms],
                "copy_ms_steps": [round(v, 3) for v in e2e_copy_ms],
                "gap_ms_steps": [round(comp_ev[k][1].elapsed_time(comp_ev[k + 1][0]), 3)
                                 for k in range(e2e_steps - 1)],
                "h2d_bytes_per_step": int(hx.numel() * hx.element_size() +
                                          hw.numel() * hw.element_size() + hy.numel() * 8),
                "d2h_bytes_per_step": 4},
        "clocks": clk,
        "gpu_launches": launches_per_step * args.steps,
        "peak_mem_gb": peak_mem / 1e9,
        "workspace_gb": max(fwd_ws, bwd_ws) / 1e9,
        "logits_bf16_gb": 2 * T * V / 1e9,
        "context": context,
        "single_call": single,
    }
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--no-single-call", action="store_true",
                    help="skip timing the single-call (no recompute) schedule")
    ap.add_argument("--no-context", action="store_true",
                    help="skip the PyTorch eager context measurement")
    ap.add_argument("--oracle-tokens", type=int, default=64,
                    help="token sample per oracle step (CPU baseline / reference arm)")
    ap.add_argument("--tune", action="append", default=[], metavar="NAME=VALUE",
                    help="set a libflce tuning key before timing (repeatable): " +
                         ", ".join(sorted(TUNING_KEYS)))
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    try:
        args.tuning = parse_tuning(args.tune)
    except ValueError as exc:
        ap.error(str(exc))
    wl = WORKLOADS[args.workload]

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if world > 1 and args.impl == "ours":
        import torch
        import torch.distributed as tdist

        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        tdist.init_process_group("nccl")
        dist = tdist
    try:
        if args.impl == "reference":
            run_reference(args, wl, rank, world)
        else:
            run_ours(args, wl, rank, world, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
