"""Benchmark of the vocab-parallel cross-entropy forward + backward on GB300.

One step = vpce_forward (partial statistics + combine) and vpce_backward (dlogits
in place) over one batch of seeded synthetic logits: s = 8192 rows,
V = 128256 (t = 8 shards of 16032 columns, bf16), N(0, 3^2) with +5 on the
target column of 30% of rows -- the Llama-3-70B LM-head shape.

Prints one JSON line (rank 0).  `value` is tokens/s over all ranks; the line
also carries the 3-pass HBM GB/s, the roofline of the dominant kernel, the
end-to-end number with host buffers, the clocks seen during the timed region,
and (rank 0, N = 1) the fp64 CPU oracle timed on a bounded sample.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
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
# NCCL prints its version banner on stdout at communicator set-up; the bench
# prints exactly one JSON line there (a caller's own setting wins)
os.environ.setdefault("NCCL_DEBUG", "WARN")
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from vocab_sharded_lm_gb300 import synth  # noqa: E402

METRIC = "VPCE fwd+bwd tokens/s & HBM GB/s (% of peak), s=8192 V=128256 bf16, 1 GB300"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0


def _tensor_peaks():
    """(burst, sustained, kind) dense bf16 TFLOP/s."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d["bf16_tflops_sustained"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, FALLBACK_BF16_TFLOPS_SUSTAINED, "fallback"


def _env_rank():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def _workload_desc(w):
    return (f"{w.name}: s={w.s} V={w.V} t={w.t} x {w.V // w.t} {w.dtype} logits ~N(0,{w.sigma:g}^2)"
            + (f", +{w.boost:g} on the target of {int(w.boost_frac * 100)}% of rows" if w.boost_frac else "")
            + (f", {int(w.ignore_frac * 100)}% ignore_index" if w.ignore_frac else "")
            + (f", +{w.spike:g} spike per row" if w.spike else "")
            + f", targets {w.targets}")


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.out = None

    def start(self):
        try:
            self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50",
                 "-i", str(self.dev)], stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.flush()
        self.out.seek(0)
        rows = [l.strip().split(", ") for l in self.out.read().splitlines() if l.strip()]
        self.out.close()
        os.unlink(self.out.name)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax = float(r[2])
                for n, v in zip(names, r[5:9]):
                    if v.strip() == "Active":
                        reasons.add(n)
            except (ValueError, IndexError):
                continue
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------
# traffic recorded by ncu for the dominant kernel (per launch), if still current
# ----------------------------------------------------------------------------
# the source file of each kernel whose ncu traffic is recorded; the shared
# device headers count for all of them
# each kernel's source file and the headers it includes beyond the shared ones
_KERNEL_FILES = {"stream_fused_kernel": ("vpce_fused.cu",), "backward_kernel": ("vpce_backward.cu",),
                 "partial_stats_kernel": ("vpce_forward.cu",), "gemm_stats_kernel": ("vpce_gemm.cu", "vpce_tc.cuh"),
                 "gemm_bwd_kernel": ("vpce_gemm_bwd.cu", "vpce_tc.cuh")}


def _kernel_source_hash(kernel: str) -> str:
    """Hash of the code (comments removed, whitespace runs collapsed) of a
    kernel's source file and the headers it includes: an edit of comments or
    layout keeps its stored counters."""
    h = hashlib.sha256()
    for f in ("vpce_device.cuh", "vpce_kernels.cuh", "vpce_chunk.cuh", *_KERNEL_FILES[kernel]):
        with open(os.path.join(ROOT, "vocab_sharded_lm_gb300", "csrc", f), encoding="utf-8") as fh:
            code = re.sub(r"/\*.*?\*/", "", fh.read(), flags=re.S)
        code = re.sub(r"\s+", " ", re.sub(r"//[^\n]*", "", code))
        h.update(code.encode())
    return h.hexdigest()[:16]


def _ncu_traffic(kernel: str, workload: str):
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except Exception:
        return None
    ent = d.get(kernel, {}).get(workload)
    if not ent or ent.get("source_hash") != _kernel_source_hash(kernel):
        return None
    return ent.get("dram_bytes_per_launch")


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------
def _bind_to_gpu_cpus(dev) -> None:
    """Restrict this process to the host CPUs local to the GPU (from sysfs),
    so that pinned host buffers land on the memory node next to it.  No-op
    where the information is missing."""
    import torch

    try:
        pr = torch.cuda.get_device_properties(dev)
        bus = f"{pr.pci_domain_id:04x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0"
        with open(f"/sys/bus/pci/devices/{bus}/local_cpulist") as f:
            spec = f.read().strip()
        cpus = set()
        for part in spec.split(","):
            lo, _, hi = part.partition("-")
            cpus.update(range(int(lo), int(hi or lo) + 1))
        if cpus:
            os.sched_setaffinity(0, cpus)
    except (OSError, ValueError, AttributeError):
        pass


def _max_over_ranks(x: float, device=None) -> float:
    """The largest x over the ranks of the default process group (x itself
    without one).  `device` holds the collective's tensor: a CUDA device for
    NCCL, None (host) for gloo."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _weak_scaling_value(units_per_rank: int, world: int, max_ms: float) -> float:
    """Whole-job throughput: the units all ranks processed over the slowest
    rank's time."""
    return world * units_per_rank / (max_ms * 1e-3)


def run_ours(args):
    import torch
    import torch.distributed as dist

    from vocab_sharded_lm_gb300 import _build, vpce

    rank, world, local = _env_rank()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    _build.build()
    vpce.load_library()

    w = synth.WORKLOADS[args.workload]
    if args.rows:
        w = w.replace(s=args.rows)  # smaller batch of the same shard geometry (profiling captures)
    # every rank runs its own batch (independent problems, weak scaling)
    if world > 1:
        w = w.replace(index=w.index + 100 * rank) if rank else w
    meta = synth.row_meta(w)
    vs = synth.even_vocab_start(w.V, w.t)
    e = w.elem_bytes
    buf_bytes = w.s * w.V * e
    free, _ = torch.cuda.mem_get_info(dev)
    nbuf = max(2, min(args.warmup + args.steps, int(0.5 * free // buf_bytes), args.max_buffers))

    pristine = synth.device_shards(w, meta, vs, device=dev)
    bufs = [[p.clone() for p in pristine] for _ in range(nbuf)]
    y = torch.from_numpy(meta.targets).to(dev)
    ws = [vpce.new_workspace(w.t, w.s, dev) for _ in range(2)]
    loss = torch.empty((), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    fused = args.path == "fused"

    def run_step(b, yy, wk):
        if fused:
            vpce.vpce_forward_backward(b, yy, vs, ignore_index=w.ignore_index, loss_out=loss, workspace=wk)
        else:
            vpce.vpce_forward(b, yy, vs, ignore_index=w.ignore_index, loss_out=loss, workspace=wk)
            vpce.vpce_backward(b, yy, wk, vs, ignore_index=w.ignore_index)

    def step(k, ev=None):
        b = bufs[k % nbuf]
        wk = ws[k % 2]
        if ev is not None:
            ev[0].record(stream)
        if fused:
            vpce.vpce_forward_backward(b, y, vs, ignore_index=w.ignore_index, loss_out=loss, workspace=wk)
            if ev is not None:
                ev[1].record(stream)
        else:
            vpce.vpce_forward(b, y, vs, ignore_index=w.ignore_index, loss_out=loss, workspace=wk)
            if ev is not None:
                ev[1].record(stream)
            vpce.vpce_backward(b, y, wk, vs, ignore_index=w.ignore_index)
        if ev is not None:
            ev[2].record(stream)

    for k in range(args.warmup):
        step(k)
    torch.cuda.synchronize(dev)
    # restore every buffer so that the timed steps start from generated logits
    for b in bufs:
        for d, p in zip(b, pristine):
            d.copy_(p)
    torch.cuda.synchronize(dev)

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t0.record(stream)
    for k in range(args.steps):
        step(k, evs[k])
    t1.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    total_ms = t0.elapsed_time(t1)
    fwd_ms = [ev[0].elapsed_time(ev[1]) for ev in evs]
    bwd_ms = [ev[1].elapsed_time(ev[2]) for ev in evs]
    total_ms = _max_over_ranks(total_ms, dev)

    # ---------------- end to end through the public API: every step copies its
    # logits and targets from pinned host memory and reads its loss back.
    # Two device input buffers on a copy stream, so the next step's copy runs
    # while the current step computes (dlogits stay on the device, where the
    # LM-head backward consumes them).
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    _bind_to_gpu_cpus(dev)  # pinned buffers on the GPU's own host memory node
    host_in = [p.cpu().pin_memory() for p in pristine]
    host_y = torch.from_numpy(meta.targets).pin_memory()
    host_loss = torch.empty(e2e_steps, dtype=torch.float32).pin_memory()
    dbufs = [bufs[0], bufs[1 % nbuf]]
    ydevs = [torch.empty_like(y), torch.empty_like(y)]
    losses = [torch.empty((), dtype=torch.float32, device=dev) for _ in range(2)]
    copy_stream = torch.cuda.Stream(dev)
    h2d_done = [torch.cuda.Event() for _ in range(2)]
    used = [torch.cuda.Event() for _ in range(2)]
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    warm = 2  # untimed: the first copies from freshly pinned pages are slow
    for k in range(-warm, e2e_steps):
        if k == 0:
            stream.synchronize()
            copy_stream.synchronize()
            e0.record(copy_stream)
        b = k % 2
        with torch.cuda.stream(copy_stream):
            if k >= 2 - warm:
                copy_stream.wait_event(used[b])
            for d, h in zip(dbufs[b], host_in):
                d.copy_(h, non_blocking=True)
            ydevs[b].copy_(host_y, non_blocking=True)
            h2d_done[b].record(copy_stream)
        stream.wait_event(h2d_done[b])
        if fused:
            vpce.vpce_forward_backward(dbufs[b], ydevs[b], vs, ignore_index=w.ignore_index, loss_out=losses[b],
                                       workspace=ws[b])
        else:
            vpce.vpce_forward(dbufs[b], ydevs[b], vs, ignore_index=w.ignore_index, loss_out=losses[b],
                              workspace=ws[b])
            vpce.vpce_backward(dbufs[b], ydevs[b], ws[b], vs, ignore_index=w.ignore_index)
        host_loss[max(k, 0)].copy_(losses[b], non_blocking=True)
        used[b].record(stream)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = _max_over_ranks(e0.elapsed_time(e1) / e2e_steps, dev)
    h2d = buf_bytes + w.s * 8
    d2h = 4

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    peak, peak_kind = _peaks()
    ms_step = total_ms / args.steps
    tokens_s = _weak_scaling_value(w.s * args.steps, world, total_ms)
    n_valid = int(np.sum(meta.targets != w.ignore_index))
    three_pass = 3 * w.s * w.V * e
    gbs_3pass = three_pass / (ms_step * 1e-3) / 1e9
    # algorithmic HBM bytes of the in-place gradient writer: read + write of
    # every valid row's logits, ignored rows written only, plus the per-row
    # target (8 B) and logsumexp (4 B)
    grad_bytes = (2 * n_valid + (w.s - n_valid)) * w.V * e + w.s * 12
    fwd_bytes = n_valid * w.V * e + w.s * (8 + 8 * w.t + 4)
    fwd_mean_ms = statistics.mean(fwd_ms)
    bwd_mean_ms = statistics.mean(bwd_ms) if not fused else None
    if fused:
        # dominant (only) kernel pair: prologue + fused forward/backward, whose
        # HBM floor is one read and one write of the logits
        dom_kernel, dom_ms, dom_bytes = "stream_fused_kernel", fwd_mean_ms, grad_bytes
    else:
        dom_kernel, dom_ms, dom_bytes = "backward_kernel", bwd_mean_ms, grad_bytes
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    traffic = _ncu_traffic(dom_kernel, w.name)
    out = {
        "metric": METRIC,
        "value": round(tokens_s, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        # the arithmetic type of the path: logits of logits_dtype are widened
        # to fp32, reduced in fp32 (fp64 batch sum) and dlogits rounded back
        "dtype": "f32",
        "data": "synthetic (seeded counter-based generator; no dataset)",
        "config": {
            "workload": _workload_desc(w),
            "global_batch": w.s * world,
            "seq_len": w.s,
            "logits_dtype": w.dtype,
            "arithmetic": f"{w.dtype} logits in, fp32 arithmetic, {w.dtype} dlogits out",
            "parallelism": f"vocab shards t={w.t} on one GPU; {world} independent replica(s)",
            "l2": f"inputs larger than L2: each step's logits are {buf_bytes / 1e9:.2f} GB, "
                  f"{nbuf} distinct buffers cycled (beyond {nbuf} steps a buffer holds the previous "
                  f"pass's dlogits: same shape and work)",
            "path": ("vpce_forward_backward (fused: stats warps stream each row from HBM, grad warps "
                     "re-read it from L2 a row later; about 1 HBM read + 1 HBM write of the logits)") if fused else
                    "vpce_forward + vpce_backward (split, 3 logit passes)",
        },
        "hbm_gbs_3pass": round(gbs_3pass, 1),
        "hbm_frac_nominal_8000": round(gbs_3pass / NOMINAL_HBM_GBS, 4),
        "hbm_frac_measured_peak": round(gbs_3pass / peak, 4),
        "fwd_ms": None if fused else round(fwd_mean_ms, 5),
        "bwd_ms": None if fused else round(bwd_mean_ms, 5),
        "fused_ms": round(fwd_mean_ms, 5) if fused else None,
        "fwd_gbs": None if fused else round(fwd_bytes / (fwd_mean_ms * 1e-3) / 1e9, 1),
        "hbm_gbs_floor_fused": round(2 * w.s * w.V * e / (ms_step * 1e-3) / 1e9, 1) if fused else None,
        "roofline": {
            "kernel": dom_kernel,
            "bound": "hbm",
            "achieved": round(achieved, 1),
            "peak": peak,
            "peak_kind": peak_kind,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": traffic,
            "algorithmic_bytes_per_launch": dom_bytes,
        },
        "e2e": {
            "value": round(_weak_scaling_value(w.s, world, e2e_ms), 1),
            "unit": "tokens/s",
            "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "steps": e2e_steps,
            "ms_per_step": round(e2e_ms, 4),
            "note": "pinned host logits + targets copied in every step (copy stream, double-buffered), "
                    "loss read back; dlogits stay on the device",
        },
        "gpu_launches": (2 if fused else 3) * args.steps,
        "clocks": clk,
    }
    if fused:
        out["config"]["fused_plan"] = vpce.vpce_fused_plan(
            vpce.VPCE_BF16 if w.dtype == "bf16" else vpce.VPCE_FP32, vs, w.s)
    if world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"], out["cpu_baseline_one_core"] = cpu_baseline(
            w, meta, vs, budget_s=args.cpu_seconds, wl=args.workload, s_override=args.rows)
    print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()


# ----------------------------------------------------------------------------
# the pages' multi-card method: the vocabulary split over the processes
# ----------------------------------------------------------------------------
DISTRIBUTED_METRIC = "VPCE fwd+bwd tokens/s, vocabulary split over N processes (one GPU each), s=8192 V=128256 bf16"


def _free_port() -> int:
    import socket

    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def run_distributed(args, backend=None, device: str = "cuda", emit=print):
    """One shared batch whose vocabulary is split over the N processes ("Distributed
    Training III: Model Parallelism", CMU 11-868 Lecture 16 notes, §5.5; "LLM
    Internals" §7.3.4): rank r holds shards [r t/N, (r+1) t/N) of the workload's t.
    A step is distributed.forward (local partial statistics, the rank's shards
    folded to one (max, sum exp) pair per row, one all-gather of the pairs, one
    all-reduce of the target logits, the combine on every rank) and
    distributed.backward (dlogits in place, no communication).  The batch is
    the same on every rank, so the work per rank shrinks as N grows (strong
    scaling); tokens/s counts each token once.  ``backend`` and ``device='cpu'``
    let the orchestration run on CPU ranks over gloo (tests); the GPU run uses
    the library's kernels and NCCL."""
    import torch
    import torch.distributed as dist

    from vocab_sharded_lm_gb300 import distributed

    rank, world, local = _env_rank()
    cpu = device == "cpu"
    own_group = False
    if not dist.is_initialized():
        if world == 1:
            # a group of one, so that the exchange runs as written
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            os.environ.setdefault("MASTER_PORT", str(_free_port()))
            dist.init_process_group("gloo" if cpu else "nccl", rank=0, world_size=1)
        else:
            dist.init_process_group("gloo" if cpu else "nccl")
        own_group = True
    if cpu:
        dev = torch.device("cpu")
    else:
        from vocab_sharded_lm_gb300 import _build, vpce

        torch.cuda.set_device(local)
        dev = torch.device("cuda", local)
        _build.build()
        vpce.load_library()

    w = synth.WORKLOADS[args.workload]
    if args.rows:
        w = w.replace(s=args.rows)
    if w.t % world:
        if rank == 0:
            emit(json.dumps({"metric": DISTRIBUTED_METRIC, "unavailable":
                             f"{w.t} shards do not split evenly over {world} processes"}))
        if own_group:
            dist.destroy_process_group()
        return
    per = w.t // world
    vs = synth.even_vocab_start(w.V, w.t)
    vs_local = vs[rank * per:(rank + 1) * per + 1]
    meta = synth.row_meta(w)  # one batch, the same targets on every rank
    e = w.elem_bytes
    slice_bytes = w.s * (vs_local[-1] - vs_local[0]) * e
    if cpu:
        host = synth.shards_host(w, meta, vs_local)
        pristine = [torch.from_numpy(h.astype(np.float32) if w.dtype == "fp32" else h) for h in host]
        nbuf = 2
    else:
        pristine = synth.device_shards(w, meta, vs_local, device=dev)
        free, _ = torch.cuda.mem_get_info(dev)
        nbuf = max(2, min(args.warmup + args.steps, int(0.5 * free // max(slice_bytes, 1)), args.max_buffers))
    bufs = [[p.clone() for p in pristine] for _ in range(nbuf)]
    y = torch.from_numpy(meta.targets).to(dev)
    be = backend or distributed.CudaBackend()
    ws = [be.new_workspace(per, w.s, dev) for _ in range(2)]
    last = {}

    def step(k):
        b = bufs[k % nbuf]
        loss, _, wk = distributed.forward(b, vs_local, y, w.V, ignore_index=w.ignore_index, backend=be,
                                          workspace=ws[k % 2])
        distributed.backward(b, vs_local, y, wk, ignore_index=w.ignore_index, backend=be)
        last["loss"] = loss

    for k in range(args.warmup):
        step(k)
    for b in bufs:  # the timed steps start from generated logits
        for d, p_ in zip(b, pristine):
            d.copy_(p_)
    coll_dev = None if cpu else dev
    clocks = None if cpu else ClockSampler(local)
    if clocks is not None:
        clocks.start()
    dist.barrier()
    if cpu:
        t_start = time.perf_counter()
        for k in range(args.steps):
            step(k)
        total_ms = (time.perf_counter() - t_start) * 1e3
    else:
        stream = torch.cuda.current_stream(dev)
        torch.cuda.synchronize(dev)
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for k in range(args.steps):
            step(k)
        t1.record(stream)
        torch.cuda.synchronize(dev)
        total_ms = t0.elapsed_time(t1)
    dist.barrier()
    clk = clocks.stop() if clocks is not None else None
    total_ms = _max_over_ranks(total_ms, coll_dev)
    loss_v = float(last["loss"])

    # end to end: every step copies this rank's logits slice and the targets
    # in from pinned host memory and reads the loss back
    if cpu:
        e2e_ms, h2d, d2h = total_ms / args.steps, 0, 0
    else:
        e2e_steps = max(1, min(args.steps, args.e2e_steps))
        host_in = [p_.cpu().pin_memory() for p_ in pristine]
        host_y = torch.from_numpy(meta.targets).pin_memory()
        host_loss = torch.empty(e2e_steps, dtype=torch.float32).pin_memory()
        torch.cuda.synchronize(dev)
        dist.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for k in range(e2e_steps):
            b = bufs[k % nbuf]
            for d, h in zip(b, host_in):
                d.copy_(h, non_blocking=True)
            y.copy_(host_y, non_blocking=True)
            step(k)
            host_loss[k].copy_(last["loss"].reshape(()), non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = _max_over_ranks(e0.elapsed_time(e1) / e2e_steps, coll_dev)
        h2d, d2h = slice_bytes + w.s * 8, 4
    if rank != 0:
        if own_group:
            dist.destroy_process_group()
        return
    ms_step = total_ms / args.steps
    out = {
        "metric": DISTRIBUTED_METRIC,
        "value": round(w.s * args.steps / (total_ms * 1e-3), 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "strong",
        "vs_baseline": None,
        # logits of logits_dtype widened to fp32 for the arithmetic
        "dtype": "f32",
        "data": "synthetic (seeded counter-based generator; no dataset)",
        "config": {
            "workload": _workload_desc(w),
            "global_batch": w.s,
            "seq_len": w.s,
            "logits_dtype": w.dtype,
            "parallelism": f"vocabulary split: {world} process(es) x {per} of the {w.t} shards, one shared batch",
            "path": "distributed.forward + distributed.backward: vpce_partials, vpce_fold_partials, all_gather of "
                    "one (max, sum exp) pair per row and rank, all_reduce of the target logits, "
                    "vpce_combine_partials, vpce_backward",
            "backend": "gloo, CPU ranks" if cpu else "NCCL",
        },
        "exchange": {
            # what one rank puts on the wire per step: its folded pair per row
            # (all-gather) and its target-logit vector (all-reduce) -- the
            # pages' three fp32 scalars per token
            "bytes_sent_per_rank": 12 * w.s if world > 1 else 0,
            "bytes_per_token": 12,
        },
        "loss": loss_v,
        "e2e": {
            "value": round(w.s / (e2e_ms * 1e-3), 1),
            "unit": "tokens/s",
            "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "ms_per_step": round(e2e_ms, 4),
        },
        # vpce_partials, vpce_fold_partials, vpce_combine_partials and vpce_backward:
        # one kernel each (the collectives are NCCL's)
        "gpu_launches": 0 if cpu else 4 * args.steps,
        "clocks": clk,
    }
    emit(json.dumps(out))
    if own_group:
        dist.destroy_process_group()


# ----------------------------------------------------------------------------
# the fp64 oracle on the host cores: CPU baseline and the reference arm
# ----------------------------------------------------------------------------
class _RowPool:
    """A fixed, seeded pool of rows of the workload (host copies, generated
    once); oracle steps draw their samples from it."""

    def __init__(self, w, meta, vs, size=64, seed=1):
        from oracle import vpce_oracle as O

        rng = np.random.default_rng(seed)
        self.O = O
        self.rows = np.sort(rng.choice(w.s, size=min(size, w.s), replace=False))
        self.host = [synth.logits_rows(w, self.rows, vs[i], vs[i + 1], meta) for i in range(w.t)]
        self.y = meta.targets[self.rows]
        self.w, self.vs = w, vs
        self.n_valid = int(np.sum(meta.targets != w.ignore_index))
        self.cursor = 0

    def step(self, k: int) -> None:
        """Oracle loss + dlogits of the next k rows of the pool (cyclic)."""
        idx = (self.cursor + np.arange(k)) % len(self.rows)
        self.cursor = (self.cursor + k) % len(self.rows)
        z = self.O.assemble([h[idx] for h in self.host], self.vs, self.w.dtype)
        ref = self.O.cross_entropy(z, self.y[idx], self.w.ignore_index, n_valid=self.n_valid)
        self.O.dlogits(z, self.y[idx], self.w.ignore_index, n_valid=self.n_valid, lse=ref["lse"])


def _oracle_worker(job):
    """One host core's share of an oracle timing, in a spawned process (host
    only, no CUDA): builds its own seeded row pool, runs `warmup` untimed steps,
    waits for the common start time `t_start` (wall clock) so that every core
    is busy while any core is timed, then runs `steps` timed steps of `rows`
    rows (or, with steps = 0, as many as fit in `budget_s`).  Returns
    (rows timed, seconds)."""
    wl, s_override, seed, rows, warmup, steps, budget_s, t_start = job
    w = synth.WORKLOADS[wl]
    if s_override:
        w = w.replace(s=s_override)
    meta = synth.row_meta(w)
    vs = synth.even_vocab_start(w.V, w.t)
    pool = _RowPool(w, meta, vs, seed=seed)
    for _ in range(warmup):
        pool.step(rows)
    delay = t_start - time.time()
    if delay > 0:
        time.sleep(delay)
    done, t0 = 0, time.perf_counter()
    while (done < steps * rows) if steps else (time.perf_counter() - t0 < budget_s):
        pool.step(rows)
        done += rows
    return done, time.perf_counter() - t0


def _host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _oracle_all_cores(wl, s_override, rows, warmup, steps, budget_s, margin_s):
    """The oracle on every host core at once: one spawned worker per core (a
    fresh interpreter, safe after CUDA has been initialised here), each with
    single-threaded numpy.  Returns (rows/s summed over the workers, workers,
    [(rows, seconds)])."""
    import concurrent.futures as cf
    import multiprocessing as mp

    n = _host_cores()
    keys = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")
    saved = {k: os.environ.get(k) for k in keys}
    for k in keys:
        os.environ[k] = "1"
    try:
        t_start = time.time() + margin_s
        jobs = [(wl, s_override, 1 + i, rows, warmup, steps, budget_s, t_start) for i in range(n)]
        with cf.ProcessPoolExecutor(max_workers=n, mp_context=mp.get_context("spawn")) as ex:
            res = list(ex.map(_oracle_worker, jobs))
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    return sum(d / t for d, t in res), n, res


def cpu_baseline(w, meta, vs, budget_s=10.0, rows_per_batch=16, wl=None, s_override=0):
    """The oracle on the host: on one core, then on every core at once (the
    reported figure)."""
    t0 = time.perf_counter()
    pool = _RowPool(w, meta, vs)
    build_s = time.perf_counter() - t0
    done = 0
    elapsed = 0.0
    while elapsed < budget_s:
        t0 = time.perf_counter()
        pool.step(rows_per_batch)
        elapsed += time.perf_counter() - t0
        done += rows_per_batch
    one = done / elapsed
    rate, n, res = _oracle_all_cores(wl or w.name, s_override, rows_per_batch, 1, 0, budget_s,
                                     margin_s=5.0 + 4.0 * build_s)
    rows_all = sum(d for d, _ in res)
    return ({"value": round(rate, 2), "unit": "tokens/s", "cores": n, "kind": "oracle",
             "sample": f"{rows_all} rows of the workload over {n} spawned single-threaded workers (each a seeded "
                       f"pool of {len(pool.rows)} rows, batches of {rows_per_batch}, full V={w.V}), fp64 numpy, "
                       f"forward loss + dlogits, {budget_s:.0f} s each, all cores busy at once"},
            {"value": round(one, 2), "unit": "tokens/s", "cores": 1, "kind": "oracle",
             "sample": f"{done} rows on one core, {elapsed:.1f} s"})


def run_reference(args):
    rank, world, _ = _env_rank()
    if rank != 0:
        return
    w = synth.WORKLOADS[args.workload]
    if args.rows:
        w = w.replace(s=args.rows)
    meta = synth.row_meta(w)
    vs = synth.even_vocab_start(w.V, w.t)
    t0 = time.perf_counter()
    pool = _RowPool(w, meta, vs)
    build_s = time.perf_counter() - t0
    # rows per step and core: about 45 s of timed work per core in total
    t0 = time.perf_counter()
    pool.step(1)
    per_row = time.perf_counter() - t0
    rows_per_step = int(max(1, min(args.ref_rows, 45.0 / max(args.steps * per_row, 1e-9))))
    # every host core runs the oracle at once, one spawned worker per core,
    # each its own W untimed and K timed steps
    value, n, res = _oracle_all_cores(args.workload, args.rows, rows_per_step, args.warmup, args.steps, 0.0,
                                      margin_s=5.0 + 4.0 * build_s + args.warmup * rows_per_step * per_row)
    dt = max(t for _, t in res)
    out = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded counter-based generator; no dataset)",
        "config": {"workload": _workload_desc(w), "global_batch": w.s, "seq_len": w.s,
                   "logits_dtype": w.dtype,
                   "parallelism": "fp64 CPU oracle (the pages print no code, so there is no reference "
                                  "implementation to install)",
                   "sample": f"{rows_per_step} rows per step and core, {n} cores, each from a seeded pool of "
                             f"{len(pool.rows)} rows, full V={w.V}"},
        "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "cores": n, "kind": "oracle",
                         "sample": f"{rows_per_step} rows of the workload per step on each of {n} spawned "
                                   f"single-threaded workers, fp64 numpy, all cores busy at once"},
        "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


# ----------------------------------------------------------------------------
# the LM-head GEMM fused with the forward loss (vpce_lmhead_forward)
# ----------------------------------------------------------------------------
LMHEAD_METRIC = "LM-head GEMM + VPCE forward tokens/s & TFLOP/s (% of peak), s=8192 h=8192 V=128256 bf16, 1 GB300"
LMHEAD_TRAIN_METRIC = ("LM-head GEMM + VPCE forward and backward (dX, dW) tokens/s & TFLOP/s (% of peak), "
                       "s=8192 h=8192 V=128256 bf16, 1 GB300")


def run_lmhead(args):
    import torch

    from vocab_sharded_lm_gb300 import _build, vpce
    from oracle import vpce_oracle as O

    rank, world, local = _env_rank()
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    _build.build()
    vpce.load_library()
    m = synth.LMHEADS[synth.LMHEAD_BENCH]
    if args.rows:
        m = m.replace(s=args.rows)
    if args.vocab:  # a smaller head of the same hidden size (profiling captures that hold a few GB)
        m = m.replace(V=args.vocab, t=args.shards or m.t)
    vs = synth.even_vocab_start(m.V, m.t)
    meta = synth.lmhead_meta(m)
    x, ws = synth.lmhead_device(m, vs, device=dev)
    y = torch.from_numpy(meta.targets).to(dev)
    wk = torch.empty(vpce.vpce_lmhead_workspace_bytes(m.s), dtype=torch.uint8, device=dev)
    loss = torch.empty((), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    train = args.path == "lmhead_train"
    if train:
        gx = torch.empty_like(x)
        gw = [torch.zeros((w.shape[0], m.h), dtype=torch.float32, device=dev) for w in ws]
        twk = torch.empty(vpce.vpce_lmhead_forward_backward_workspace_bytes(m.s, m.V, m.h), dtype=torch.uint8,
                          device=dev)

    def call(xi, yi, li, wki):
        if train:
            vpce.vpce_lmhead_forward_backward(xi, ws, yi, vs, ignore_index=m.ignore_index, loss_out=li,
                                              grad_hidden=gx, grad_weight_shards=gw, workspace=twk)
        else:
            vpce.vpce_lmhead_forward(xi, ws, yi, vs, ignore_index=m.ignore_index, loss_out=li, workspace=wki)

    def step():
        call(x, y, loss, wk)

    for _ in range(args.warmup):
        step()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for k in range(args.steps):
        evs[k][0].record(stream)
        step()
        evs[k][1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    total_ms = _max_over_ranks(t0.elapsed_time(t1), dev)
    call_ms = statistics.mean(a.elapsed_time(b) for a, b in evs)

    # end to end: the step's hidden states (and targets) copied in from pinned
    # host memory, the loss read back; the head's weights stay on the device
    hx = x.cpu().pin_memory()
    hy = torch.from_numpy(meta.targets).pin_memory()
    xb = [x, torch.empty_like(x)]
    yb = [y, torch.empty_like(y)]
    lb = [torch.empty((), dtype=torch.float32, device=dev) for _ in range(2)]
    wkb = [wk, torch.empty_like(wk)]
    host_loss = torch.empty(max(1, args.e2e_steps), dtype=torch.float32).pin_memory()
    cs = torch.cuda.Stream(dev)
    done = [torch.cuda.Event() for _ in range(2)]
    used = [torch.cuda.Event() for _ in range(2)]
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    n_e2e = max(1, args.e2e_steps)
    warm = 2
    for k in range(-warm, n_e2e):
        if k == 0:
            stream.synchronize()
            cs.synchronize()
            e0.record(cs)
        b = k % 2
        with torch.cuda.stream(cs):
            if k >= 2 - warm:
                cs.wait_event(used[b])
            xb[b].copy_(hx, non_blocking=True)
            yb[b].copy_(hy, non_blocking=True)
            done[b].record(cs)
        stream.wait_event(done[b])
        call(xb[b], yb[b], lb[b], wkb[b])
        host_loss[max(k, 0)].copy_(lb[b], non_blocking=True)
        used[b].record(stream)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = _max_over_ranks(e0.elapsed_time(e1) / n_e2e, dev)
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    # forward: one product (the logits); training: also dX and dW
    flops = 2.0 * m.s * m.h * m.V * (3 if train else 1)
    burst, sustained, kind = _tensor_peaks()
    achieved = flops / (call_ms * 1e-3) / 1e12
    ms_step = total_ms / args.steps
    out = {
        "metric": LMHEAD_TRAIN_METRIC if train else LMHEAD_METRIC,
        "value": round(_weak_scaling_value(m.s * args.steps, world, total_ms), 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded counter-based generator; no dataset or trained weights)",
        "config": {
            "workload": (f"{m.name}: X [{m.s}, {m.h}] ~N(0,{m.sigma_x:g}^2), head [{m.V}, {m.h}] in t={m.t} "
                         f"vocabulary shards ~N(0,({m.logit_sigma:g}/sqrt(h))^2) (logits ~N(0,{m.logit_sigma:g}^2)), "
                         f"bf16, targets uniform"),
            "global_batch": m.s * world,
            "seq_len": m.s,
            "parallelism": f"vocab shards t={m.t} on one GPU; {world} independent replica(s)",
            "l2": f"inputs larger than L2: the head is {sum(w.numel() for w in ws) * 2 / 1e9:.2f} GB",
            "path": "vpce_lmhead_forward (tcgen05 GEMM, fp32 accumulators in TMEM, loss statistics in the "
                    "epilogue; the logits are never written), then the shard combine"
                    + ("; training: vpce_lmhead_forward_backward, per 8192-row chunk the same GEMM keeping the "
                       "chunk's fp32 logits, a row kernel (logsumexp, loss, bf16 dZ), then two tcgen05 kernels "
                       "dX = dZ W (bf16 out) and dW += dZ^T X (TMA tile reductions)" if train else ""),
        },
        "tflops": round(achieved, 1),
        "roofline": {
            "kernel": "gemm_stats_kernel" + (" + row kernel + gemm_bwd_kernel dX, dW (the whole step)" if train else ""),
            "bound": "tensor",
            "achieved": round(achieved, 1),
            "peak": burst,
            "peak_kind": f"{kind} burst (cuBLAS bf16)",
            "unit": "TFLOP/s",
            "frac": round(achieved / burst, 4),
            "frac_of_sustained": round(achieved / sustained, 4),
            "traffic": None if train else _ncu_traffic("gemm_stats_kernel", m.name),
            "algorithmic_flops_per_launch": flops,
            "note": ("achieved = 6 s h V (logits, dX, dW) / mean CUDA-event time of one training step" if train else
                     "achieved = 2 s h V / mean CUDA-event time of one call (the GEMM launch plus the few-us combine)"),
        },
        "e2e": {
            "value": round(_weak_scaling_value(m.s, world, e2e_ms), 1),
            "unit": "tokens/s",
            "h2d_bytes_per_step": int(x.numel() * 2 + m.s * 8),
            "d2h_bytes_per_step": 4,
            "steps": n_e2e,
            "ms_per_step": round(e2e_ms, 4),
            "note": "pinned host hidden states + targets copied in every step (copy stream, double-buffered), "
                    "loss read back; the head's weights stay on the device",
        },
        "gpu_launches": (2 + (m.s + 8191) // 8192 * 4 if train else 2) * args.steps,
        "clocks": clk,
    }
    if train:
        out["gpu_launches_note"] = ("the n_valid prologue and the loss sum, and per row chunk the logits GEMM, the "
                                    "row kernel and the dX and dW kernels")
    if world == 1 and not args.no_cpu_baseline and not train:
        # the oracle on a bounded sample: a few rows against the first vocabulary
        # rows of the head (read back from the device generator), scaled to the
        # full vocabulary (the oracle's cost is linear in V)
        nv = min(8192, m.V)
        w_sample = ws[0][:nv].view(torch.int16).cpu().numpy().view(np.uint16)
        rows = np.arange(4)
        x_sample = x[:4].view(torch.int16).cpu().numpy().view(np.uint16)
        t_start = time.perf_counter()
        done_rows = 0
        while time.perf_counter() - t_start < args.cpu_seconds:
            z = O.lmhead_logits(x_sample, [w_sample], [0, nv])
            O.cross_entropy(z, np.minimum(meta.targets[rows], nv - 1))
            done_rows += len(rows)
        dt = time.perf_counter() - t_start
        out["cpu_baseline"] = {
            "value": round(done_rows / dt * nv / m.V, 3),
            "unit": "tokens/s",
            "cores": os.cpu_count(),
            "kind": "oracle",
            "sample": f"{done_rows} rows x {nv} of {m.V} vocabulary rows (fp64 numpy matmul on up to {os.cpu_count()} BLAS threads + loss), "
                      f"{dt:.1f} s, scaled by {nv}/{m.V}",
        }
    print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()


# ----------------------------------------------------------------------------
# the vocabulary-parallel input embedding (forward + backward)
# ----------------------------------------------------------------------------
EMBED_METRIC = "vocab-parallel embedding fwd+bwd tokens/s & HBM GB/s (% of peak), s=8192 h=8192 V=128256 bf16, 1 GB300"


def _embedding_launches(s):
    """Kernels one forward + backward launches for s ids: the gather, then per
    16384-row chunk the sort-and-run-scan cluster and the accumulation."""
    return 1 + 2 * ((s + 16383) // 16384)


def run_embedding(args):
    import torch

    from vocab_sharded_lm_gb300 import _build, vpce
    from oracle import vpce_oracle as O

    rank, world, local = _env_rank()
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    _build.build()
    vpce.load_library()
    V, h, t = 128256, 8192, 8
    s = args.rows or 8192
    vs = synth.even_vocab_start(V, t)
    idw = synth.Workload("embedding_ids", 6, s, V, 1, "bf16", 1.0, "zipf1.1")
    ids_host = synth.row_meta(idw).targets
    ids = torch.from_numpy(ids_host).to(dev)
    tab = synth.table_device(idw.seed, vs, h, device=dev)
    gout = synth.grad_device(idw.seed, s, h, device=dev)
    grads = [torch.zeros((vs[i + 1] - vs[i], h), dtype=torch.float32, device=dev) for i in range(t)]
    out = torch.empty((s, h), dtype=torch.bfloat16, device=dev)
    wk = torch.empty(vpce.vpce_embedding_backward_workspace_bytes(), dtype=torch.uint8, device=dev)
    flag = torch.zeros((), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        vpce.vpce_embedding_forward(tab, ids, vs, out=out, flag=flag)
        if ev:
            ev[1].record(stream)
        vpce.vpce_embedding_backward(gout, ids, grads, vs, workspace=wk)
        if ev:
            ev[2].record(stream)

    for _ in range(args.warmup):
        step()
    evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for k in range(args.steps):
        step(evs[k])
    t1.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    total_ms = _max_over_ranks(t0.elapsed_time(t1), dev)
    fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    bwd_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)

    # end to end: ids and the output gradient copied in each step, the flag read back
    h_ids = torch.from_numpy(ids_host).pin_memory()
    h_g = gout.cpu().pin_memory()
    n_e2e = max(1, args.e2e_steps)
    h_flag = torch.empty(n_e2e, dtype=torch.int32).pin_memory()
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for k in range(n_e2e):
        ids.copy_(h_ids, non_blocking=True)
        gout.copy_(h_g, non_blocking=True)
        step()
        h_flag[k].copy_(flag, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = _max_over_ranks(e0.elapsed_time(e1) / n_e2e, dev)
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    uniq = int(np.unique(ids_host[(ids_host >= 0) & (ids_host < V)]).size)
    fwd_bytes = 2 * s * h * 2 + 8 * s
    bwd_bytes = s * h * 2 + 2 * uniq * h * 4 + 8 * s
    peak, kind = _peaks()
    ms_step = total_ms / args.steps
    achieved = (fwd_bytes + bwd_bytes) / ((fwd_ms + bwd_ms) * 1e-3) / 1e9
    out_line = {
        "metric": EMBED_METRIC,
        "value": round(_weak_scaling_value(s * args.steps, world, total_ms), 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded counter-based generator; no dataset or trained weights)",
        "config": {
            "workload": f"table [{V}, {h}] bf16 in t={t} vocabulary shards, {s} ids Zipf(1.1) ({uniq} distinct), "
                        f"output gradient [{s}, {h}] bf16, fp32 gradient table",
            "global_batch": s * world,
            "seq_len": s,
            "parallelism": f"vocab shards t={t} on one GPU; {world} independent replica(s)",
            "l2": "the table (2.10 GB) and gradient table (4.20 GB) are larger than L2; the rows one step touches "
                  "(128 MB out, 128 MB gradient) are re-read by the next step only in part",
            "path": "vpce_embedding_forward (row gather) + vpce_embedding_backward (sort, per-id sums, fp32 add)",
        },
        "fwd_ms": round(fwd_ms, 5),
        "bwd_ms": round(bwd_ms, 5),
        "roofline": {
            "kernel": "the whole step: embed_forward_kernel, embed_sort_runs_kernel, embed_accum_kernel",
            "bound": "hbm",
            "achieved": round(achieved, 1),
            "peak": peak,
            "peak_kind": kind,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": None,
            "algorithmic_bytes_per_step": fwd_bytes + bwd_bytes,
            "note": "forward: the gathered rows read and written; backward: the gradient rows read and the "
                    "distinct ids' fp32 rows read and written",
        },
        "e2e": {
            "value": round(_weak_scaling_value(s, world, e2e_ms), 1),
            "unit": "tokens/s",
            "h2d_bytes_per_step": int(s * 8 + s * h * 2),
            "d2h_bytes_per_step": 4,
            "steps": n_e2e,
            "ms_per_step": round(e2e_ms, 4),
            "note": "pinned host ids and output gradient copied in every step, the id flag read back; the "
                    "tables stay on the device",
        },
        "gpu_launches": _embedding_launches(s) * args.steps,
        "clocks": clk,
    }
    if world == 1 and not args.no_cpu_baseline:
        rows = np.arange(min(s, 512))
        tab_host = [e.view(torch.int16).cpu().numpy().view(np.uint16) for e in tab]
        g_host = O.widen(gout[:len(rows)].view(torch.int16).cpu().numpy().view(np.uint16), "bf16")
        t_start = time.perf_counter()
        n_done = 0
        while time.perf_counter() - t_start < args.cpu_seconds:
            O.embedding_forward(tab_host, vs, ids_host[rows])
            O.embedding_backward(g_host, ids_host[rows], vs, h)
            n_done += len(rows)
        dt = time.perf_counter() - t_start
        out_line["cpu_baseline"] = {"value": round(n_done / dt, 2), "unit": "tokens/s", "cores": 1,
                                    "kind": "oracle",
                                    "sample": f"{n_done} ids (batches of {len(rows)}), fp64 numpy forward + "
                                              f"backward on one host core, {dt:.1f} s"}
    print(json.dumps(out_line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=synth.BENCH_WORKLOAD, choices=list(synth.WORKLOADS))
    ap.add_argument("--max-buffers", type=int, default=48)
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="seconds of oracle timing on one core, and again on every core")
    ap.add_argument("--ref-rows", type=int, default=32)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--path", choices=["fused", "split", "lmhead", "lmhead_train", "embedding", "distributed"],
                    default="fused",
                    help="fused: vpce_forward_backward; split: vpce_forward then vpce_backward; "
                         "lmhead: the LM-head GEMM fused with the forward loss; embedding: the vocabulary-parallel "
                         "input embedding; distributed: one batch with its vocabulary split over the torchrun "
                         "processes (each its own metric)")
    ap.add_argument("--vocab", type=int, default=0,
                    help="LM-head paths: vocabulary size of a smaller head (profiling captures)")
    ap.add_argument("--shards", type=int, default=0, help="LM-head paths with --vocab: vocabulary shards")
    ap.add_argument("--rows", type=int, default=0,
                    help="override the workload's row count (small profiling captures only)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.path in ("lmhead", "lmhead_train"):
        run_lmhead(args)
    elif args.path == "embedding":
        run_embedding(args)
    elif args.path == "distributed":
        run_distributed(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
