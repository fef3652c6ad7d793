#!/usr/bin/env python3
"""Ring Attention forward benchmark on GB300.

It reports causal-adjusted attention TFLOP/s, and the fraction of dense
BF16 tensor peak, for ``ra_ring_forward``.  One step is one full forward:
in bf16 a single launch runs all P ring steps (every virtual rank folds
each visiting K/V block into its state, kept on chip) and the finalize; in
fp32 it is the state init, one launch per ring step and the finalize.  A
step runs over one batch of the workload, with the inputs resident in HBM.

FLOP convention: 4*d FLOPs per allowed (query, key) pair per query head
(QK^T and PV, two each).  The causal pair count is N^2/2 ("causal-adjusted").
The exact count N(N+1)/2 is reported as well.

The JSON line also carries:
  e2e           the same metric through ra_ring_forward_host.  That call
                copies pinned host Q/K/V to the device, runs, and copies O
                and LSE back, every step.
  roofline      the dominant kernel's achieved TFLOP/s (the fused ring in
                bf16, the block update in fp32) against the measured
                dense BF16 peak, timed by the library's per-launch CUDA
                events on the launching stream, with its DRAM bytes per
                launch from the committed ncu record while the kernel's
                source is the one recorded.
  cpu_baseline  the fp64 CPU oracle on a bounded sample of the same
                workload, on this host's cores.
  clocks        SM clocks and throttle reasons sampled during the timed
                region.

--impl reference times the CPU oracle alone: a bounded sample per step, on
the same workload, metric and unit.

Decode runs (--decode decode-1m | decode-1m-q4) time ra_decode_forward: a
few query tokens against a 1M-token K/V history in P shards: the split-K
chunk kernel, then one launch that merges every partial state and
finalizes.  That path is HBM-bound, so its metric is the K/V bytes read per
second, and its roofline is the chunk kernel against the measured HBM copy
bandwidth.

Backward runs (--backward) time ra_ring_backward on the workload, given
the forward's outputs: the pre-pass, then per ring step the dQ and the
dK/dV kernels.  The FLOP convention is the FlashAttention one for the
backward: five products per pair (S recomputed, dP, dV, dK, dQ), 10*d
FLOPs per allowed pair per query head, causal-adjusted.

Masked runs (--layout zigzag|striped, --window W, --docs K, --n-valid V)
time ra_ring_forward_masked on the same workload laid out and masked that
way.  Their metric counts 4*d FLOPs per allowed (query, key) pair per query
head, the exact count under the mask; they carry no e2e figure (the host
entry point has no masked form).

Multi-GPU (torchrun): each rank runs an independent replica of the
workload on its own GPU.  The per-GPU work is fixed, the time is the max
over ranks, and the value is the sum over ranks.
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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
METRIC = "causal-adjusted attention TFLOP/s on 1 GB300 and % of dense BF16 tensor peak"
METRIC_MASKED = "attention TFLOP/s over the allowed (query, key) pairs on 1 GB300"


class MaskRun:
    """Layout and mask of a masked run, with the per-position quantities the
    FLOP count and the oracle sample need (host index arithmetic only)."""

    def __init__(self, w, layout="contiguous", window=0, docs=0, n_valid=-1, seed=0):
        import numpy as np

        self.layout, self.window = layout, int(window)
        self.n_valid = w.N if n_valid is None or n_valid < 0 else min(int(n_valid), w.N)
        self.docs = int(docs)
        N = w.N
        if self.docs > 0:
            rng = np.random.default_rng(1000 + seed)
            cuts = np.sort(rng.choice(np.arange(1, self.n_valid), size=self.docs - 1,
                                      replace=False))
            self.cu = np.concatenate([[0], cuts, [self.n_valid]]).astype(np.int64)
        else:
            self.cu = np.array([0, self.n_valid], dtype=np.int64)
        p = np.arange(N, dtype=np.int64)
        d = np.clip(np.searchsorted(self.cu, p, side="right") - 1, 0, len(self.cu) - 2)
        self.doc = np.where(p < self.n_valid, d, -1)
        lo, hi = self.cu[d], np.minimum(self.cu[d + 1], self.n_valid)
        if w.causal:
            hi = np.minimum(hi, p + 1)
        if self.window > 0:
            lo = np.maximum(lo, p - self.window + 1)
            if not w.causal:
                hi = np.minimum(hi, p + self.window)
        self.keys = np.where(p < self.n_valid, np.maximum(hi - lo, 0), 0)  # per position
        self.pairs = int(self.keys.sum())

    def active(self):
        return (self.layout != "contiguous" or self.window > 0 or self.docs > 0
                or self.n_valid < len(self.keys))

    def describe(self):
        return {"layout": self.layout, "window": self.window, "docs": self.docs,
                "n_valid": self.n_valid, "allowed_pairs": self.pairs}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(x: float, ws: int) -> float:
    """Max of a host float over ranks (identity at world size 1)."""
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist

    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" \
        else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist

        dist.barrier()


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, log_dir: str | None = None):
        """The raw samples go to log_dir/clocks_gpu<i>.csv when log_dir is
        given (--clock-log), else to a temporary file."""
        import tempfile

        self.gpu = gpu_index
        self.proc = None
        self.keep = bool(log_dir)
        if log_dir:
            self.path = os.path.join(log_dir, f"clocks_gpu{gpu_index}.csv")
        else:
            self.path = os.path.join(tempfile.gettempdir(), f"ra_clocks_{os.getpid()}_{gpu_index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.gpu)], stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sms, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sms.append(float(parts[1]))
                    maxes.append(float(parts[2]))
                except ValueError:
                    continue
                for nm, val in zip(names, parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(nm)
        if not self.keep:
            try:
                os.remove(self.path)
            except OSError:
                pass
        if not sms:
            return None
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxes),
                "reasons": sorted(reasons), "samples": len(sms)}


def timed_warmup(step, warmup, dev):
    """Run the warm-up steps; return their mean wall time in seconds."""
    import torch

    torch.cuda.synchronize(dev)
    t0 = time.time()
    for _ in range(warmup):
        step()
    torch.cuda.synchronize(dev)
    return (time.time() - t0) / max(1, warmup)


CLOCK_WINDOW_S = 1.0  # shortest sampled window: five nvidia-smi samples
CLOCK_PAD_S = 0.5


def clock_pad(step, dev, seconds):
    """Untimed steps of the same workload for about `seconds` of wall time,
    run inside the clock sampler's window just before and just after a
    timed region shorter than CLOCK_WINDOW_S, so the samples see the GPU
    under the same load as the timed steps."""
    import torch

    if seconds <= 0:
        return
    t_end = time.time() + seconds
    while time.time() < t_end:
        step()
        torch.cuda.synchronize(dev)


def pad_seconds(est_step_s, steps):
    return CLOCK_PAD_S if est_step_s * steps < CLOCK_WINDOW_S else 0.0


def note_window(clk, pad):
    if clk is not None:
        clk["window"] = ("timed region" if pad == 0 else
                         f"timed region with {pad:.1f} s of untimed steps of the same workload "
                         "on each side (region shorter than the sampling needs)")
    return clk


# ------------------------------------------------------------------ traffic record
FORWARD_SOURCES = ("umma_kernel.cu", "fwd_tile.cuh", "ptx.cuh", "ra_internal.h")
DECODE_SOURCES = ("decode_kernel.cu", "ptx.cuh", "ra_internal.h")
STATE_SOURCES = ("state_kernels.cu", "ra_internal.h")


def gpu_index_of(local: int) -> int:
    """The physical GPU index nvidia-smi knows this rank's device by."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    if vis and "," not in vis and vis.strip().isdigit():
        return int(vis)
    return local


def kernel_digest(files=FORWARD_SOURCES) -> str:
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "blockwise_online_softmax_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, profile: str = "block_update_bf16_traffic.md",
                     files=FORWARD_SOURCES):
    """DRAM bytes per launch of the dominant kernel from its committed ncu
    summary, if it was taken on the current source of that kernel (digest
    of `files` matches), else None."""
    p = os.path.join(ROOT, "profiles", profile)
    try:
        text = open(p).read()
    except OSError:
        return None
    dig = re.search(r"kernel_digest:\s*([0-9a-f]+)", text)
    val = re.search(rf"traffic_bytes_per_launch\[{re.escape(workload)}\]:\s*([0-9.eE+]+)", text)
    if not dig or not val or dig.group(1) != kernel_digest(files):
        return None
    return float(val.group(1))


# ------------------------------------------------------------------ CPU oracle sample
ARM_PARTS = {"0xd4f": "Arm Neoverse V2", "0xd40": "Arm Neoverse V1", "0xd0c": "Arm Neoverse N1",
             "0xd49": "Arm Neoverse N2"}


def cpu_model() -> str:
    """The host CPU's model name, or its Arm part number (named when known)."""
    fields = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if ":" in line:
                    key, val = line.split(":", 1)
                    fields.setdefault(key.strip().lower(), val.strip())
    except OSError:
        pass
    if "model name" in fields:
        return fields["model name"]
    if "cpu part" in fields:
        part = fields["cpu part"]
        return f"{ARM_PARTS.get(part, 'Arm')} (cpu part {part})"
    import platform

    return platform.processor() or platform.machine()


FULL_PARITY_MAX_N = 8192  # up to this length every output row is compared


def parity_check(w, q, k, v, out, lse, per_block: int = 2):
    """Parity of the timed run's own output against the fp64 oracle: every
    row when N <= FULL_PARITY_MAX_N (the small workloads, a few seconds of
    oracle time), else sampled rows ({0, 1, 127, 128, c/2, c-1} and
    `per_block` random rows of every block); all heads, each row over its
    full key range."""
    import numpy as np
    import torch

    import oracle
    from blockwise_online_softmax_gb300 import inputs

    if w.N <= FULL_PARITY_MAX_N:
        rows = np.arange(w.N, dtype=np.int64)
    else:
        rows = inputs.sample_rows(w, random_per_block=per_block)
    idx = torch.from_numpy(rows).to(out.device)
    got_o = out.index_select(0, idx).cpu().double().numpy()
    got_l = lse.index_select(0, idx).cpu().double().numpy()
    t0 = time.perf_counter()
    ref_o, ref_l = oracle.attention(q, k, v, causal=w.causal, rows=rows)
    dt = time.perf_counter() - t0
    fin = np.isfinite(ref_l)
    e_o = float(np.abs(got_o - ref_o).max())
    e_l = float((np.abs(got_l[fin] - ref_l[fin]) / np.maximum(1.0, np.abs(ref_l[fin]))).max())
    tol_o, tol_l = (1e-2, 1e-3) if w.dtype == "bf16" else (1e-5, 1e-5)
    return {"rows": int(len(rows)), "all_rows": bool(len(rows) == w.N), "heads": w.heads,
            "max_abs_o": e_o, "max_rel_lse": e_l,
            "tol_o": tol_o, "tol_lse": tol_l, "pass": bool(e_o <= tol_o and e_l <= tol_l),
            "oracle_s": dt}


def oracle_sample(w, q, k, v, target_s: float, seed: int = 7, mask: MaskRun | None = None,
                  threads: int | None = None):
    """Time the fp64 oracle on sampled query rows (all heads, full key
    range), sized to take about ``target_s`` seconds.  Returns (TFLOP/s,
    cores, description).  With ``mask``, q/k/v are in sequence order and the
    oracle applies the mask's window and documents."""
    import numpy as np

    import oracle

    cores = threads or os.cpu_count() or 1
    rng = np.random.default_rng(seed)
    kw = {}
    if mask is not None:
        kw = dict(window=mask.window, q_doc=mask.doc, k_doc=mask.doc)

    def flops(rows):
        if mask is not None:
            keys = mask.keys[rows]
        else:
            keys = (rows + 1) if w.causal else np.full_like(rows, w.N)
        return float(4.0 * w.d * w.heads * keys.sum())

    # calibrate on a few rows
    probe = np.sort(rng.integers(w.N // 2, w.N, size=max(2, cores // w.heads + 1)))
    t0 = time.perf_counter()
    oracle.partial_state(q, k, v, causal=w.causal, rows=probe, threads=cores, **kw)
    dt = time.perf_counter() - t0
    rate = max(flops(probe), 1.0) / max(dt, 1e-6)
    # rows drawn uniformly over the sequence; expected FLOPs per row
    if mask is not None:
        per_row = 4.0 * w.d * w.heads * max(mask.pairs / w.N, 1.0)
    else:
        per_row = 4.0 * w.d * w.heads * (w.N / 2 if w.causal else w.N)
    n_rows = int(max(1, min(w.N, target_s * rate / per_row)))
    rows = np.sort(rng.choice(w.N, size=n_rows, replace=False))
    t0 = time.perf_counter()
    oracle.partial_state(q, k, v, causal=w.causal, rows=rows, threads=cores, **kw)
    dt = time.perf_counter() - t0
    f = flops(rows)
    desc = (f"{n_rows} query rows drawn uniformly from {w.N}, all {w.heads} heads, each over its "
            f"full {'masked' if mask is not None else 'causal'} key range ({f:.3e} FLOPs, "
            f"{dt:.1f} s)")
    return f / dt / 1e12, cores, desc, dt


# ------------------------------------------------------------------ decode
METRIC_DECODE = "decode attention: K/V bytes read per second on 1 GB300 (HBM-bound)"


def run_decode(args, ws, rank, local):
    import numpy as np
    import torch

    import blockwise_online_softmax_gb300 as ra
    import oracle
    from blockwise_online_softmax_gb300 import binding, inputs

    w = inputs.DECODE_WORKLOADS[args.decode]
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    binding.lib()
    peaks, peak_src = load_peaks()
    q, k, v = inputs.make_decode(w)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    out = torch.empty((w.n_q, w.heads, w.d), dtype=torch.float32, device=dev)
    lse = torch.empty((w.n_q, w.heads), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        ra.ra_decode_forward(qd, kd, vd, P=w.P, out=out, lse=lse, stream=stream)

    est = timed_warmup(step, args.warmup, dev)
    pad = pad_seconds(est, args.steps)
    ra.ra_device_status(stream)
    clocks = ClockSampler(gpu_index_of(local), args.clock_log)
    clocks.start()
    clock_pad(step, dev, pad)
    ra.ra_trace_reset()
    ra.ra_trace_enable(True)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    barrier(ws)
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(ws)
    ra.ra_trace_enable(False)
    clock_pad(step, dev, pad)
    clk = note_window(clocks.stop(), pad)
    ra.ra_device_status(stream)
    ms_step = reduce_max(ev0.elapsed_time(ev1), ws) / args.steps
    kinds = ("decode_split", "decode_combine", "merge", "finalize", "state_init")
    trace = {kd_: ra.ra_trace_query(kd_) for kd_ in kinds}
    ra.ra_trace_reset()
    value = ws * w.kv_bytes() / (ms_step * 1e-3) / 1e9
    n_split, ms_split = trace["decode_split"]
    achieved = w.kv_bytes() * n_split / (ms_split * 1e-3) / 1e9 if ms_split > 0 else None
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        # The oracle over every query row, on as many query heads as fit the
        # time budget; its rate is scaled to the same unit (K/V bytes of the
        # whole step per second).
        cores = os.cpu_count() or 1
        qpos = w.n_kv - w.n_q + np.arange(w.n_q)
        g = w.heads // w.kv_heads
        t0 = time.perf_counter()
        oracle.partial_state(q[:, :g], k[:, :1], v[:, :1], causal=True, q_pos=qpos,
                             threads=cores)
        per_kv_head = time.perf_counter() - t0
        nh = int(max(1, min(w.kv_heads, args.cpu_seconds / max(per_kv_head, 1e-6))))
        t0 = time.perf_counter()
        oracle.partial_state(q[:, :g * nh], k[:, :nh], v[:, :nh], causal=True, q_pos=qpos,
                             threads=cores)
        dt = time.perf_counter() - t0
        frac = nh / w.kv_heads
        cpu = {"value": w.kv_bytes() * frac / dt / 1e9, "unit": "GB/s", "cores": cores,
               "kind": "oracle",
               "sample": f"all {w.n_q} query rows of the {g * nh} query heads of {nh} of "
                         f"{w.kv_heads} KV heads, full history ({dt:.1f} s)"}
    if rank != 0:
        return
    line = {
        "metric": METRIC_DECODE, "value": value, "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "n_q": w.n_q, "n_kv": w.n_kv, "P": w.P,
                   "heads": w.heads, "kv_heads": w.kv_heads, "d": w.d, "causal": True,
                   "seed": w.seed, "parallelism": f"replicas{ws}",
                   "kv_bytes_per_step": w.kv_bytes(), "flops_per_step": w.flops(),
                   "l2": "K and V (4.3 GB) exceed L2; no flush"},
        "clocks": clk, "e2e": None,
        "gpu_launches": sum(n for n, _ in trace.values()),
        "kernel_ms": {kd_: t / args.steps for kd_, (n, t) in trace.items()},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": (achieved / peaks["hbm_gbs"]) if achieved else None,
                     "traffic": recorded_traffic(w.name, "decode_tc_traffic.md", DECODE_SOURCES),
                     "kernel": "decode split-K chunks (tcgen05, TMA)",
                     "peak_kind": f"hbm_gbs ({peak_src})"},
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ state kernels
METRIC_STATE = ("state kernels (init, merge, finalize): algorithmic HBM GB/s over one "
                "init + two merges + one finalize of the workload's [N, heads] state")


def state_bytes(d: int) -> dict:
    """Algorithmic bytes per (row, head) of each state kernel: m and l are
    fp32 scalars, O~ is d fp32 values; merge reads two states and writes
    one; finalize reads one state and writes out (d values) and LSE."""
    st = 8 + 4 * d
    return {"state_init": st, "merge": 3 * st, "finalize": st + 4 + 4 * d}


def run_state(args, w, ws, rank, local):
    import numpy as np
    import torch

    import blockwise_online_softmax_gb300 as ra
    from blockwise_online_softmax_gb300 import binding

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    binding.lib()
    peaks, peak_src = load_peaks()
    R, H, d = w.N, w.heads, w.d
    gen = torch.Generator(device=dev)
    gen.manual_seed(w.seed)

    def partial_state():
        # A synthetic partial state: a running max near a typical LSE, a
        # positive sum and O~ of that scale.
        m = torch.randn((R, H), generator=gen, device=dev) * 2 + 5
        l = torch.rand((R, H), generator=gen, device=dev) * 99 + 1
        o = torch.randn((R, H, d), generator=gen, device=dev) * l[..., None]
        return m, l, o

    b, c = partial_state(), partial_state()
    a = (torch.empty((R, H), device=dev), torch.empty((R, H), device=dev),
         torch.empty((R, H, d), device=dev))
    out = torch.empty((R, H, d), device=dev)
    lse = torch.empty((R, H), device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        ra.ra_state_init(*a, stream=stream)
        ra.ra_merge(*a, *b, stream=stream)     # a = identity (+) b
        ra.ra_merge(*a, *c, stream=stream)     # the general case
        ra.ra_finalize(*a, out=out, lse=lse, stream=stream)

    est = timed_warmup(step, args.warmup, dev)
    pad = pad_seconds(est, args.steps)
    ra.ra_device_status(stream)
    clocks = ClockSampler(gpu_index_of(local), args.clock_log)
    clocks.start()
    clock_pad(step, dev, pad)
    ra.ra_trace_reset()
    ra.ra_trace_enable(True)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    barrier(ws)
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(ws)
    ra.ra_trace_enable(False)
    clock_pad(step, dev, pad)
    clk = note_window(clocks.stop(), pad)
    ra.ra_device_status(stream)
    ms_step = reduce_max(ev0.elapsed_time(ev1), ws) / args.steps
    per_rh = state_bytes(d)
    trace = {kd_: ra.ra_trace_query(kd_) for kd_ in per_rh}
    ra.ra_trace_reset()
    kernels = {}
    for kd_, (n, ms) in trace.items():
        gbs = per_rh[kd_] * R * H * n / (ms * 1e-3) / 1e9 if ms > 0 else None
        kernels[kd_] = {"launches_per_step": n / args.steps, "ms_per_launch": ms / max(n, 1),
                        "bytes_per_launch": per_rh[kd_] * R * H, "achieved_gbs": gbs,
                        "frac": gbs / peaks["hbm_gbs"] if gbs else None}
    step_bytes = R * H * (per_rh["state_init"] + 2 * per_rh["merge"] + per_rh["finalize"])
    value = ws * step_bytes / (ms_step * 1e-3) / 1e9
    dom = kernels["merge"]
    # parity of the run's own output on sampled rows: the oracle's merge and
    # finalize (fp64 numpy) over the same three states
    parity = None
    cpu = None
    if rank == 0:
        import oracle.online as online

        rows = np.random.default_rng(5).choice(R, size=min(R, 256), replace=False)
        sel = torch.from_numpy(rows).to(dev)

        def pick(st):
            return tuple(x.index_select(0, sel).double().cpu().numpy() for x in st)

        sb, sc_ = pick(b), pick(c)
        t0 = time.perf_counter()
        ref = online.merge(online.merge(online.identity_state(len(rows), H, d), sb), sc_)
        ref_out, ref_lse = online.finalize(ref)
        dt = time.perf_counter() - t0
        got_o = out.index_select(0, sel).double().cpu().numpy()
        got_l = lse.index_select(0, sel).double().cpu().numpy()
        e_o = float(np.abs(got_o - ref_out).max())
        e_l = float((np.abs(got_l - ref_lse) / np.maximum(1.0, np.abs(ref_lse))).max())
        parity = {"rows": "256 seeded rows, all heads", "max_abs_out": e_o, "lse_rel": e_l,
                  "bar_out": 1e-5, "bar_lse": 1e-5, "pass": e_o <= 1e-5 and e_l <= 1e-5}
        if ws == 1 and not args.no_cpu_baseline:
            cpu = {"value": step_bytes * (len(rows) / R) / dt / 1e9, "unit": "GB/s", "cores": 1,
                   "kind": "oracle",
                   "sample": f"merge, merge and finalize of {len(rows)} rows x {H} heads in "
                             f"fp64 numpy ({dt * 1e3:.1f} ms)"}
    if rank != 0:
        return
    line = {
        "metric": METRIC_STATE, "value": value, "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": w.name, "rows": R, "heads": H, "d": d, "seed": w.seed,
                   "parallelism": f"replicas{ws}", "bytes_per_step": step_bytes,
                   "bytes_per_row_head": per_rh,
                   "l2": f"each state {R * H * (8 + 4 * d) / 1e9:.2f} GB, larger than L2; "
                         "no flush"},
        "clocks": clk, "e2e": None,
        "gpu_launches": sum(n for n, _ in trace.values()),
        "kernels": kernels,
        "roofline": {"bound": "hbm", "achieved": dom["achieved_gbs"], "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": dom["frac"],
                     "traffic": recorded_traffic(w.name, "state_kernels_traffic.md",
                                                 STATE_SOURCES),
                     "kernel": "merge", "peak_kind": f"hbm_gbs ({peak_src})"},
        "cpu_baseline": cpu,
        "parity": parity,
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ ring steps
METRIC_STEPS = ("causal-adjusted attention TFLOP/s of the step-by-step ring (state init, "
                "one block-update launch per ring step with (m, l, O~) in HBM, finalize)")


def run_steps(args, w, ws, rank, local):
    import torch

    import blockwise_online_softmax_gb300 as ra
    from blockwise_online_softmax_gb300 import binding, inputs

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    binding.lib()
    peaks, peak_src = load_peaks()
    q, k, v = workload_inputs(w)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    m = torch.empty((w.N, w.heads), device=dev)
    l = torch.empty((w.N, w.heads), device=dev)
    o = torch.empty((w.N, w.heads, w.d), device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        # out and lse are written in place over o and m, as ra_ring_forward's
        # own fp32 path does.
        ra.ra_state_init(m, l, o, stream=stream)
        for s_ in range(w.P):
            ra.ra_ring_step(qd, kd, vd, m, l, o, P=w.P, s=s_, causal=w.causal, stream=stream)
        ra.ra_finalize(m, l, o, out=o, lse=m, stream=stream)

    est = timed_warmup(step, args.warmup, dev)
    pad = pad_seconds(est, args.steps)
    ra.ra_device_status(stream)
    clocks = ClockSampler(gpu_index_of(local), args.clock_log)
    clocks.start()
    clock_pad(step, dev, pad)
    ra.ra_trace_reset()
    ra.ra_trace_enable(True)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    barrier(ws)
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(ws)
    ra.ra_trace_enable(False)
    clock_pad(step, dev, pad)
    clk = note_window(clocks.stop(), pad)
    ra.ra_device_status(stream)
    ms_step = reduce_max(ev0.elapsed_time(ev1), ws) / args.steps
    kinds = ("state_init", "block_update_bf16", "finalize")
    trace = {kd_: ra.ra_trace_query(kd_) for kd_ in kinds}
    ra.ra_trace_reset()
    f_adj, f_exact = w.flops_causal_adjusted(), w.flops_exact()
    value = ws * f_adj / (ms_step * 1e-3) / 1e12
    n_upd, ms_upd = trace["block_update_bf16"]
    achieved = f_exact * args.steps / (ms_upd * 1e-3) / 1e12 if ms_upd > 0 else None
    peak = peaks["bf16_tflops_sustained"]
    # Algorithmic bytes of one (rank, step) pair with a full block: Q_i and
    # K_j, V_j read once, the state (m, l, O~ of block i) read and written.
    el = 2
    pair_bytes = (w.c * w.heads * w.d * el + 2 * w.c * w.kv_heads * w.d * el
                  + 2 * w.c * w.heads * (8 + 4 * w.d))
    parity = None
    if rank == 0 and not args.no_check:
        parity = parity_check(w, q, k, v, o, m)
    if rank != 0:
        return
    line = {
        "metric": METRIC_STEPS, "value": value, "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic",
        "frac_of_dense_bf16_peak": value / ws / peaks["bf16_tflops"], "peak_source": peak_src,
        "config": {**forward_config(w, ws), "path": "ra_state_init + P x ra_ring_step + "
                   "ra_finalize", "algorithmic_bytes_per_full_pair": pair_bytes},
        "clocks": clk, "e2e": None,
        "gpu_launches": sum(n for n, _ in trace.values()),
        "kernel_ms": {kd_: t / args.steps for kd_, (n, t) in trace.items()},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": (achieved / peak) if achieved else None,
                     "traffic": recorded_traffic(w.name, "block_update_bf16_traffic.md"),
                     "kernel": "block update (tcgen05), one launch per ring step",
                     "peak_kind": f"bf16_tflops_sustained ({peak_src})",
                     "frac_of_burst": (achieved / peaks["bf16_tflops"]) if achieved else None},
        "cpu_baseline": None,
        "parity": parity,
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ backward
METRIC_BWD = ("backward attention TFLOP/s (10*d FLOPs per allowed pair per query head, "
              "causal-adjusted) on 1 GB300")


def run_backward(args, w, ws, rank, local):
    import numpy as np
    import torch

    import blockwise_online_softmax_gb300 as ra
    import oracle
    from blockwise_online_softmax_gb300 import binding, inputs

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    binding.lib()
    peaks, peak_src = load_peaks()
    q, k, v = workload_inputs(w)
    g = inputs.randn_chunked((w.N, w.heads, w.d), w.seed, 3).to(torch.bfloat16)
    qd, kd, vd, gd = q.to(dev), k.to(dev), v.to(dev), g.to(dev)
    stream = torch.cuda.current_stream(dev)
    out, lse = ra.ra_ring_forward(qd, kd, vd, P=w.P, causal=w.causal, stream=stream)
    dq = torch.empty((w.N, w.heads, w.d), dtype=torch.float32, device=dev)
    dk = torch.empty((w.N, w.kv_heads, w.d), dtype=torch.float32, device=dev)
    dv = torch.empty_like(dk)

    def step():
        ra.ra_ring_backward(qd, kd, vd, out, lse, gd, P=w.P, causal=w.causal, dq=dq, dk=dk,
                            dv=dv, stream=stream)

    est = timed_warmup(step, args.warmup, dev)
    pad = pad_seconds(est, args.steps)
    ra.ra_device_status(stream)
    clocks = ClockSampler(gpu_index_of(local), args.clock_log)
    clocks.start()
    clock_pad(step, dev, pad)
    ra.ra_trace_reset()
    ra.ra_trace_enable(True)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    barrier(ws)
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(ws)
    ra.ra_trace_enable(False)
    clock_pad(step, dev, pad)
    clk = note_window(clocks.stop(), pad)
    ra.ra_device_status(stream)
    ms_step = reduce_max(ev0.elapsed_time(ev1), ws) / args.steps
    trace = {kd_: ra.ra_trace_query(kd_) for kd_ in ("bwd_pre", "bwd_dq", "bwd_dkdv")}
    ra.ra_trace_reset()
    f_adj = 2.5 * w.flops_causal_adjusted()
    f_exact = 2.5 * w.flops_exact()
    value = ws * f_adj / (ms_step * 1e-3) / 1e12
    ms_dq, ms_dkdv = trace["bwd_dq"][1], trace["bwd_dkdv"][1]
    # dQ kernel: S, dP, dQ products (3 of the 5); dK/dV kernel: S, dP, dV, dK (4).
    ach_dq = (0.6 * f_exact * args.steps) / (ms_dq * 1e-3) / 1e12 if ms_dq > 0 else None
    ach_dkdv = (0.8 * f_exact * args.steps) / (ms_dkdv * 1e-3) / 1e12 if ms_dkdv > 0 else None
    peak = peaks["bf16_tflops_sustained"]
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cores = os.cpu_count() or 1
        rng = np.random.default_rng(7)
        rows = np.sort(rng.choice(w.N, size=max(1, cores), replace=False))
        t0 = time.perf_counter()
        oracle.grad_q(q, k, v, g, causal=w.causal, rows=rows, threads=cores)
        dt = time.perf_counter() - t0
        keys = (rows + 1) if w.causal else np.full_like(rows, w.N)
        # grad_q makes three passes over a row's keys (scores, D, dQ): count
        # the S, dP and dQ products, 6*d FLOPs per pair per head.
        f = 6.0 * w.d * w.heads * float(keys.sum())
        cpu = {"value": f / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": f"dQ of {len(rows)} query rows drawn uniformly, all {w.heads} heads, "
                         f"full causal key range ({f:.3e} FLOPs of S, dP, dQ, {dt:.1f} s)"}
    if rank != 0:
        return
    line = {
        "metric": METRIC_BWD, "value": value, "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic",
        "frac_of_dense_bf16_peak": value / ws / peaks["bf16_tflops"], "peak_source": peak_src,
        "config": {"workload": w.name, "N": w.N, "P": w.P, "c": w.c, "heads": w.heads,
                   "kv_heads": w.kv_heads, "d": w.d, "causal": w.causal, "recipe": w.recipe,
                   "seed": w.seed, "parallelism": f"replicas{ws}",
                   "flops_per_step_causal_adjusted": f_adj, "flops_per_step_exact": f_exact,
                   "l2": "inputs larger than L2; no flush"},
        "clocks": clk, "e2e": None,
        "gpu_launches": sum(n for n, _ in trace.values()),
        "kernel_ms": {kd_: t / args.steps for kd_, (n, t) in trace.items()},
        "roofline": {"bound": "tensor", "achieved": ach_dkdv, "peak": peak, "unit": "TFLOP/s",
                     "frac": (ach_dkdv / peak) if ach_dkdv else None, "traffic": None,
                     "kernel": "backward dK/dV (tcgen05)",
                     "peak_kind": f"bf16_tflops_sustained ({peak_src})",
                     "dq_kernel_achieved": ach_dq},
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ arms
def head_slice(w, heads: int):
    """The workload restricted to its first `heads` query heads and their KV
    heads.  The inputs are the full workload's tensors cut to those heads
    (the same values), so the slice is the same problem on fewer heads."""
    import dataclasses

    g = w.heads // w.kv_heads
    if heads <= 0 or heads > w.heads or heads % g:
        raise SystemExit(f"--heads must be a positive multiple of {g} up to {w.heads}")
    return dataclasses.replace(w, name=f"{w.name}[:{heads} heads]", heads=heads,
                               kv_heads=heads // g,
                               extra={**w.extra, "full": w.name, "full_heads": w.heads,
                                      "full_kv_heads": w.kv_heads})


def workload_inputs(w):
    """(q, k, v) of the workload; for a head slice, the full workload's
    tensors cut to its heads."""
    from blockwise_online_softmax_gb300 import inputs

    full = w.extra.get("full")
    if full is None:
        return inputs.make_workload(w)
    q, k, v = inputs.make_workload(inputs.WORKLOADS[full])
    return (q[:, :w.heads].contiguous(), k[:, :w.kv_heads].contiguous(),
            v[:, :w.kv_heads].contiguous())


def forward_config(w, ws):
    """The workload description both arms print, key for key."""
    return {
        "workload": w.name, "N": w.N, "P": w.P, "c": w.c, "heads": w.heads,
        "kv_heads": w.kv_heads, "d": w.d, "causal": w.causal, "input_dtype": w.dtype,
        "recipe": w.recipe, "seed": w.seed, "parallelism": f"replicas{ws}",
        "flops_per_step_causal_adjusted": w.flops_causal_adjusted(),
        "flops_per_step_exact": w.flops_exact(),
        "l2": (f"footprint {footprint_bytes(w) / 1e6:.0f} MB fits in L2: a {L2_FLUSH_BYTES >> 20}"
               " MiB buffer is written between timed steps, outside their events"
               if needs_l2_flush(w) else
               f"footprint {footprint_bytes(w) / 1e9:.2f} GB, larger than L2; no flush"),
    }


L2_BYTES = 129 * 10**6
L2_FLUSH_BYTES = 512 << 20


def footprint_bytes(w) -> int:
    """Q, K, V as stored plus the fp32 O and LSE one forward touches."""
    el = 2 if w.dtype == "bf16" else 4
    return w.N * (w.heads + 2 * w.kv_heads) * w.d * el + w.N * w.heads * (w.d + 1) * 4


def needs_l2_flush(w) -> bool:
    return footprint_bytes(w) < 2 * L2_BYTES


def run_reference(args, w, ws, rank):
    if rank != 0:
        return
    from blockwise_online_softmax_gb300 import inputs

    q, k, v = workload_inputs(w)
    per_step = args.ref_step_seconds
    for _ in range(args.warmup):
        oracle_sample(w, q, k, v, per_step / 4)
    vals, secs, desc, cores = [], [], "", 1
    for s in range(args.steps):
        val, cores, desc, dt = oracle_sample(w, q, k, v, per_step, seed=100 + s)
        vals.append(val)
        secs.append(dt)
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * statistics.median(secs), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": forward_config(w, ws),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": "per step: " + desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def run_ours(args, w, ws, rank, local):
    import torch

    import blockwise_online_softmax_gb300 as ra
    from blockwise_online_softmax_gb300 import binding, inputs

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    binding.lib()
    peaks, peak_src = load_peaks()

    q, k, v = workload_inputs(w)
    mask = args.mask
    if mask is not None:
        pos = binding.layout_positions(w.N, w.P, mask.layout)
        qd, kd, vd = q[pos].to(dev), k[pos].to(dev), v[pos].to(dev)
        cu = torch.tensor(mask.cu, dtype=torch.int32, device=dev) if mask.docs > 0 else None
    else:
        qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    out = torch.empty((w.N, w.heads, w.d), dtype=torch.float32, device=dev)
    lse = torch.empty((w.N, w.heads), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        if mask is None:
            ra.ra_ring_forward(qd, kd, vd, P=w.P, causal=w.causal, out=out, lse=lse,
                               stream=stream)
        else:
            ra.ra_ring_forward_masked(qd, kd, vd, P=w.P, layout=mask.layout, causal=w.causal,
                                      window=mask.window, n_valid=mask.n_valid, cu_seqlens=cu,
                                      out=out, lse=lse, stream=stream)

    est = timed_warmup(step, args.warmup, dev)
    pad = pad_seconds(est, args.steps)
    ra.ra_device_status(stream)
    torch.cuda.synchronize(dev)
    barrier(ws)

    clocks = ClockSampler(gpu_index_of(local), args.clock_log)
    clocks.start()
    clock_pad(step, dev, pad)
    ra.ra_trace_reset()
    ra.ra_trace_enable(True)
    # A workload that fits in L2 gets a flush (a write larger than L2)
    # between timed steps; each step is then timed by its own event pair so
    # the flush stays outside.
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev) \
        if needs_l2_flush(w) else None
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    torch.cuda.synchronize(dev)
    barrier(ws)
    for i in range(args.steps):
        if flush is not None:
            flush.zero_()
        ev0[i].record(stream)
        step()
        ev1[i].record(stream)
    torch.cuda.synchronize(dev)
    barrier(ws)
    ra.ra_trace_enable(False)
    clock_pad(step, dev, pad)
    clk = note_window(clocks.stop(), pad)
    ra.ra_device_status(stream)
    per_step = [a.elapsed_time(b) for a, b in zip(ev0, ev1)]
    ms_total = sum(per_step) if flush is not None else ev0[0].elapsed_time(ev1[-1])
    n_upd, ms_upd = ra.ra_trace_query("block_update_bf16" if w.dtype == "bf16"
                                      else "block_update_f32")
    n_fz, ms_fz = ra.ra_trace_query("ring_fused_bf16")
    n_fz32, ms_fz32 = ra.ra_trace_query("ring_fused_f32")
    n_init, ms_init = ra.ra_trace_query("state_init")
    n_fin, ms_fin = ra.ra_trace_query("finalize")
    ra.ra_trace_reset()
    # The dominant kernel: the fused ring (one launch per forward: tcgen05 in
    # bf16, FFMA in fp32), or the one-step block update (P launches).
    if n_fz > 0:
        dom_ms, dom_name, dom_profile = ms_fz, "fused ring forward (tcgen05)", \
            "ring_fused_bf16_traffic.md"
    elif n_fz32 > 0:
        dom_ms, dom_name, dom_profile = ms_fz32, "fused ring forward (fp32 FFMA)", None
    else:
        dom_ms, dom_name, dom_profile = ms_upd, "block update (tcgen05)", \
            "block_update_bf16_traffic.md"
    n_fz += n_fz32
    ms_fz += ms_fz32

    ms_max = reduce_max(ms_total, ws)
    ms_step = ms_max / args.steps
    if mask is None:
        f_adj = w.flops_causal_adjusted()
        f_exact = w.flops_exact()
    else:
        f_adj = f_exact = 4.0 * w.d * w.heads * mask.pairs
    value = ws * f_adj / (ms_step * 1e-3) / 1e12

    # roofline of the dominant kernel: algorithmic FLOPs of all its launches
    # (exact allowed-pair count) over their summed time.
    achieved = (f_exact * args.steps) / (dom_ms * 1e-3) / 1e12 if dom_ms > 0 else None
    peak = peaks["bf16_tflops_sustained"]
    traffic = recorded_traffic(w.name, dom_profile) if dom_profile else None

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        val, cores, desc, _ = oracle_sample(w, q, k, v, args.cpu_seconds, mask=mask)
        val1, _, desc1, _ = oracle_sample(w, q, k, v, min(3.0, args.cpu_seconds / 5), seed=11,
                                          mask=mask, threads=1)
        cpu = {"value": val, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": desc, "cpu_model": cpu_model(), "value_1core": val1,
               "sample_1core": desc1}
    parity = None
    if rank == 0 and mask is None and not args.no_check:
        parity = parity_check(w, q, k, v, out, lse)
    if mask is not None:
        if rank == 0:
            line = {
                "metric": METRIC_MASKED, "value": value, "unit": "TFLOP/s", "n_gpus": ws,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": w.dtype, "data": "synthetic",
                "frac_of_dense_bf16_peak": value / ws / peaks["bf16_tflops"],
                "peak_source": peak_src,
                "config": {"workload": w.name, "N": w.N, "P": w.P, "c": w.c, "heads": w.heads,
                           "kv_heads": w.kv_heads, "d": w.d, "causal": w.causal,
                           "recipe": w.recipe, "seed": w.seed, "mask": mask.describe(),
                           "parallelism": f"replicas{ws}", "flops_per_step": f_adj,
                           "l2": "inputs larger than L2 (Q alone exceeds 129 MB); no flush"},
                "clocks": clk, "e2e": None, "gpu_launches": n_upd + n_fz + n_init + n_fin,
                "kernel_ms": {"ring_fused": ms_fz / args.steps,
                              "block_update": ms_upd / args.steps,
                              "state_init": ms_init / args.steps,
                              "finalize": ms_fin / args.steps},
                "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak,
                             "unit": "TFLOP/s", "frac": (achieved / peak) if achieved else None,
                             "traffic": None, "kernel": dom_name,
                             "peak_kind": f"bf16_tflops_sustained ({peak_src})"},
                "cpu_baseline": cpu,
            }
            print(json.dumps(line), flush=True)
        return

    if w.dtype == "bf16":
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": (achieved / peak) if achieved else None, "traffic": traffic,
                "kernel": dom_name,
                "peak_kind": f"bf16_tflops_sustained ({peak_src})",
                "frac_of_burst": (achieved / peaks["bf16_tflops"]) if achieved else None}
    else:
        # fp32 FFMA path: the FP32 pipe peak from unit counts and clock,
        # SMs x 128 FMA lanes x 2 FLOPs x max SM clock.
        import torch as _t

        sms = _t.cuda.get_device_properties(dev).multi_processor_count
        alu_peak = sms * 128 * 2 * 2.07e9 / 1e12
        roof = {"bound": "alu", "achieved": achieved, "peak": alu_peak, "unit": "TFLOP/s",
                "frac": (achieved / alu_peak) if achieved else None, "traffic": None,
                "kernel": dom_name,
                "peak_kind": f"{sms} SMs x 128 FP32 lanes x 2 FLOPs x 2070 MHz"}

    # end to end through the host-buffer entry point
    qp, kp, vp = q.pin_memory(), k.pin_memory(), v.pin_memory()
    out_h = torch.empty((w.N, w.heads, w.d), dtype=torch.float32, pin_memory=True)
    lse_h = torch.empty((w.N, w.heads), dtype=torch.float32, pin_memory=True)
    ra.ra_ring_forward_host(qp, kp, vp, P=w.P, causal=w.causal, out=out_h, lse=lse_h,
                            stream=stream)
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    barrier(ws)
    t0 = time.perf_counter()
    e2e_step_ms = []
    for _ in range(e2e_steps):
        t1 = time.perf_counter()
        ra.ra_ring_forward_host(qp, kp, vp, P=w.P, causal=w.causal, out=out_h, lse=lse_h,
                                stream=stream)
        e2e_step_ms.append((time.perf_counter() - t1) * 1e3)
    e2e_s = reduce_max(time.perf_counter() - t0, ws) / e2e_steps
    h2d = sum(t.numel() * t.element_size() for t in (q, k, v))
    d2h = out_h.numel() * 4 + lse_h.numel() * 4
    e2e_value = ws * f_adj / e2e_s / 1e12

    if rank != 0:
        return
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic",
        "frac_of_dense_bf16_peak": value / ws / peaks["bf16_tflops"],
        "frac_of_dense_bf16_peak_sustained": value / ws / peaks["bf16_tflops_sustained"],
        "peak_source": peak_src,
        "config": forward_config(w, ws),
        "clocks": clk,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "step_ms": [round(t, 2) for t in e2e_step_ms]},
        "gpu_launches": n_upd + n_fz + n_init + n_fin,
        "kernel_ms": {"ring_fused": ms_fz / args.steps,
                      "block_update": ms_upd / args.steps, "state_init": ms_init / args.steps,
                      "finalize": ms_fin / args.steps},
        "roofline": roof,
        "cpu_baseline": cpu,
        "ms_per_step_median": statistics.median(per_step),
        "ms_per_step_best": min(per_step),
        "parity": parity,
    }
    print(json.dumps(line), flush=True)


def main():
    from blockwise_online_softmax_gb300.inputs import WORKLOADS

    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="gqa-128k", choices=sorted(WORKLOADS))
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-step-seconds", type=float, default=6.0)
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--clock-log", default=None,
                    help="directory for the raw nvidia-smi clock samples of the timed region")
    ap.add_argument("--no-check", action="store_true",
                    help="skip the sampled-row parity check of the timed run's output")
    ap.add_argument("--layout", default="contiguous", choices=["contiguous", "zigzag", "striped"])
    ap.add_argument("--window", type=int, default=0, help="sliding window (0 = none)")
    ap.add_argument("--docs", type=int, default=0, help="packed documents (0 = one sequence)")
    ap.add_argument("--n-valid", type=int, default=-1, help="valid length (-1 = N)")
    ap.add_argument("--decode", default=None, choices=["decode-1m", "decode-1m-q4"],
                    help="time the decode path on this workload instead")
    ap.add_argument("--backward", action="store_true",
                    help="time the backward ring (ra_ring_backward) instead")
    ap.add_argument("--state", action="store_true",
                    help="time the state kernels (init, merge, finalize) on the workload's state")
    ap.add_argument("--ring-steps", action="store_true",
                    help="time the step-by-step ring (init, P x ra_ring_step, finalize)")
    ap.add_argument("--heads", type=int, default=0,
                    help="run on the first H query heads (and their KV heads) of the workload "
                         "only; for profiling a full-length slice in a few GB")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be >= 3")
    ws, rank, local = dist_info()
    w = WORKLOADS[args.workload]
    if args.heads:
        w = head_slice(w, args.heads)
    args.mask = MaskRun(w, args.layout, args.window, args.docs, args.n_valid, seed=w.seed)
    if not args.mask.active():
        args.mask = None
    elif args.impl == "reference":
        ap.error("masked runs have no reference arm; time the oracle through cpu_baseline")
    if ws > 1:
        import torch
        import torch.distributed as dist

        backend = "nccl" if (torch.cuda.is_available() and args.impl == "ours") else "gloo"
        if args.impl == "ours" and torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    try:
        if (args.state or args.ring_steps) and args.impl == "reference":
            ap.error("state and ring-step runs have no reference arm; the oracle is the "
                     "cpu_baseline or the parity check")
        if args.state:
            run_state(args, w, ws, rank, local)
        elif args.ring_steps:
            run_steps(args, w, ws, rank, local)
        elif args.backward:
            if args.impl == "reference":
                ap.error("backward runs have no reference arm; the oracle is the cpu_baseline")
            run_backward(args, w, ws, rank, local)
        elif args.decode is not None:
            if args.impl == "reference":
                ap.error("decode runs have no reference arm; time the oracle through cpu_baseline")
            run_decode(args, ws, rank, local)
        elif args.impl == "reference":
            run_reference(args, w, ws, rank)
        else:
            run_ours(args, w, ws, rank, local)
    finally:
        if ws > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    main()
