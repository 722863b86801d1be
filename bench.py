"""Benchmark of the varlen ViT attention hot path on GB300.

One step = the whole path over one packed batch: the 2D RoPE table and
positions (vit_rope_freqs), the fused QK-RMSNorm + RoPE prologue
(vit_qk_norm_rope) and the segment-aware varlen attention (vit_varlen_attn,
scheduler + attention kernels). Metric: useful attention TFLOP/s,
4 * sum(L_i^2) * H * D per step (cross-segment blocks and tile padding are not
counted), plus tokens/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config 1..5] [--impl ours|reference]

Prints one JSON line (rank 0). With N > 1 (launched by torchrun) every rank
runs its own replica of the batch: there is no exchange on this path.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from vision_encoder_varlen_gb300 import workloads as wl  # noqa: E402

METRIC = "varlen ViT attention TFLOP/s (4·ΣLi²·H·D) and tokens/s on 1 GB300; % of BF16 peak"
L2_BYTES = 129 * 2 ** 20
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return PEAKS_FALLBACK, "fallback"


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max(x: float, device) -> float:
    """Max over ranks (identity without an initialised process group)."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def rank_inputs(w: wl.Workload, rank: int) -> dict:
    """This rank's shard of the job: a batch of the workload's shape with its own seeded values,
    so N ranks process N different batches (weak scaling, no exchange between ranks)."""
    return w.tensors(seed_offset=rank)


def job_tflops(flops_per_rank: float, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: every rank's useful flops over the slowest rank's step time."""
    return flops_per_rank * world / (ms_per_step * 1e-3) / 1e12


# ------------------------------------------------------------------ clocks during the timed region

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        self.f = None
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:             # no nvidia-smi: the line reports clocks as null
            self.proc = None
            if self.f is not None:
                self.f.close()
            if self.path and os.path.exists(self.path):
                os.unlink(self.path)
            self.path = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return None
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx = max(mx, float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        load = [s for s in sm if s > 0.5 * mx] or sm
        return {"sm_mhz": statistics.median(load), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ the GPU arm

class Path:
    """Device-resident buffers and the three calls of one step."""

    def __init__(self, vit, w: wl.Workload, t: dict, device, lse: bool = False, interleaved: bool = False,
                 fused_q: bool = False, short_max: int | None = None):
        self.vit, self.w = vit, w
        self.interleaved, self.fused_q, self.short_max = interleaved, fused_q, short_max
        self.max_pos = int(w.grid_hw.max())
        T, H, D, B = w.total_tokens, w.heads, w.head_dim, w.num_segments
        self.grid = torch.from_numpy(w.grid_hw.copy()).to(device)
        self.q, self.k, self.v = (t[n].to(device) for n in ("q", "k", "v"))
        self.nw = t["norm_w"].to(device) if t["norm_w"] is not None else None
        self.qr = torch.empty_like(self.q)
        self.kr = torch.empty_like(self.k)
        self.out = torch.empty_like(self.q)
        self.lse = torch.empty((T, H), dtype=torch.float32, device=device) if lse else None
        self.ws = torch.empty(vit.workspace_size(T, H, B, D), dtype=torch.uint8, device=device)
        self.status = vit.new_status(device)

    def step(self):
        vit, w = self.vit, self.w
        inv_freq, pos, cu = vit.rope_freqs(self.grid, w.total_tokens, w.head_dim, w.theta, status=self.status)
        if self.fused_q:
            # position table, K pre-stage, attention that normalises and rotates Q as it loads it
            cs = vit.rope_table(inv_freq, w.head_dim, self.max_pos)
            vit.encoder_attn(self.q, self.k, self.v, cu, w.max_seqlen, pos, inv_freq, cs, self.nw, w.eps,
                             interleaved=self.interleaved, k_out=self.kr, out=self.out, workspace=self.ws,
                             status=self.status, lse=self.lse, short_max=self.short_max)
            return
        vit.qk_norm_rope(self.q, self.k, pos, inv_freq, self.nw, w.eps, q_out=self.qr, k_out=self.kr,
                         interleaved=self.interleaved)
        vit.varlen_attn(self.qr, self.kr, self.v, cu, w.max_seqlen, out=self.out, workspace=self.ws,
                        status=self.status, lse=self.lse, short_max=self.short_max)


class E2EPipeline:
    """The path as a serving loop runs it, through the public API from pinned host buffers: every
    step uploads its inputs (q, k, v, the grid list, the norm weights) and downloads its output.
    Uploads go on one copy stream and downloads on another, into two sets of device buffers, so
    step i+1's inputs travel up and step i's output travels down while a step computes. (Three
    upload streams measured the same: the host link, not one copy engine, is the limit.)"""

    def __init__(self, vit, w, host, device, fused_q=False):
        self.vit, self.w, self.host, self.fused_q = vit, w, host, fused_q
        T, H, D, B = w.total_tokens, w.heads, w.head_dim, w.num_segments
        self.up = torch.cuda.Stream(device)
        self.down = torch.cuda.Stream(device)
        self.bufs = []
        for _ in range(2):
            self.bufs.append({
                "grid": torch.empty_like(host["grid"], device=device),
                "q": torch.empty((T, H, D), dtype=torch.bfloat16, device=device),
                "k": torch.empty((T, H, D), dtype=torch.bfloat16, device=device),
                "v": torch.empty((T, H, D), dtype=torch.bfloat16, device=device),
                "nw": torch.empty_like(host["nw"], device=device) if host["nw"] is not None else None,
                "out": torch.empty((T, H, D), dtype=torch.bfloat16, device=device),
                "ws": torch.empty(vit.workspace_size(T, H, B, D), dtype=torch.uint8, device=device),
                "uploaded": torch.cuda.Event(), "consumed": torch.cuda.Event(), "downloaded": torch.cuda.Event(),
                "used": False,
            })

    def _upload(self, b):
        buf, host = self.bufs[b], self.host
        with torch.cuda.stream(self.up):
            if buf["used"]:
                self.up.wait_event(buf["consumed"])          # the step that last read these inputs is done
            for name in ("grid", "q", "k", "v", "nw"):
                if buf[name] is not None:
                    buf[name].copy_(host[name], non_blocking=True)
            buf["uploaded"].record(self.up)

    def _compute(self, b):
        vit, w, buf = self.vit, self.w, self.bufs[b]
        cur = torch.cuda.current_stream()
        cur.wait_event(buf["uploaded"])
        if buf["used"]:
            cur.wait_event(buf["downloaded"])                # this buffer's previous output has left
        inv_freq, pos, cu = vit.rope_freqs(buf["grid"], w.total_tokens, w.head_dim, w.theta)
        if self.fused_q:
            cs = vit.rope_table(inv_freq, w.head_dim, int(w.grid_hw.max()))
            vit.encoder_attn(buf["q"], buf["k"], buf["v"], cu, w.max_seqlen, pos, inv_freq, cs, buf["nw"], w.eps,
                             k_out=buf["k"], out=buf["out"], workspace=buf["ws"])
        else:
            vit.qk_norm_rope(buf["q"], buf["k"], pos, inv_freq, buf["nw"], w.eps, inplace=True)
            vit.varlen_attn(buf["q"], buf["k"], buf["v"], cu, w.max_seqlen, out=buf["out"], workspace=buf["ws"])
        buf["consumed"].record(cur)
        buf["used"] = True

    def _download(self, b):
        buf = self.bufs[b]
        with torch.cuda.stream(self.down):
            self.down.wait_event(buf["consumed"])
            self.host["out"].copy_(buf["out"], non_blocking=True)
            buf["downloaded"].record(self.down)

    def run(self, steps: int, start_event=None):
        """Enqueue `steps` steps; the current stream waits for the last download at the end."""
        if start_event is not None:
            self.up.wait_event(start_event)
        self._upload(0)
        for i in range(steps):
            if i + 1 < steps:
                self._upload((i + 1) % 2)
            self._compute(i % 2)
            self._download(i % 2)
        torch.cuda.current_stream().wait_event(self.bufs[(steps - 1) % 2]["downloaded"])


def load_traffic(kernel: str, workload: str):
    """dram read+write bytes per launch of `kernel` on `workload`, from the committed ncu summary
    (profiles/traffic.json), or None when there is none or the kernel source changed since."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    for e in d.get(kernel, []):
        if e.get("workload") != workload or not e.get("source"):
            continue
        with open(os.path.join(ROOT, e["source"]), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest()[:16] != e.get("source_sha256_16"):
                return None
        return e.get("bytes_per_launch")
    return None


def kernel_algorithmic_flops(w: wl.Workload, kernel: str, short_max: int) -> float:
    """Useful flops a kernel processes per step: 4 L^2 H D over the segments it owns
    (attn_long: segments longer than min(short_max, 64) tokens; attn_tiny: the rest)."""
    tiny_max = min(short_max, 64)
    L = w.lengths.astype(np.float64)
    L = L[L > tiny_max] if kernel == "attn_long" else L[L <= tiny_max]
    return float(4.0 * np.sum(L * L) * w.heads * w.head_dim)


def cpu_baseline_sample(w: wl.Workload, t: dict, target_s: float):
    """The fp64 oracle, as it stands, on a bounded sample: the first query rows of
    the longest image (all heads, all its keys), grown until ~target_s of CPU work."""
    import oracle
    bits = [wl.bf16_bits(t[n]) for n in ("q", "k", "v")]
    nw = wl.bf16_bits(t["norm_w"]) if t["norm_w"] is not None else None
    cu = w.cu_seqlens
    seg = int(np.argmax(w.lengths))
    a, L = int(cu[seg]), int(w.lengths[seg])
    rows_n, spent, flops, calls = 4, 0.0, 0.0, 0
    t_start = time.perf_counter()
    while spent < target_s:
        n = min(rows_n, L)
        rows = np.arange(a, a + n)
        t0 = time.perf_counter()
        oracle.full_path(w.grid_hw, *bits, nw, w.eps, w.theta, rows=rows)
        dt = time.perf_counter() - t0
        spent += dt
        flops += 4.0 * n * L * w.heads * w.head_dim
        calls += 1
        if dt < target_s / 8:
            rows_n *= 2
    wall = time.perf_counter() - t_start
    return {"value": flops / wall / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{calls} oracle calls over query rows [first {rows_n} max] of the {L}-token image, all "
                      f"{w.heads} heads and all its keys (RoPE/norm of every token included), {wall:.1f} s wall",
            "seconds": wall, "useful_flops": flops}


SUSTAINED_AFTER_S = 2.0      # a timed region at least this long is judged against the sustained peak


def working_set_bytes(w: wl.Workload) -> int:
    """q, k, v, q', k', out of one step."""
    return 6 * w.total_tokens * w.heads * w.head_dim * 2


def needs_flush(w: wl.Workload) -> bool:
    return working_set_bytes(w) < 2 * L2_BYTES


def config_dict(w: wl.Workload, args, world: int) -> dict:
    """The workload a line measures; the same dict for both arms."""
    ws = working_set_bytes(w)
    return {"workload": w.name, "tokens": w.total_tokens, "segments": w.num_segments, "heads": w.heads,
            "head_dim": w.head_dim, "qk_norm": w.qk_norm, "max_seqlen": w.max_seqlen,
            "useful_flops_per_step": w.useful_flops,
            "rope": "interleaved" if args.interleaved else "rotate_half", "lse": bool(args.lse),
            "q_prologue": "fused into the attention Q load" if args.fused_q else "separate pass",
            "l2": "L2 flushed between steps" if needs_flush(w) else
            f"inputs larger than L2 ({ws / 2 ** 20:.0f} MiB working set)",
            "parallelism": f"data-parallel over {world} ranks, one batch each, no exchange" if world > 1
            else "single"}


def time_steps(step, steps: int, stream, flush_buf) -> float:
    """Total device ms of `steps` calls of step(): back to back when flush_buf is None, else
    each step alone after a write of flush_buf (larger than L2), events around the step only."""
    if flush_buf is None:
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
        return ev0.elapsed_time(ev1)
    total = 0.0
    for _ in range(steps):
        flush_buf.zero_()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        step()
        ev1.record(stream)
        torch.cuda.synchronize()
        total += ev0.elapsed_time(ev1)
    return total


def roofline_entry(vit, w: wl.Workload, kt: dict, short_max: int, peaks: dict, peaks_src: str, timed_s: float,
                   fused_q: bool):
    """The dominant kernel's achieved rate: its algorithmic work per launch over its mean
    event-timed launch duration, against the measured peak of its bound. A contraction takes the
    burst bf16 peak unless its timed region ran SUSTAINED_AFTER_S or longer."""
    if not kt:
        return None
    dom = max(kt.items(), key=lambda kv: kv[1][1])[0]
    n, tot = kt[dom]
    avg_s = tot / n * 1e-3
    T, H, D = w.total_tokens, w.heads, w.head_dim
    if dom == "attn_long":
        alg = kernel_algorithmic_flops(w, dom, short_max)
        key = "bf16_tflops_sustained" if timed_s >= SUSTAINED_AFTER_S else "bf16_tflops"
        peak = peaks[key]
        achieved = alg / avg_s / 1e12
        return {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": load_traffic(dom, w.name),
                "peak_source": f"{peaks_src} {key} (timed region {timed_s:.2f} s)",
                "algorithmic_flops_per_launch": alg, "avg_ms": tot / n}
    tiny_max = min(short_max, 64)
    L = w.lengths
    if dom == "attn_tiny":           # q, k, v read and out written once per token it owns
        alg = 8.0 * float(L[L <= tiny_max].sum()) * H * D
    elif dom == "qk_norm_rope":      # q and k (k alone with --fused-q) read and written once
        alg = (4.0 if fused_q else 8.0) * T * H * D
    else:
        alg = 8.0 * T
    achieved = alg / avg_s / 1e9
    return {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / peaks["hbm_gbs"], "traffic": load_traffic(dom, w.name),
            "peak_source": f"{peaks_src} hbm_gbs", "algorithmic_bytes_per_launch": alg, "avg_ms": tot / n}


def measure_device(vit, path, w, steps: int, warmup: int, stream, device, flush_buf, barrier=lambda: None):
    """Warm up, then time `steps` steps with every launch event-timed on its stream.
    Returns (ms per step, {kernel: (launches, total ms)}, launches, clock summary)."""
    for _ in range(warmup):
        path.step()
    torch.cuda.synchronize()
    code = vit.read_status(path.status)
    if code != 0:
        raise RuntimeError(f"{w.name}: device status {code}: {vit.status_string(code)}")
    barrier()
    torch.cuda.synchronize()
    launches0 = vit.launch_count()
    vit.kernel_timing_read()
    with ClockSampler(device.index or 0) as clocks:
        vit.kernel_timing(True)
        try:
            total_ms = time_steps(path.step, steps, stream, flush_buf if needs_flush(w) else None)
        finally:
            vit.kernel_timing(False)
        kt = vit.kernel_timing_read()
    torch.cuda.synchronize()
    barrier()
    return total_ms / steps, kt, vit.launch_count() - launches0, clocks.summary()


def measure_graph(path, w, steps: int, stream, flush_buf) -> float:
    """ms per step when the whole step is captured once in a CUDA graph and replayed (how a
    serving loop that buckets its shapes runs it: no per-launch host cost)."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        path.step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        path.step()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    ms = time_steps(g.replay, steps, stream, flush_buf if needs_flush(w) else None) / steps
    del g
    return ms


def per_config_entry(vit, idx: int, args, rank: int, device, stream, flush_buf, peaks, peaks_src) -> dict:
    """One of the smaller workloads, measured in the same run as the headline line."""
    w = wl.make_config(idx)
    path = Path(vit, w, rank_inputs(w, rank), device, lse=args.lse, interleaved=args.interleaved,
                fused_q=args.fused_q, short_max=args.short_max)
    ms, kt, launches, clk = measure_device(vit, path, w, args.steps, args.warmup, stream, device, flush_buf)
    short_max = args.short_max if args.short_max is not None else vit.DEFAULT_SHORT_MAX
    timed_s = ms * args.steps / 1e3
    graph_ms = measure_graph(path, w, args.steps, stream, flush_buf)
    return {"config": config_dict(w, args, 1), "ms_per_step": ms, "tflops": w.useful_flops / (ms * 1e-3) / 1e12,
            "tokens_per_s": w.total_tokens / (ms * 1e-3), "graph_ms_per_step": graph_ms,
            "graph_tflops": w.useful_flops / (graph_ms * 1e-3) / 1e12,
            "kernels": {name: {"launches": n, "avg_ms": tot / max(n, 1)} for name, (n, tot) in kt.items()},
            "gpu_launches": launches, "clocks": clk,
            "roofline": roofline_entry(vit, w, kt, short_max, peaks, peaks_src, timed_s, args.fused_q)}


def run_ours(args, rank, world, local):
    import vision_encoder_varlen_gb300 as vit
    from vision_encoder_varlen_gb300 import _build
    if rank == 0:
        _build.build()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    w = wl.make_config(args.config)
    t = rank_inputs(w, rank)
    T, H, D = w.total_tokens, w.heads, w.head_dim
    path = Path(vit, w, t, device, lse=args.lse, interleaved=args.interleaved, fused_q=args.fused_q,
                short_max=args.short_max)
    stream = torch.cuda.current_stream()
    tensor_bytes = T * H * D * 2
    flush_buf = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device=device)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    # ---- timed region: K steps, per-kernel CUDA events recorded live on the launch stream
    local_ms, kt, launches, clk = measure_device(vit, path, w, args.steps, args.warmup, stream, device, flush_buf,
                                                 barrier)
    ms = reduce_max(local_ms, device)

    # ---- end to end through the public API from pinned host memory
    e2e = None
    if not args.no_e2e:
        host = {"grid": torch.from_numpy(w.grid_hw.copy()).pin_memory(),
                "q": t["q"].pin_memory(), "k": t["k"].pin_memory(), "v": t["v"].pin_memory(),
                "nw": t["norm_w"].pin_memory() if t["norm_w"] is not None else None,
                "out": torch.empty((T, H, D), dtype=torch.bfloat16).pin_memory()}
        h2d = 3 * tensor_bytes + host["grid"].numel() * 4 + (host["nw"].numel() * 2 if host["nw"] is not None else 0)
        d2h = tensor_bytes
        pipe = E2EPipeline(vit, w, host, device, args.fused_q)
        pipe.run(3)                                          # warm-up
        torch.cuda.synchronize()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e2e_steps = max(2, args.steps)                       # same count as the device-timed leg
        e0.record(stream)
        pipe.run(e2e_steps, start_event=e0)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = reduce_max(e0.elapsed_time(e1) / e2e_steps, device)
        e2e = {"value": job_tflops(w.useful_flops, world, e2e_ms), "unit": "TFLOP/s", "ms_per_step": e2e_ms,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "overlap": "step i+1's upload and step i's download on two copy streams run during compute"}

    # ---- the other workloads of the study, each measured alone in this run (one GPU only), and
    # the short-segment workload (4096 images of 16-64 tokens) that the tiny-segment kernel serves
    per_config = None
    if world == 1 and args.config == 5 and not args.no_per_config:
        peaks, peaks_src = load_peaks()
        per_config = {str(i): per_config_entry(vit, i, args, rank, device, stream, flush_buf, peaks, peaks_src)
                      for i in (1, 2, 3, 4, 7)}

    if rank != 0:
        return
    peaks, peaks_src = load_peaks()
    flops = w.useful_flops
    value = job_tflops(flops, world, ms)
    short_max = args.short_max if args.short_max is not None else vit.DEFAULT_SHORT_MAX
    timed_s = ms * args.steps / 1e3
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_dict(w, args, world),
        "tokens_per_s": T * world / (ms * 1e-3),
        "frac_of_bf16_peak": value / world / peaks["bf16_tflops"],
        "clocks": clk,
        "e2e": e2e,
        "gpu_launches": launches,
        "kernels": {name: {"launches": n, "avg_ms": tot / max(n, 1)} for name, (n, tot) in kt.items()},
        "roofline": roofline_entry(vit, w, kt, short_max, peaks, peaks_src, timed_s, args.fused_q),
    }
    if per_config is not None:
        line["per_config"] = per_config
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_sample(w, t, args.cpu_seconds)
    print(json.dumps(line), flush=True)


def run_split_sweep(args):
    """Attention time with every segment on the tiny-segment (warp-MMA) kernel vs every segment on
    the tcgen05 kernel, for bands of random segment lengths up to the tiny kernel's 64 tokens (one
    JSON line per band and head_dim)."""
    import vision_encoder_varlen_gb300 as vit
    from vision_encoder_varlen_gb300 import _build
    _build.build()
    rng = np.random.default_rng(0)
    for D in (80, 128):
        for lo, hi in ((4, 16), (16, 32), (32, 64)):
            lengths = rng.integers(lo, hi + 1, size=8192 if hi <= 32 else (4096 if hi <= 128 else 2048))
            w = wl.from_lengths(lengths, 16, D, max_seqlen_meta=4096)
            g = torch.Generator(device="cuda").manual_seed(1)
            T = w.total_tokens
            q, k, v = (torch.randn(T, 16, D, device="cuda", generator=g).to(torch.bfloat16) for _ in range(3))
            cu = torch.from_numpy(w.cu_seqlens).cuda()
            ws = torch.empty(vit.workspace_size(T, 16, w.num_segments, D), dtype=torch.uint8, device="cuda")
            out = torch.empty_like(q)
            res = {}
            for name, sm in (("tiny_kernel_ms", 64), ("tcgen05_kernel_ms", 0)):
                for _ in range(args.warmup):
                    vit.varlen_attn(q, k, v, cu, 4096, out=out, workspace=ws, short_max=sm)
                torch.cuda.synchronize()
                vit.kernel_timing_read()
                vit.kernel_timing(True)
                for _ in range(args.steps):
                    vit.varlen_attn(q, k, v, cu, 4096, out=out, workspace=ws, short_max=sm)
                vit.kernel_timing(False)
                kt = vit.kernel_timing_read()
                res[name] = sum(t for _, t in kt.values()) / args.steps
            print(json.dumps({"sweep": "split", "head_dim": D, "lengths": [lo, hi], "segments": int(len(lengths)),
                              "tokens": T, **res}), flush=True)


def run_reference(args, rank, world):
    """The reference arm: the fp64 oracle, as it stands, on the host cores; each
    step is a bounded sample (query rows of the longest image, all heads)."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    w = wl.make_config(args.config)
    t = w.tensors()
    bits = [wl.bf16_bits(t[n]) for n in ("q", "k", "v")]
    nw = wl.bf16_bits(t["norm_w"]) if t["norm_w"] is not None else None
    seg = int(np.argmax(w.lengths))
    a, L = int(w.cu_seqlens[seg]), int(w.lengths[seg])
    n = max(1, min(L, args.ref_rows))
    rows = np.arange(a, a + n)
    for _ in range(args.warmup):
        oracle.full_path(w.grid_hw, *bits, nw, w.eps, w.theta, rows=rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.full_path(w.grid_hw, *bits, nw, w.eps, w.theta, rows=rows)
    wall = time.perf_counter() - t0
    flops = 4.0 * n * L * w.heads * w.head_dim
    value = flops * args.steps / wall / 1e12
    sample = f"{n} query rows of the {L}-token image per step, all {w.heads} heads and all its keys"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": wall / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(w, args, world),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=5, choices=[1, 2, 3, 4, 5, 6, 7],
                    help="workload 1..5 (default 5); 6 = a single 128x128 image for profiler captures; "
                         "7 = 4096 small images for the tiny-segment kernel")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end measurement")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-workload block (workloads 1-4 and the short-segment workload 7, measured "
                         "after the headline workload 5)")
    ap.add_argument("--sweep-split", action="store_true",
                    help="time both attention kernels over bands of segment lengths and exit")
    ap.add_argument("--short-max", type=int, default=None,
                    help="segments longer than min(this, 64) run on the tcgen05 kernel (library default 64)")
    ap.add_argument("--ref-rows", type=int, default=16)
    ap.add_argument("--lse", action="store_true", help="also write the per-row log-sum-exp [T, H] each step")
    ap.add_argument("--fused-q", action="store_true",
                    help="normalise and rotate Q inside the attention kernels (K alone in the pre-stage)")
    ap.add_argument("--interleaved", action="store_true",
                    help="rotate adjacent pairs (the complex_rope mode) instead of (m, m + D/2)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local = dist_env()
    if args.sweep_split:
        run_split_sweep(args)
        return
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    try:
        run_ours(args, rank, world, local)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
