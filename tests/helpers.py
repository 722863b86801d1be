"""Shared helpers of the GPU tests: run the CUDA path, compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import vision_encoder_varlen_gb300 as vit
from vision_encoder_varlen_gb300 import workloads as wl

# Output tolerance against the fp64 oracle (bf16 in, fp32 accumulate, bf16 out).
MAX_ABS = 2e-2
MEAN_ABS = 2e-3


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_close(gpu: torch.Tensor, ref: np.ndarray, max_abs=MAX_ABS, mean_abs=MEAN_ABS, what=""):
    g = to_f64(gpu)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite GPU output"
    err = np.abs(g - ref)
    mx, mean = float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0
    assert mx <= max_abs, f"{what}: max-abs {mx:.3e} > {max_abs:.1e} (mean {mean:.3e})"
    assert mean <= mean_abs, f"{what}: mean-abs {mean:.3e} > {mean_abs:.1e}"
    return mx, mean


def gpu_full_path(w: wl.Workload, t: dict, device="cuda", status=None):
    """rope_freqs -> qk_norm_rope -> varlen_attn on the GPU; returns (out, q', k', cu, pos, inv_freq)."""
    T, D = w.total_tokens, w.head_dim
    grid = torch.from_numpy(w.grid_hw.copy()).to(device)
    inv_freq, pos, cu = vit.rope_freqs(grid, T, D, w.theta, status=status)
    q, k, v = (t[n].to(device) for n in ("q", "k", "v"))
    nw = t["norm_w"].to(device) if t["norm_w"] is not None else None
    qr, kr = vit.qk_norm_rope(q, k, pos, inv_freq, nw, w.eps)
    out = vit.varlen_attn(qr, kr, v, cu, w.max_seqlen, status=status)
    return out, qr, kr, cu, pos, inv_freq


def stratified_rows(w: wl.Workload, per_long_segment: int = 2048, item_rows: int = 256, item_stride: int = 4,
                    seed: int = 0, small_cap: int = 4096) -> np.ndarray:
    """Rows to check at full size: every row of segments up to small_cap tokens; in longer ones
    per_long_segment rows: the first, second, second-to-last and last rows of the segment, for every
    item_stride-th block of item_rows query rows the first and last row of each of its two 128-row
    halves (the first and last TMEM lane of both Q tiles of a work item), and a seeded random set
    for the rest."""
    rng = np.random.default_rng(seed)
    cu = w.cu_seqlens.astype(np.int64)
    rows = []
    for i in range(w.num_segments):
        a, b = int(cu[i]), int(cu[i + 1])
        L = b - a
        if L == 0:
            continue
        if L <= small_cap:
            rows.append(np.arange(a, b))
            continue
        fixed = {a, a + 1, b - 2, b - 1}
        half = item_rows // 2
        for blk in range(0, (L + item_rows - 1) // item_rows, item_stride):
            q0 = a + blk * item_rows
            fixed.update({q0, q0 + half - 1, q0 + half, q0 + item_rows - 1})
        fixed = np.array(sorted(x for x in fixed if a <= x < b))
        assert len(fixed) <= per_long_segment
        rest = np.setdiff1d(np.arange(a, b), fixed)
        extra = rng.choice(rest, size=min(len(rest), per_long_segment - len(fixed)), replace=False)
        rows.append(np.unique(np.concatenate([fixed, extra])))
    return np.concatenate(rows) if rows else np.zeros(0, dtype=np.int64)


def sample_rows(w: wl.Workload, big_rows: int, seed: int = 0, small_cap: int = 4096) -> np.ndarray:
    """Rows to check: every row of segments up to small_cap tokens; for longer ones the first, last,
    128-tile boundary rows and a seeded random set, big_rows in total per long segment."""
    rng = np.random.default_rng(seed)
    cu = w.cu_seqlens.astype(np.int64)
    rows = []
    for i in range(w.num_segments):
        a, b = int(cu[i]), int(cu[i + 1])
        L = b - a
        if L == 0:
            continue
        if L <= small_cap:
            rows.append(np.arange(a, b))
            continue
        fixed = {a, a + 1, b - 2, b - 1}
        for tb in range(128, L, 128 * max(1, L // (128 * 16))):
            fixed.update({a + tb - 1, a + tb})
        fixed = sorted(x for x in fixed if a <= x < b)
        extra = rng.choice(np.arange(a, b), size=max(0, big_rows - len(fixed)), replace=False)
        rows.append(np.unique(np.concatenate([np.array(fixed), extra])))
    return np.concatenate(rows) if rows else np.zeros(0, dtype=np.int64)
