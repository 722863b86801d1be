"""Residual report: the CUDA path and the pages' eager rounding, each against the exact oracle.

Not a test (nothing here passes or fails). For each workload it prints how far the CUDA
path's attention output is from the exact fp64 oracle, how far the rounding mimic of the
eager modules (oracle/mimic.py) is from the same oracle, and how far the two are from each
other; for the prologue, the share of q', k' elements where the CUDA path and the mimic
give the same bf16 bits and the largest difference in bf16 units of the element's
rotation-pair norm. Rows: every row of
segments up to ``--small-cap`` tokens, a sample of the longer ones (first, last, 128-tile
boundaries and seeded random rows).

    python tests/report_residuals.py               # CUDA path, mimic, oracle (GPU + built library)
    python tests/report_residuals.py --cpu-only    # mimic against the oracle only
"""
from __future__ import annotations

import argparse
import os
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import oracle                                               # noqa: E402
from oracle import mimic                                    # noqa: E402
from vision_encoder_varlen_gb300 import workloads as wl     # noqa: E402


def _rows(w: wl.Workload, big_rows: int, small_cap: int, seed: int = 0) -> np.ndarray:
    rng = np.random.default_rng(seed)
    cu = w.cu_seqlens.astype(np.int64)
    out = []
    for i in range(w.num_segments):
        a, b = int(cu[i]), int(cu[i + 1])
        if b - a <= small_cap:
            out.append(np.arange(a, b))
            continue
        fixed = {a, a + 1, b - 2, b - 1}
        for tb in range(128, b - a, 128 * max(1, (b - a) // (128 * 16))):
            fixed.update({a + tb - 1, a + tb})
        fixed = np.array(sorted(fixed))
        extra = rng.choice(np.arange(a, b), size=max(0, big_rows - fixed.size), replace=False)
        out.append(np.unique(np.concatenate([fixed, extra])))
    return np.concatenate(out) if out else np.zeros(0, dtype=np.int64)


def _pair_units(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    """|a - b| in bf16 units (2^(floor(log2 r) - 7)) of r, the norm of the element's
    rotate-half pair (m, m + D/2). A rotation that nearly cancels leaves an output far
    smaller than r, where one fp32 rounding more or less (a fused multiply-add, a one-unit
    sin or rsqrt) is many units of that output but well under one unit of r."""
    a, b = oracle.widen(a_bits), oracle.widen(b_bits)
    D = b.shape[-1]
    r = np.sqrt(b[..., : D // 2] ** 2 + b[..., D // 2:] ** 2)
    r = np.concatenate([r, r], axis=-1)
    unit = 2.0 ** (np.floor(np.log2(np.maximum(r, 2.0 ** -126))) - 7)
    return np.abs(a - b) / unit


def _gpu(w: wl.Workload, t: dict, rows: np.ndarray):
    """The CUDA path (rope_freqs -> qk_norm_rope -> varlen_attn); returns out rows and q', k' bits."""
    import torch
    import vision_encoder_varlen_gb300 as vit

    T, D = w.total_tokens, w.head_dim
    grid = torch.from_numpy(w.grid_hw.copy()).cuda()
    inv_freq, pos, cu = vit.rope_freqs(grid, T, D, w.theta)
    q, k, v = (t[n].cuda() for n in ("q", "k", "v"))
    nw = t["norm_w"].cuda() if t["norm_w"] is not None else None
    qr, kr = vit.qk_norm_rope(q, k, pos, inv_freq, nw, w.eps)
    out = vit.varlen_attn(qr, kr, v, cu, w.max_seqlen)
    torch.cuda.synchronize()
    idx = torch.from_numpy(rows).cuda()
    return (out[idx].float().cpu().numpy().astype(np.float64),
            wl.bf16_bits(qr[idx].cpu()), wl.bf16_bits(kr[idx].cpu()))


def report(idx: int, use_gpu: bool, big_rows: int, small_cap: int) -> dict:
    w = wl.make_config(idx)
    t = w.tensors()
    rows = _rows(w, big_rows, small_cap)
    bits = {n: wl.bf16_bits(t[n]) for n in ("q", "k", "v")}
    nw = None if t["norm_w"] is None else wl.bf16_bits(t["norm_w"])
    t0 = time.time()
    exact = oracle.full_path(w.grid_hw, bits["q"], bits["k"], bits["v"], nw, w.eps, w.theta, rows=rows)
    eager = mimic.full_path(w.grid_hw, bits["q"], bits["k"], bits["v"], nw, w.eps, w.theta, rows=rows)
    res = {"workload": w.name, "rows": int(rows.size), "T": w.total_tokens,
           "mimic_vs_exact": (float(np.max(np.abs(eager - exact))), float(np.mean(np.abs(eager - exact))))}
    if use_gpu:
        out, qb, kb = _gpu(w, t, rows)
        _, pos = oracle.grid_positions(w.grid_hw)
        res["gpu_vs_exact"] = (float(np.max(np.abs(out - exact))), float(np.mean(np.abs(out - exact))))
        res["gpu_vs_mimic"] = (float(np.max(np.abs(out - eager))), float(np.mean(np.abs(out - eager))))
        same, worst = [], 0.0
        for name, gb, wrow in (("q", qb, 0), ("k", kb, 1)):
            ref = mimic.norm_rope(bits[name][rows], pos[rows], w.theta, None if nw is None else nw[wrow],
                                  w.qk_norm, w.eps)
            same.append(float(np.mean(gb == ref)))
            worst = max(worst, float(_pair_units(gb, ref).max()))
        res["prologue_same_bits"] = min(same)
        res["prologue_max_units"] = worst
    res["seconds"] = round(time.time() - t0, 1)
    return res


def main() -> None:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--cpu-only", action="store_true", help="skip the CUDA path")
    ap.add_argument("--workloads", default="1,2,3,4,5")
    ap.add_argument("--big-rows", type=int, default=256, help="rows sampled per long segment")
    ap.add_argument("--small-cap", type=int, default=1024, help="segments up to this many tokens: every row")
    a = ap.parse_args()
    print("| workload | rows | mimic - exact (max / mean) | CUDA - exact (max / mean) | CUDA - mimic (max / mean)"
          " | prologue vs mimic: same bits, max units of pair norm | s |")
    print("|---|---|---|---|---|---|---|")
    for idx in (int(x) for x in a.workloads.split(",")):
        r = report(idx, not a.cpu_only, a.big_rows, a.small_cap)
        fmt = lambda p: f"{p[0]:.2e} / {p[1]:.2e}"          # noqa: E731
        gpu = (fmt(r["gpu_vs_exact"]), fmt(r["gpu_vs_mimic"]),
               f"{100 * r['prologue_same_bits']:.3f} %, {r['prologue_max_units']:.2f}") if "gpu_vs_exact" in r \
            else ("-", "-", "-")
        cells = [r["workload"], r["rows"], fmt(r["mimic_vs_exact"]), *gpu, r["seconds"]]
        print("| " + " | ".join(str(c) for c in cells) + " |", flush=True)


if __name__ == "__main__":
    main()
