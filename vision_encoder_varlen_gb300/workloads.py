"""Seeded synthetic workloads for varlen ViT encoder attention.

This module only builds inputs: image patch grids, the packed-token offsets
that delimit them, bf16 q/k/v drawn from N(0, 1) and QK-RMSNorm weights drawn
from 1 + 0.1*N(0, 1). It holds none of the attention, norm or RoPE arithmetic,
so the CUDA path and the CPU oracle can both be fed from it.

Workload shapes follow the five cases of the varlen ViT attention study:
a tiny two-image case, one 32x32 image, eight mid-size images with QK-norm,
32 log-uniform near-square images at head_dim 128, and one 256x256 image mixed
with seven small ones whose max_seqlen metadata is padded to the 131072 bucket
(the cuDNN CUDA-graph bucket table of tokenspeed ``mm_encoder_attention.py``,
``VIT_CUDNN_SEQLEN_BUCKETS``).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

SEED_BASE = 20261202


@dataclass(frozen=True)
class Workload:
    name: str
    grids: tuple            # ((h, w), ...) patch grid per image, in packing order
    heads: int
    head_dim: int
    qk_norm: bool
    eps: float = 1e-6
    theta: float = 10000.0
    max_seqlen_meta: int | None = None   # padded bound passed as max_seqlen; None = true max
    seed: int = SEED_BASE
    note: str = field(default="", compare=False)

    # ---- packing metadata (plain bookkeeping of the grid list) ----
    @property
    def lengths(self) -> np.ndarray:
        return np.array([h * w for h, w in self.grids], dtype=np.int64)

    @property
    def num_segments(self) -> int:
        return len(self.grids)

    @property
    def total_tokens(self) -> int:
        return int(self.lengths.sum())

    @property
    def cu_seqlens(self) -> np.ndarray:
        cu = np.zeros(self.num_segments + 1, dtype=np.int64)
        cu[1:] = np.cumsum(self.lengths)
        return cu.astype(np.int32)

    @property
    def grid_hw(self) -> np.ndarray:
        return np.array(self.grids, dtype=np.int32).reshape(-1, 2)

    @property
    def max_seqlen(self) -> int:
        true_max = int(self.lengths.max()) if self.num_segments else 0
        if self.max_seqlen_meta is None:
            return max(true_max, 1)
        return int(self.max_seqlen_meta)

    @property
    def useful_flops(self) -> float:
        """4 * sum(L_i^2) * H * D: QK^T and PV inside each segment only."""
        L = self.lengths.astype(np.float64)
        return float(4.0 * np.sum(L * L) * self.heads * self.head_dim)

    # ---- seeded tensors ----
    def tensors(self, seed_offset: int = 0) -> dict:
        """q, k, v as bf16 CPU tensors [T, H, D]; norm_w bf16 [2, D] (q row, k row) or None."""
        g = torch.Generator().manual_seed(self.seed + seed_offset)
        T, H, D = self.total_tokens, self.heads, self.head_dim
        out = {}
        for name in ("q", "k", "v"):
            out[name] = torch.randn((T, H, D), generator=g, dtype=torch.float32).to(torch.bfloat16)
        if self.qk_norm:
            w = 1.0 + 0.1 * torch.randn((2, D), generator=g, dtype=torch.float32)
            out["norm_w"] = w.to(torch.bfloat16)
        else:
            out["norm_w"] = None
        return out


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bf16 bit patterns of a CPU bf16 tensor as a uint16 numpy array (same shape)."""
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def bits_to_bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


def _uniform_grids(rng: np.random.Generator, n: int, h_lo, h_hi, w_lo, w_hi):
    return tuple((int(rng.integers(h_lo, h_hi + 1)), int(rng.integers(w_lo, w_hi + 1))) for _ in range(n))


def _near_square_grids(rng: np.random.Generator, n: int, lo: int, hi: int):
    grids = []
    for _ in range(n):
        L = math.exp(rng.uniform(math.log(lo), math.log(hi)))
        h = max(1, int(round(math.sqrt(L))))
        w = max(1, int(round(L / h)))
        grids.append((h, w))
    return tuple(grids)


def make_config(idx: int) -> Workload:
    """The five workloads, index 1..5."""
    rng = np.random.default_rng(SEED_BASE + idx)
    seed = SEED_BASE + 100 * idx
    if idx == 1:
        return Workload("tiny_8x8+6x10_h4_d32", ((8, 8), (6, 10)), 4, 32, False, seed=seed)
    if idx == 2:
        return Workload("single_32x32_h16_d80", ((32, 32),), 16, 80, False, seed=seed)
    if idx == 3:
        return Workload("8img_16x16..64x48_h16_d80_qknorm", _uniform_grids(rng, 8, 16, 64, 16, 48),
                        16, 80, True, seed=seed)
    if idx == 4:
        return Workload("32img_logu64..4096_h16_d128_qknorm", _near_square_grids(rng, 32, 64, 4096),
                        16, 128, True, seed=seed)
    if idx == 5:
        grids = ((256, 256),) + _uniform_grids(rng, 7, 8, 32, 8, 32)
        return Workload("mixed_256x256+7small_h16_d80_qknorm_max131072", grids, 16, 80, True,
                        max_seqlen_meta=131072, seed=seed)
    if idx == 6:
        # not one of the five study shapes: a single 128x128 image used for profiler captures
        # (168 MB of q/k/v/out, above the 129 MB L2, ~1.5 ms of attention)
        return Workload("profile_128x128_h16_d80_qknorm", ((128, 128),), 16, 80, True, seed=seed)
    if idx == 7:
        # not one of the five study shapes: 4096 small images (16..64 tokens) that all run on the
        # tiny-segment kernel, for its HBM-bandwidth measurement (~1.5 GB of q/k/v/out)
        return Workload("short_4096img_4..8_h16_d80_qknorm", _uniform_grids(rng, 4096, 4, 8, 4, 8), 16, 80, True,
                        seed=seed)
    raise ValueError(f"no workload {idx}")


def from_lengths(lengths, heads: int, head_dim: int, qk_norm: bool = False, seed: int = SEED_BASE + 7,
                 max_seqlen_meta: int | None = None, name: str = "lengths") -> Workload:
    """A workload whose images are 1 x L strips (any length, including 0)."""
    grids = tuple((1, int(L)) if L > 0 else (0, 0) for L in lengths)
    return Workload(name, grids, heads, head_dim, qk_norm, max_seqlen_meta=max_seqlen_meta, seed=seed)
