"""Rounding mimic of the pages' eager modules (test infrastructure, debug only).

TEST INFRASTRUCTURE ONLY, and never a pass/fail criterion for the CUDA path: the
exact fp64 oracle (``vit_oracle.c``) is what parity is measured against. This
module evaluates the same steps with the roundings that the eager PyTorch modules
of the vLLM Dots ``vision_attention`` page make, so that a residual between the
CUDA path and the exact oracle can be put beside the residual the pages' own
eager path carries. Every fp32 or bf16 operation is modelled as its exact result
rounded once (round to nearest, ties to even) to the operation's type:

* ``VisionRotaryEmbedding`` (``__init__``, ``_compute_freqs``): the exponent
  2j/dim, the power theta^e and the reciprocal each rounded to fp32; the angle
  pos * inv_freq rounded to fp32 (``torch.outer`` in fp32); cos and sin rounded
  to fp32.
* ``_RMSNorm.forward`` / ``_norm``: x widened to fp32, the sum of squares and
  the mean each rounded to fp32, mean + eps (eps as an fp32 scalar) rounded,
  the reciprocal square root rounded, x times it rounded to fp32, cast back to
  bf16 (``type_as``), then the product with the bf16 weight rounded to bf16.
* The rotary application, which the pages call but do not print: applied in
  fp32 and cast once (the reading the CUDA path also takes) -- both products
  rounded to fp32, their sum or difference rounded to fp32, then to bf16.
* ``VisionAttention.forward`` (dense block-diagonal mask) and
  ``VisionAttentionV2.forward`` (one segment at a time), which give the same
  values here because a masked score plus the most negative bf16 stays that
  value and its fp32 exponential is exactly 0: q k^T as a bf16 matmul (the
  exact dot product rounded to bf16), divided by sqrt(head_dim) in fp32 and
  rounded to bf16, a softmax in fp32 (x - max, exp, the row sum and the
  quotient each rounded to fp32), the weights cast to bf16, then the bf16
  matmul with v (the exact sum rounded to bf16).

A model, not a bit-for-bit copy of any one run of those modules: PyTorch does
not fix the order of its fp32 reductions, nor how its kernels evaluate exp,
pow and rsqrt, and such differences move a bf16 result by one unit in rare
near-ties. The pins in ``tests/test_oracle_mimic.py`` hold this module to
PyTorch's own CPU operations within exactly that.
"""
from __future__ import annotations

import numpy as np

from . import grid_positions, widen

_BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127    # largest finite bfloat16
_BF16_MIN_NORMAL = 2.0 ** -126


def f32(x) -> np.ndarray:
    """Round fp64 values to fp32 (IEEE round to nearest even), returned as fp64."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def bf16_round(x) -> np.ndarray:
    """Round fp64 values to bfloat16 (8 significant bits, fp32's exponent range,
    round to nearest, ties to even), returned as fp64; NaN and infinities pass
    through, magnitudes past the largest finite bf16 (by at least half a unit)
    become infinite, and bf16 subnormals (multiples of 2^-133) are kept.

    Rounds the fp64 value directly, so there is no intermediate fp32 rounding."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    bits = x.view(np.uint64)
    # keep the top 7 of fp64's 52 fraction bits: add just under half of the dropped
    # range plus the lowest kept bit (ties to even), then clear the dropped bits
    keep_lsb = (bits >> np.uint64(45)) & np.uint64(1)
    rounded = (bits + np.uint64((1 << 44) - 1) + keep_lsb) & ~np.uint64((1 << 45) - 1)
    out = rounded.view(np.float64).copy()
    out = np.where(np.abs(out) > _BF16_MAX, np.copysign(np.inf, x), out)
    tiny = np.abs(x) < _BF16_MIN_NORMAL
    if np.any(tiny):
        out[tiny] = np.rint(x[tiny] * 2.0 ** 133) * 2.0 ** -133   # fixed spacing below the normals
    return np.where(np.isfinite(x), out, x)


def to_bits(x) -> np.ndarray:
    """uint16 bit patterns of values that already lie on the bf16 grid."""
    return (np.asarray(x, dtype=np.float64).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def inv_freq_fp32(dim: int, theta: float = 10000.0) -> np.ndarray:
    """VisionRotaryEmbedding's inv_freq [dim/2] as fp32 arithmetic produces it (fp64 values)."""
    e = f32(np.arange(0, dim, 2, dtype=np.float64) / dim)
    return f32(1.0 / f32(np.power(f32(theta), e)))


def _angles(pos: np.ndarray, D: int, theta: float):
    """fp32 cos and sin [T, D/2]: row angles on the first D/4 pairs, column angles on the rest."""
    inv = inv_freq_fp32(D // 2, theta)                        # D/4 entries
    pos = np.asarray(pos, dtype=np.int64).reshape(-1, 2).astype(np.float64)
    a = np.concatenate([f32(np.outer(pos[:, 0], inv)), f32(np.outer(pos[:, 1], inv))], axis=1)
    return f32(np.cos(a)), f32(np.sin(a))


def _rms_norm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """_RMSNorm on bf16 values x [..., D] (fp64 holding bf16) with bf16 weight w [D]."""
    D = x.shape[-1]
    ss = f32(np.sum(x * x, axis=-1, keepdims=True))           # squares of bf16 values are exact
    mean = f32(ss / D)
    r = f32(1.0 / np.sqrt(f32(mean + f32(eps))))
    y = bf16_round(f32(x * r))                                # cast back to the input dtype
    return bf16_round(y * w)                                  # bf16 x bf16 is exact before rounding


def norm_rope(x_bits: np.ndarray, pos: np.ndarray, theta: float = 10000.0, w_bits: np.ndarray | None = None,
              use_norm: bool = False, eps: float = 1e-6, interleaved: bool = False) -> np.ndarray:
    """Optional RMSNorm then 2D RoPE of bf16 rows x [T, H, D] with the eager modules'
    roundings; returns the bf16 bit patterns [T, H, D] (uint16)."""
    x = widen(np.asarray(x_bits, dtype=np.uint16))
    T, H, D = x.shape
    if use_norm:
        x = _rms_norm(x, widen(np.asarray(w_bits, dtype=np.uint16).reshape(D)), eps)
    c, s = _angles(pos, D, theta)                             # [T, D/2]
    c = c[:, None, :]
    s = s[:, None, :]
    y = np.empty_like(x)
    if not interleaved:
        a, b = x[..., : D // 2], x[..., D // 2:]              # pair m = (a[m], b[m])
        y[..., : D // 2] = f32(f32(a * c) - f32(b * s))
        y[..., D // 2:] = f32(f32(b * c) + f32(a * s))
    else:
        a, b = x[..., 0::2], x[..., 1::2]                     # pair m = (x[2m], x[2m+1])
        y[..., 0::2] = f32(f32(a * c) - f32(b * s))
        y[..., 1::2] = f32(f32(b * c) + f32(a * s))
    return to_bits(bf16_round(y))


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, cu_seqlens, rows=None) -> np.ndarray:
    """The eager attention of bf16 q, k, v [T, H, D] (fp64 holding bf16 values) per
    segment, scale 1/sqrt(head_dim); returns fp64 values on the bf16 grid, [T, H, D]
    or [len(rows), H, D] for the given query rows."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    T, H, D = q.shape
    cu = [int(c) for c in np.asarray(cu_seqlens).reshape(-1)]
    sqrt_d = f32(np.sqrt(D))
    want = np.arange(T) if rows is None else np.asarray(rows, dtype=np.int64).reshape(-1)
    out = np.full((want.shape[0], H, D), np.nan)
    for i in range(len(cu) - 1):
        lo, hi = cu[i], cu[i + 1]
        sel = np.nonzero((want >= lo) & (want < hi))[0]
        if sel.size == 0:
            continue
        chunk = max(1, (1 << 22) // (hi - lo))                # rows per block of scores (bounds memory)
        for h in range(H):
            kh, vh = k[lo:hi, h], v[lo:hi, h]                 # [L, D]
            for c0 in range(0, sel.size, chunk):
                rs = sel[c0:c0 + chunk]
                s = bf16_round(q[want[rs], h] @ kh.T)         # [n, L]
                s = bf16_round(f32(s / sqrt_d))
                e = f32(np.exp(f32(s - s.max(axis=-1, keepdims=True))))
                p = bf16_round(f32(e / f32(e.sum(axis=-1, keepdims=True))))
                out[rs, h] = bf16_round(p @ vh)
    return out


def full_path(grid_hw, q_bits, k_bits, v_bits, norm_w_bits=None, eps: float = 1e-6, theta: float = 10000.0,
              rows=None, interleaved: bool = False) -> np.ndarray:
    """Positions from the grid, the eager prologue, then the eager attention."""
    cu, pos = grid_positions(grid_hw)
    use_norm = norm_w_bits is not None
    wq = None if norm_w_bits is None else np.asarray(norm_w_bits)[0]
    wk = None if norm_w_bits is None else np.asarray(norm_w_bits)[1]
    qr = widen(norm_rope(q_bits, pos, theta, wq, use_norm, eps, interleaved))
    kr = widen(norm_rope(k_bits, pos, theta, wk, use_norm, eps, interleaved))
    return attention(qr, kr, widen(v_bits), cu, rows)
