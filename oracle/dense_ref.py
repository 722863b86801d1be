"""Form A of the oracle: one dense attention over the whole packed stream.

TEST INFRASTRUCTURE ONLY (tiny inputs; builds a [T, T] mask).

This follows the vLLM Dots ``VisionAttention.forward`` (vision_attention page):
a [T, T] additive mask filled with the most negative bf16 value and set to 0
on every diagonal block [cu[i], cu[i+1]), scores q k^T times the softmax scale
(the page divides by sqrt(head_dim)), the mask added, a softmax over the key
axis, and the product with v. In fp64 the masked entries underflow to exactly
0 after exp, so this equals the per-segment form wherever every token lies in
some segment.
"""
from __future__ import annotations

import numpy as np

BF16_MIN = -3.3895313892515355e38   # most negative finite bfloat16 (torch.finfo(torch.bfloat16).min)


def dense_block_diag_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, cu_seqlens,
                               scale: float | None = None) -> np.ndarray:
    T, H, D = q.shape
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    mask = np.full((T, T), BF16_MIN, dtype=np.float64)
    cu = [int(c) for c in cu_seqlens]
    for i in range(1, len(cu)):
        mask[cu[i - 1]:cu[i], cu[i - 1]:cu[i]] = 0.0
    qh = np.transpose(q, (1, 0, 2))            # [H, T, D]
    kh = np.transpose(k, (1, 0, 2))
    vh = np.transpose(v, (1, 0, 2))
    s = np.matmul(qh, np.transpose(kh, (0, 2, 1))) * scale + mask[None]
    s = s - s.max(axis=-1, keepdims=True)
    p = np.exp(s)
    p = p / p.sum(axis=-1, keepdims=True)
    o = np.matmul(p, vh)                        # [H, T, D]
    return np.transpose(o, (1, 0, 2))
