"""Seeded random cases through the whole path against the fp64 oracle, and the
size limits: the maximum segment count, and more heads than one row per
thread of the prologue allows."""
import numpy as np
import pytest
import torch

import oracle
import vision_encoder_varlen_gb300 as vit
from vision_encoder_varlen_gb300 import _build
from vision_encoder_varlen_gb300 import workloads as wl
from helpers import assert_close, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()


def _random_grids(rng, n):
    """image grids whose token counts mix empty, tiny, short and long segments"""
    grids = []
    for _ in range(n):
        kind = rng.integers(0, 10)
        if kind == 0:
            grids.append((0, int(rng.integers(1, 5))))           # an empty image
        elif kind < 5:
            grids.append((int(rng.integers(1, 9)), int(rng.integers(1, 9))))   # <= 64 tokens
        elif kind < 8:
            grids.append((int(rng.integers(8, 20)), int(rng.integers(8, 20))))
        else:
            grids.append((int(rng.integers(20, 50)), int(rng.integers(20, 60))))
    return tuple(grids)


@pytest.mark.parametrize("seed", range(12))
def test_fuzz_full_path(seed):
    rng = np.random.default_rng(1000 + seed)
    D = int(rng.choice([32, 64, 80, 96, 128]))
    H = int(rng.integers(1, 6))
    norm = bool(rng.integers(0, 2))
    interleaved = bool(rng.integers(0, 2))
    grids = _random_grids(rng, int(rng.integers(1, 14)))
    if sum(h * w for h, w in grids) == 0:
        grids = grids + ((3, 5),)
    w = wl.Workload(f"fuzz{seed}", grids, H, D, norm, seed=5000 + seed)
    t = w.tensors()
    T = w.total_tokens
    grid = torch.from_numpy(w.grid_hw.copy()).cuda()
    status = vit.new_status()
    inv_freq, pos, cu = vit.rope_freqs(grid, T, D, w.theta, status=status)
    nw = t["norm_w"].cuda() if norm else None
    qr, kr = vit.qk_norm_rope(t["q"].cuda(), t["k"].cuda(), pos, inv_freq, nw, w.eps, interleaved=interleaved)
    out, lse = vit.varlen_attn(qr, kr, t["v"].cuda(), cu, w.max_seqlen, status=status, return_lse=True)
    assert vit.read_status(status) == 0
    ref, ref_lse = oracle.full_path(w.grid_hw, *(wl.bf16_bits(t[n]) for n in ("q", "k", "v")),
                                    wl.bf16_bits(t["norm_w"]) if norm else None, w.eps, w.theta,
                                    interleaved=interleaved, return_lse=True)
    assert_close(out, ref, what=f"fuzz {seed}: D={D} H={H} norm={norm} il={interleaved} grids={grids}")
    err = np.abs(lse.cpu().numpy().astype(np.float64) - ref_lse)
    assert err.max() <= 2e-2 and err.mean() <= 2e-3


def test_maximum_segment_count():
    B = vit.MAX_SEGMENTS
    rng = np.random.default_rng(7)
    lengths = rng.integers(0, 4, size=B)
    lengths[0] = 70                                          # one segment for the tcgen05 kernel
    w = wl.from_lengths(lengths, 2, 32, max_seqlen_meta=128)
    t = w.tensors()
    status = vit.new_status()
    out = vit.varlen_attn(*(t[n].cuda() for n in ("q", "k", "v")), torch.from_numpy(w.cu_seqlens).cuda(),
                          w.max_seqlen, status=status)
    assert vit.read_status(status) == 0
    ref = oracle.attention(*(oracle.widen(wl.bf16_bits(t[n])) for n in ("q", "k", "v")), w.cu_seqlens)
    assert_close(out, ref, what="8192 segments")
    # one segment more is refused on the host
    with pytest.raises(vit.VitError):
        cu = torch.zeros(B + 2, dtype=torch.int32, device="cuda")
        vit.varlen_attn(t["q"].cuda(), t["k"].cuda(), t["v"].cuda(), cu, 4)


@pytest.mark.parametrize("interleaved", [False, True])
def test_prologue_with_more_than_128_heads(interleaved):
    # 2 * 130 rows per token do not fit one row per thread of a 256-thread block: the 8-lane
    # group layout runs instead, with the same arithmetic
    H, D = 130, 64
    w = wl.from_lengths([150, 90], H, D, qk_norm=True, seed=77)
    t = w.tensors()
    T = w.total_tokens
    grid = torch.tensor([[10, 15], [9, 10]], dtype=torch.int32).cuda()
    inv_freq, pos, cu = vit.rope_freqs(grid, T, D, w.theta)
    qr, kr = vit.qk_norm_rope(t["q"].cuda(), t["k"].cuda(), pos, inv_freq, t["norm_w"].cuda(), w.eps,
                              interleaved=interleaved)
    _, pos_ref = oracle.grid_positions(np.array([[10, 15], [9, 10]]))
    nwb = wl.bf16_bits(t["norm_w"])
    for name, got, row in (("q", qr, 0), ("k", kr, 1)):
        ref = oracle.norm_rope(wl.bf16_bits(t[name]), pos_ref, w.theta, nwb[row], True, w.eps, interleaved)
        if interleaved:
            r = np.repeat(np.sqrt(ref[..., 0::2] ** 2 + ref[..., 1::2] ** 2), 2, axis=-1)
        else:
            r = np.sqrt(ref[..., : D // 2] ** 2 + ref[..., D // 2:] ** 2)
            r = np.concatenate([r, r], axis=-1)
        assert np.all(np.abs(to_f64(got) - ref) <= 2.0 ** -6 * r + 1e-5), name
    # k alone is 130 rows per token, which does fit one row per thread: the other layout, and the
    # same bits
    _, k_only = vit.qk_norm_rope(None, t["k"].cuda(), pos, inv_freq, t["norm_w"].cuda(), w.eps,
                                 interleaved=interleaved)
    assert torch.equal(k_only, kr)
