"""GPU parity: the CUDA path, called through the C ABI, against the fp64 oracle
on the same seeded inputs (bf16 widened exactly)."""
import math

import numpy as np
import pytest
import torch

import oracle
import vision_encoder_varlen_gb300 as vit
from vision_encoder_varlen_gb300 import _build
from vision_encoder_varlen_gb300 import workloads as wl
from helpers import MAX_ABS, MEAN_ABS, assert_close, gpu_full_path, stratified_rows, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    assert vit.lib().vit_device_supported(torch.cuda.current_device()) == 0, "not an sm_103 device"


def test_native_library_is_loaded():
    vit.lib()
    maps = open("/proc/self/maps").read()
    assert vit.LIB_PATH in maps


@pytest.mark.parametrize("idx", [1, 2, 3, 4, 5])
def test_rope_freqs_exact(idx):
    w = wl.make_config(idx)
    status = vit.new_status()
    grid = torch.from_numpy(w.grid_hw.copy()).cuda()
    inv_freq, pos, cu = vit.rope_freqs(grid, w.total_tokens, w.head_dim, w.theta, status=status)
    assert vit.read_status(status) == 0
    cu_ref, pos_ref = oracle.grid_positions(w.grid_hw)
    assert np.array_equal(cu.cpu().numpy(), cu_ref)                       # bit-exact
    assert np.array_equal(pos.cpu().numpy(), pos_ref)                     # bit-exact
    # fp32 table (the page builds it in float32) against the fp64 closed form
    np.testing.assert_allclose(inv_freq.cpu().numpy(), oracle.rope_inv_freq(w.head_dim // 2, w.theta),
                               rtol=1e-6, atol=0)


def _prologue_bound(ref: np.ndarray) -> np.ndarray:
    """Per-element bound for bf16 prologue outputs.

    bf16 keeps 8 significant bits, so one rounding errs by at most u = 2^-8
    relative. The GPU rounds the normalised value, rounds again after the
    weight multiply, and rounds the fp32 rotation of each pair (a, b) once
    more. With |a| + |b| <= sqrt(2) * r (r = the pair norm, which the rotation
    preserves) the error is below (2 * sqrt(2) + 1) * u * r ~= 0.015 * r;
    fp32 angle and powf/sincosf errors add < 1e-4 * r for positions < 1000.
    Bound used: 2^-6 * r + 1e-5 (2^-6 = 0.0156).
    """
    D = ref.shape[-1]
    r = np.sqrt(ref[..., : D // 2] ** 2 + ref[..., D // 2:] ** 2)
    r = np.concatenate([r, r], axis=-1)
    return 2.0 ** -6 * r + 1e-5


@pytest.mark.parametrize("idx", [1, 2, 3, 4, 5])
def test_prologue_parity(idx):
    w = wl.make_config(idx)
    t = w.tensors()
    _, qr, kr, _, _, _ = gpu_full_path(w, t)
    torch.cuda.synchronize()
    _, pos = oracle.grid_positions(w.grid_hw)
    nw = None if t["norm_w"] is None else wl.bf16_bits(t["norm_w"])
    for name, got, wrow in (("q", qr, 0), ("k", kr, 1)):
        ref = oracle.norm_rope(wl.bf16_bits(t[name]), pos, w.theta, None if nw is None else nw[wrow],
                               w.qk_norm, w.eps)
        g = to_f64(got)
        bound = _prologue_bound(ref)
        bad = np.abs(g - ref) > bound
        assert not bad.any(), f"{name}: {bad.sum()} elements outside the bf16 bound, worst " \
                              f"{np.max(np.abs(g - ref) - bound):.3e}"


@pytest.mark.parametrize("idx", [1, 2, 3, 4])
def test_full_path_parity(idx, split):
    w = wl.make_config(idx)
    t = w.tensors()
    status = vit.new_status()
    out, *_ = gpu_full_path(w, t, status=status)
    assert vit.read_status(status) == 0
    ref = oracle.full_path(w.grid_hw, *(wl.bf16_bits(t[n]) for n in ("q", "k", "v")),
                           None if t["norm_w"] is None else wl.bf16_bits(t["norm_w"]), w.eps, w.theta)
    assert_close(out, ref, what=w.name)


def test_full_path_parity_mixed_long_short_sampled():
    """The 256x256 + 7 small images case at full size, in the benchmark's launch configuration:
    all rows of the small images, and 2048 stratified rows of the 65536-token image (the first
    and last row of both 128-row Q tiles of every 4th 256-row work item, the segment's ends,
    and a seeded random set), every head."""
    w = wl.make_config(5)
    t = w.tensors()
    status = vit.new_status()
    out, *_ = gpu_full_path(w, t, status=status)
    assert vit.read_status(status) == 0
    rows = stratified_rows(w, per_long_segment=2048, seed=5)
    assert len(rows) >= 2048
    ref = oracle.full_path(w.grid_hw, *(wl.bf16_bits(t[n]) for n in ("q", "k", "v")),
                           wl.bf16_bits(t["norm_w"]), w.eps, w.theta, rows=rows)
    assert_close(out[torch.from_numpy(rows).cuda()], ref, what=w.name)


LENGTH_CASES = [
    ([64, 60], 4, 32),
    ([1], 2, 80),
    ([0, 1, 0, 63, 64, 65, 127, 128, 129, 0], 3, 80),
    ([300, 1, 257, 511, 512, 513], 2, 128),
    ([5, 3000, 7], 2, 80),
    ([7, 9, 2100], 2, 64),
    ([200, 33, 96, 17], 4, 96),
    ([1000], 1, 32),
    # enough items that long blocks keep two Q tiles: the last block of 300, 513, 2000 and the
    # single block of 100 have at most 128 rows and run as split items, those of 400 and 640 do not
    ([300, 400, 100, 513, 640, 2000], 16, 80),
    ([300, 1, 257, 511, 512, 513, 130], 16, 128),
    ([129, 200, 700, 96, 1100], 12, 64),
    # tiny segments with an odd head count or one head: the tiny kernel's one-head items, beside
    # the two-head items the even head counts above take
    ([17, 64, 3, 40], 3, 96),
    ([33, 48, 64, 16, 1], 5, 80),
    ([5, 40, 64, 1], 1, 32),
    # two-head items at head_dim 80, whose unit code is compiled per count of 16-key groups: every
    # count (1-4) with full and ragged last groups
    ([1, 16, 17, 31, 32, 33, 47, 48, 49, 63, 64, 24, 40, 8], 4, 80),
]


# "default" passes no option (the plain entry points, the library's own split); the others pass
# their split with every call
SPLITS = {"default": None, "all_long": 0, "split_32": 32}


@pytest.fixture(params=list(SPLITS))
def split(request):
    with vit.kernel_split(SPLITS[request.param]):
        yield request.param


@pytest.mark.parametrize("lengths,H,D", LENGTH_CASES)
def test_attention_parity_lengths(lengths, H, D, split):
    w = wl.from_lengths(lengths, H, D, max_seqlen_meta=131072)
    t = w.tensors()
    cu = torch.from_numpy(w.cu_seqlens).cuda()
    q, k, v = (t[n].cuda() for n in ("q", "k", "v"))
    status = vit.new_status()
    out = vit.varlen_attn(q, k, v, cu, w.max_seqlen, status=status)
    assert vit.read_status(status) == 0
    ref = oracle.attention(*(oracle.widen(wl.bf16_bits(t[n])) for n in ("q", "k", "v")), w.cu_seqlens)
    assert_close(out, ref, what=str(lengths))


def test_tiny_four_head_items_match_the_oracle_and_two_head_items(split):
    """At head_dim 80 with a head count divisible by four, a segment bound of at most 24 tokens
    makes the tiny-segment kernel take four heads per item (two otherwise). The per-unit
    arithmetic is the same, so the two layouts agree bit for bit; both are held to the oracle."""
    lengths = [4, 16, 9, 1, 12, 24, 7, 3, 17]
    w = wl.from_lengths(lengths, 8, 80)
    t = w.tensors()
    cu = torch.from_numpy(w.cu_seqlens).cuda()
    q, k, v = (t[n].cuda() for n in ("q", "k", "v"))
    four = vit.varlen_attn(q, k, v, cu, 24)            # bound 24: four heads per item
    two = vit.varlen_attn(q, k, v, cu, 131072)          # loose bound: two heads per item
    assert torch.equal(four, two)
    ref = oracle.attention(*(oracle.widen(wl.bf16_bits(t[n])) for n in ("q", "k", "v")), w.cu_seqlens)
    assert_close(four, ref, what="four-head items")


def test_attention_parity_explicit_scale(split):
    w = wl.from_lengths([130, 70], 2, 80)
    t = w.tensors()
    q, k, v = (t[n].cuda() for n in ("q", "k", "v"))
    out = vit.varlen_attn(q, k, v, torch.from_numpy(w.cu_seqlens).cuda(), w.max_seqlen, scale=0.05)
    ref = oracle.attention(*(oracle.widen(wl.bf16_bits(t[n])) for n in ("q", "k", "v")), w.cu_seqlens, scale=0.05)
    assert_close(out, ref, what="scale=0.05")
