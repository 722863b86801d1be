"""GPU parity of the extended calls: the per-row log-sum-exp output of the
attention, the interleaved-pair ("complex_rope") rotary mode of the prologue,
and prologue calls that leave q or k out. CUDA path through the C ABI against
the fp64 oracle, on the seeded workloads."""
import math

import numpy as np
import pytest
import torch

import oracle
import vision_encoder_varlen_gb300 as vit
from vision_encoder_varlen_gb300 import _build
from vision_encoder_varlen_gb300 import workloads as wl
from helpers import assert_close, sample_rows, to_f64

pytestmark = pytest.mark.gpu

# lse tolerance (absolute, natural log). The fp32 score of a row errs by < 1e-4 (D <= 128 exact
# bf16 products summed in fp32, |q||k| scale <= ~12); each exp2 term errs by < 2e-6 relative
# (ex2.approx plus the fp32 rounding of its argument, |arg| < 40) and the fp32 row sum of up to
# 65536 terms adds < 4e-5 relative, so ln(l) moves by < 5e-5. 1e-3 leaves a 5x margin.
LSE_ABS = 1e-3
# Through the whole path the prologue hands attention bf16 q' and k' (the pages cast back to the
# input dtype) while the oracle keeps them in fp64: each element then differs by up to 2^-9
# relative, which moves every score by ~1e-3 (random signs over D terms) and the worst of ~10^5
# rows by several times that. There lse is held to the path's output tolerance instead.
PATH_MAX_ABS, PATH_MEAN_ABS = 2e-2, 2e-3

# "default" passes no option (the plain entry points, the library's own split); the others pass
# their split with every call
SPLITS = {"default": None, "all_long": 0, "split_32": 32}


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    assert vit.lib().vit_device_supported(torch.cuda.current_device()) == 0, "not an sm_103 device"


@pytest.fixture(params=list(SPLITS))
def split(request):
    with vit.kernel_split(SPLITS[request.param]):
        yield request.param


def _widen(t, names=("q", "k", "v")):
    return [oracle.widen(wl.bf16_bits(t[n])) for n in names]


def _assert_lse(got: torch.Tensor, ref: np.ndarray, what: str, max_abs=LSE_ABS, mean_abs=None):
    g = got.detach().cpu().numpy().astype(np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite lse"
    err = np.abs(g - ref)
    mx = float(err.max()) if g.size else 0.0
    assert mx <= max_abs, f"{what}: lse max-abs {mx:.3e} > {max_abs:.0e}"
    if mean_abs is not None and g.size:
        assert float(err.mean()) <= mean_abs, f"{what}: lse mean-abs {err.mean():.3e} > {mean_abs:.0e}"


LSE_CASES = [
    ([64, 60], 4, 32),
    ([1, 2, 3], 2, 80),
    ([0, 1, 0, 63, 64, 65, 127, 128, 129, 0], 3, 80),
    ([300, 1, 257, 511, 512, 513], 2, 128),
    ([5, 3000, 7], 2, 80),
    ([200, 33, 96, 17], 4, 96),
    ([7, 9, 2100], 2, 64),
    # two-head tiny items at head_dim 80 over every count of 16-key groups (the tiny kernel's unit
    # code is compiled per count there)
    ([1, 16, 17, 31, 33, 48, 49, 64, 24, 40], 4, 80),
]


@pytest.mark.parametrize("lengths,H,D", LSE_CASES)
def test_lse_parity_lengths(lengths, H, D, split):
    w = wl.from_lengths(lengths, H, D, max_seqlen_meta=131072)
    t = w.tensors()
    q, k, v = (t[n].cuda() for n in ("q", "k", "v"))
    status = vit.new_status()
    out, lse = vit.varlen_attn(q, k, v, torch.from_numpy(w.cu_seqlens).cuda(), w.max_seqlen, status=status,
                               return_lse=True)
    assert vit.read_status(status) == 0
    ref, ref_lse = oracle.attention(*_widen(t), w.cu_seqlens, return_lse=True)
    assert_close(out, ref, what=str(lengths))
    _assert_lse(lse, ref_lse, str(lengths))
    # the plain call writes the same output bits
    out2 = vit.varlen_attn(q, k, v, torch.from_numpy(w.cu_seqlens).cuda(), w.max_seqlen)
    assert torch.equal(out, out2)


def test_lse_four_head_tiny_items(split):
    """A segment bound of at most 24 tokens at head_dim 80 (head count divisible by four) makes
    the tiny-segment kernel take four heads per item: its lse rows match the oracle and, bit for
    bit, those of the two-head items a loose bound gives."""
    w = wl.from_lengths([4, 16, 9, 1, 12, 24, 7, 3, 17], 8, 80)
    t = w.tensors()
    q, k, v = (t[n].cuda() for n in ("q", "k", "v"))
    cu = torch.from_numpy(w.cu_seqlens).cuda()
    out4, lse4 = vit.varlen_attn(q, k, v, cu, 24, return_lse=True)
    out2, lse2 = vit.varlen_attn(q, k, v, cu, 131072, return_lse=True)
    assert torch.equal(out4, out2) and torch.equal(lse4, lse2)
    ref, ref_lse = oracle.attention(*_widen(t), w.cu_seqlens, return_lse=True)
    assert_close(out4, ref, what="four-head items")
    _assert_lse(lse4, ref_lse, "four-head items")


def test_lse_explicit_scale_and_zero_q(split):
    w = wl.from_lengths([130, 70, 1], 2, 80)
    t = w.tensors()
    q, k, v = (t[n].cuda() for n in ("q", "k", "v"))
    cu = torch.from_numpy(w.cu_seqlens).cuda()
    _, lse = vit.varlen_attn(q, k, v, cu, w.max_seqlen, scale=0.05, return_lse=True)
    _, ref_lse = oracle.attention(*_widen(t), w.cu_seqlens, scale=0.05, return_lse=True)
    _assert_lse(lse, ref_lse, "scale=0.05")
    # q = 0: every score is 0 and lse = ln L exactly in the mathematics
    _, lse0 = vit.varlen_attn(torch.zeros_like(q), k, v, cu, w.max_seqlen, return_lse=True)
    L = np.repeat(np.diff(w.cu_seqlens), 1)
    expect = np.repeat(np.log(L.astype(np.float64)), L)[:, None].repeat(2, axis=1)
    _assert_lse(lse0, expect, "q=0")


@pytest.mark.parametrize("idx", [3, 4])
def test_lse_full_path(idx):
    w = wl.make_config(idx)
    t = w.tensors()
    grid = torch.from_numpy(w.grid_hw.copy()).cuda()
    inv_freq, pos, cu = vit.rope_freqs(grid, w.total_tokens, w.head_dim, w.theta)
    qr, kr = vit.qk_norm_rope(t["q"].cuda(), t["k"].cuda(), pos, inv_freq, t["norm_w"].cuda(), w.eps)
    out, lse = vit.varlen_attn(qr, kr, t["v"].cuda(), cu, w.max_seqlen, return_lse=True)
    ref, ref_lse = oracle.full_path(w.grid_hw, *(wl.bf16_bits(t[n]) for n in ("q", "k", "v")),
                                    wl.bf16_bits(t["norm_w"]), w.eps, w.theta, return_lse=True)
    assert_close(out, ref, what=w.name)
    _assert_lse(lse, ref_lse, w.name, PATH_MAX_ABS, PATH_MEAN_ABS)


def test_lse_mixed_long_short_sampled():
    w = wl.make_config(5)
    t = w.tensors()
    grid = torch.from_numpy(w.grid_hw.copy()).cuda()
    inv_freq, pos, cu = vit.rope_freqs(grid, w.total_tokens, w.head_dim, w.theta)
    qr, kr = vit.qk_norm_rope(t["q"].cuda(), t["k"].cuda(), pos, inv_freq, t["norm_w"].cuda(), w.eps)
    out, lse = vit.varlen_attn(qr, kr, t["v"].cuda(), cu, w.max_seqlen, return_lse=True)
    rows = sample_rows(w, big_rows=128, seed=11)
    ref, ref_lse = oracle.full_path(w.grid_hw, *(wl.bf16_bits(t[n]) for n in ("q", "k", "v")),
                                    wl.bf16_bits(t["norm_w"]), w.eps, w.theta, rows=rows, return_lse=True)
    idx = torch.from_numpy(rows).cuda()
    assert_close(out[idx], ref, what=w.name)
    _assert_lse(lse[idx], ref_lse, w.name, PATH_MAX_ABS, PATH_MEAN_ABS)


def _bound_interleaved(ref: np.ndarray) -> np.ndarray:
    """bf16 bound of the prologue output (two roundings in the norm, one after the rotation of each
    pair, each <= 2^-8 relative; see the rotate-half test) with r the norm of the adjacent pair."""
    r = np.sqrt(ref[..., 0::2] ** 2 + ref[..., 1::2] ** 2)
    return 2.0 ** -6 * np.repeat(r, 2, axis=-1) + 1e-5


@pytest.mark.parametrize("idx", [1, 2, 3, 4, 5])
def test_interleaved_prologue_parity(idx):
    w = wl.make_config(idx)
    t = w.tensors()
    grid = torch.from_numpy(w.grid_hw.copy()).cuda()
    inv_freq, pos, _ = vit.rope_freqs(grid, w.total_tokens, w.head_dim, w.theta)
    nw = t["norm_w"].cuda() if t["norm_w"] is not None else None
    qr, kr = vit.qk_norm_rope(t["q"].cuda(), t["k"].cuda(), pos, inv_freq, nw, w.eps, interleaved=True)
    _, pos_ref = oracle.grid_positions(w.grid_hw)
    nwb = None if t["norm_w"] is None else wl.bf16_bits(t["norm_w"])
    for name, got, wrow in (("q", qr, 0), ("k", kr, 1)):
        ref = oracle.norm_rope(wl.bf16_bits(t[name]), pos_ref, w.theta, None if nwb is None else nwb[wrow],
                               w.qk_norm, w.eps, interleaved=True)
        g = to_f64(got)
        bound = _bound_interleaved(ref)
        bad = np.abs(g - ref) > bound
        assert not bad.any(), f"{name}: {bad.sum()} elements outside the bf16 bound, worst " \
                              f"{np.max(np.abs(g - ref) - bound):.3e}"


@pytest.mark.parametrize("idx", [3, 4])
def test_interleaved_full_path_parity(idx):
    w = wl.make_config(idx)
    t = w.tensors()
    grid = torch.from_numpy(w.grid_hw.copy()).cuda()
    inv_freq, pos, cu = vit.rope_freqs(grid, w.total_tokens, w.head_dim, w.theta)
    qr, kr = vit.qk_norm_rope(t["q"].cuda(), t["k"].cuda(), pos, inv_freq, t["norm_w"].cuda(), w.eps,
                              interleaved=True)
    out = vit.varlen_attn(qr, kr, t["v"].cuda(), cu, w.max_seqlen)
    ref = oracle.full_path(w.grid_hw, *(wl.bf16_bits(t[n]) for n in ("q", "k", "v")), wl.bf16_bits(t["norm_w"]),
                           w.eps, w.theta, interleaved=True)
    assert_close(out, ref, what=w.name + " interleaved")


@pytest.mark.parametrize("interleaved", [False, True])
@pytest.mark.parametrize("D", [32, 64, 80, 96, 128])
def test_prologue_one_half_matches_both_bitwise(D, interleaved):
    T, H = 777, 3
    w = wl.from_lengths([T], H, D, qk_norm=True)
    t = w.tensors()
    pos = torch.randint(0, 300, (T, 2), dtype=torch.int32, generator=torch.Generator().manual_seed(D)).cuda()
    inv_freq = torch.from_numpy(oracle.rope_inv_freq(D // 2)).float().cuda()
    q, k, nw = t["q"].cuda(), t["k"].cuda(), t["norm_w"].cuda()
    qb, kb = vit.qk_norm_rope(q, k, pos, inv_freq, nw, 1e-6, interleaved=interleaved)
    qo, none_k = vit.qk_norm_rope(q, None, pos, inv_freq, nw, 1e-6, interleaved=interleaved)
    none_q, ko = vit.qk_norm_rope(None, k, pos, inv_freq, nw, 1e-6, interleaved=interleaved)
    assert none_k is None and none_q is None
    assert torch.equal(qo, qb) and torch.equal(ko, kb)


def test_interleaved_equals_rotate_half_under_permutation():
    # one mode is the other on permuted heads (element 2m -> m, 2m+1 -> m + D/2) up to the
    # order of fp32 operations inside the rotation: compare within one bf16 rounding
    T, H, D = 300, 2, 80
    w = wl.from_lengths([T], H, D, qk_norm=True)
    t = w.tensors()
    perm = torch.cat([torch.arange(0, D, 2), torch.arange(1, D, 2)])
    pos = torch.randint(0, 100, (T, 2), dtype=torch.int32, generator=torch.Generator().manual_seed(1)).cuda()
    inv_freq = torch.from_numpy(oracle.rope_inv_freq(D // 2)).float().cuda()
    q, nw = t["q"].cuda(), t["norm_w"].cuda()
    qi, _ = vit.qk_norm_rope(q, None, pos, inv_freq, nw, 1e-6, interleaved=True)
    qh, _ = vit.qk_norm_rope(q[..., perm].contiguous(), None, pos, inv_freq, nw[:, perm].contiguous(), 1e-6)
    a, b = qi[..., perm].float(), qh.float()
    # the fp32 sums of squares add in different orders, so a normalised value may round one bf16
    # ulp apart before the rotation mixes the pair: bound by the pair norm, as the parity tests do
    r = torch.sqrt(b[..., : D // 2] ** 2 + b[..., D // 2:] ** 2).repeat(1, 1, 2)
    assert torch.all((a - b).abs() <= 2.0 ** -6 * r + 1e-5)
