"""Pins of the rounding mimic (oracle/mimic.py) against things other than itself (CPU only).

The mimic evaluates the vLLM Dots vision_attention page's eager steps with each fp32 or
bf16 operation rounded once. Its rounding primitive is pinned by PyTorch's own fp32 -> bf16
cast and by a brute-force search over rationals; each step is pinned by the same step
written with PyTorch's CPU tensor operations in fp32 and bf16 (which may differ from an
exactly-rounded step by one bf16 unit in rare near-ties, so those pins allow exactly that);
and the whole prologue is checked against the exact fp64 oracle within the bound the GPU
parity tests derive for these roundings, which pins that derivation as well.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import mimic
from vision_encoder_varlen_gb300 import workloads as wl

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


def _ulp_dist(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    """Distance in bf16 units between finite bf16 bit patterns (sign-magnitude -> ordered ints)."""
    def ordered(b):
        b = b.astype(np.int32)
        return np.where(b & 0x8000, -(b & 0x7FFF), b)
    return np.abs(ordered(a_bits) - ordered(b_bits))


def _fp32_ulp_dist(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    ai = np.asarray(a, dtype=np.float32).view(np.int32).astype(np.int64)
    bi = np.asarray(b, dtype=np.float32).view(np.int32).astype(np.int64)
    return np.abs(ai - bi)


# ---------------------------------------------------------------- the rounding primitive

def test_bf16_round_equals_torch_cast_on_fp32_values():
    rng = np.random.default_rng(5)
    n = 200_000
    x = rng.standard_normal(n) * np.exp2(rng.integers(-140, 128, n).astype(np.float64))
    with np.errstate(over="ignore"):
        x = x.astype(np.float32)
    # exact ties between bf16 neighbours (both parities), the overflow threshold, the
    # smallest normal, fp32 subnormals, signed zeros and the non-finite values
    one = np.float32(1.0)
    edges = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), 1 + 2.0 ** -8 + 2.0 ** -23,
                      (2 - 2.0 ** -7) * 2.0 ** 127, (2 - 2.0 ** -8) * 2.0 ** 127, (2 - 2.0 ** -9) * 2.0 ** 127,
                      2.0 ** -126, 2.0 ** -126 * (1 - 2.0 ** -9), 2.0 ** -133, 1.5 * 2.0 ** -133,
                      2.5 * 2.0 ** -133, 2.0 ** -149, 0.0, -0.0, np.inf, -np.inf, np.nan], dtype=np.float64)
    x = np.concatenate([x, edges.astype(np.float32) * one])
    got = mimic.bf16_round(x.astype(np.float64))
    ref = torch.from_numpy(x).to(torch.bfloat16).float().numpy().astype(np.float64)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))      # -0 stays -0


def _brute_bf16(x: float) -> float:
    """Nearest bf16 to x by comparing exact rational distances to neighbouring bit patterns."""
    if x == 0.0:
        return x
    sign = -1.0 if x < 0 else 1.0
    ax = abs(x)
    top = int(np.array([ax], dtype=np.float32).view(np.uint32)[0]) >> 16
    best, best_d, best_p = None, None, None
    for p in (top - 1, top, top + 1):
        if p < 0 or p > 0x7F7F:
            continue
        val = float(np.array([p << 16], dtype=np.uint32).view(np.float32)[0])
        d = abs(Fraction(ax) - Fraction(val))
        if best is None or d < best_d or (d == best_d and p % 2 == 0):
            best, best_d, best_p = val, d, p
    return sign * best


def test_bf16_round_brute_force_on_fp64_values():
    rng = np.random.default_rng(6)
    vals = list(rng.standard_normal(1500) * np.exp2(rng.integers(-120, 120, 1500).astype(np.float64)))
    # exact midpoints and points just off them, which a rounding through fp32 first would get wrong
    for m in (1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 96.0 + 2.0 ** -2, 2.0 ** -100 * (1 + 2.0 ** -8)):
        ulp = 2.0 ** (math.frexp(m)[1] - 9)
        vals += [m, -m, m + ulp * 2.0 ** -30, m - ulp * 2.0 ** -30, m + ulp * 2.0 ** -20]
    vals += [2.0 ** -130 * 1.3, 2.0 ** -127 * 1.999]                  # bf16 subnormal range
    got = mimic.bf16_round(np.array(vals))
    for x, g in zip(vals, got):
        assert g == _brute_bf16(x), x
    # the off-midpoint case: direct rounding goes up, rounding through fp32 first ties to even (down)
    m = 1.0 + 2.0 ** -8
    x = m + 2.0 ** -9 * 2.0 ** -30
    assert mimic.bf16_round(np.array([x]))[0] == 1.0 + 2.0 ** -7
    assert mimic.bf16_round(mimic.f32(np.array([x])))[0] == 1.0


# ---------------------------------------------------------------- the table and the prologue steps

def _torch_inv_freq(dim: int, theta: float) -> torch.Tensor:
    e = (2 * torch.arange(dim // 2, dtype=torch.float32)) / dim
    return torch.reciprocal(torch.pow(torch.tensor(theta, dtype=torch.float32), e))


@pytest.mark.parametrize("dim", [8, 16, 20, 32, 40, 64])
def test_inv_freq_fp32_against_torch_and_closed_form(dim):
    got = mimic.inv_freq_fp32(dim, 10000.0)
    ref = _torch_inv_freq(dim, 10000.0).numpy()
    assert np.max(_fp32_ulp_dist(got, ref)) <= 1
    assert got[0] == 1.0
    # against the fp64 closed form: the power and the reciprocal each add 2^-24 relative, and
    # the exponent e = 2j/dim, rounded to fp32, moves theta^e by ln(theta) * e * 2^-24 relative
    exact = oracle.rope_inv_freq(dim, 10000.0)
    e = np.arange(0, dim, 2) / dim
    bound = (2.0 + e * math.log(10000.0)) * 2.0 ** -24 * 1.001
    assert np.all(np.abs(got / exact - 1.0) <= bound)


def _rand_rows(T, H, D, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((T, H, D), generator=g).to(torch.bfloat16)
    w = (1.0 + 0.1 * torch.randn((D,), generator=g)).to(torch.bfloat16)
    return x, w


# (input scale, eps): eps negligible, eps comparable to mean(x^2) (tiny inputs), eps dominant
@pytest.mark.parametrize("scale,eps", [(1.0, 1e-6), (2.0 ** -10, 1e-6), (1.0, 0.25)])
@pytest.mark.parametrize("D", [32, 80, 128])
def test_norm_step_against_torch_ops(D, scale, eps):
    x, w = _rand_rows(96, 4, D, seed=11 + D)
    x = (x.float() * scale).to(torch.bfloat16)             # a power of two: exact
    pos = np.zeros((96, 2), dtype=np.int32)                # angle 0: the rotation is the identity
    got = mimic.norm_rope(wl.bf16_bits(x), pos, 10000.0, wl.bf16_bits(w), True, eps)
    xf = x.float()
    r = torch.rsqrt(xf.square().mean(dim=-1, keepdim=True) + eps)
    ref = wl.bf16_bits((xf * r).to(torch.bfloat16) * w)
    d = _ulp_dist(got, ref)
    assert d.max() <= 1
    assert np.mean(d == 0) >= 0.99


def _torch_rope(x: torch.Tensor, pos: np.ndarray, theta: float, interleaved: bool) -> torch.Tensor:
    D = x.shape[-1]
    inv = _torch_inv_freq(D // 2, theta)
    p = torch.from_numpy(pos.astype(np.float32))
    ang = torch.cat([p[:, :1] * inv[None, :], p[:, 1:] * inv[None, :]], dim=1)[:, None, :]   # [T, 1, D/2]
    c, s = torch.cos(ang), torch.sin(ang)
    xf = x.float()
    if interleaved:
        a, b = xf[..., 0::2], xf[..., 1::2]
        y = torch.stack([a * c - b * s, b * c + a * s], dim=-1).flatten(-2)
    else:
        a, b = xf[..., : D // 2], xf[..., D // 2:]
        y = torch.cat([a * c - b * s, b * c + a * s], dim=-1)
    return y.to(torch.bfloat16)


@pytest.mark.parametrize("D", [32, 80, 128])
def test_angle_table_against_torch_fp32(D):
    # fp32 cos/sin of fp32 angles (row angles on the first D/4 pairs, column angles after)
    rng = np.random.default_rng(100 + D)
    pos = rng.integers(0, 1024, size=(500, 2)).astype(np.int32)
    c, s = mimic._angles(pos, D, 10000.0)
    inv = _torch_inv_freq(D // 2, 10000.0)
    p = torch.from_numpy(pos.astype(np.float32))
    ang = torch.cat([p[:, :1] * inv[None, :], p[:, 1:] * inv[None, :]], dim=1)
    a_got = np.concatenate([mimic.f32(np.outer(pos[:, 0], mimic.inv_freq_fp32(D // 2))),
                            mimic.f32(np.outer(pos[:, 1], mimic.inv_freq_fp32(D // 2)))], axis=1)
    assert np.array_equal(a_got, ang.double().numpy())     # the fp32 angles agree exactly
    # PyTorch's fp32 cos/sin are faithful (within one unit) rather than correctly rounded:
    # about 5 % of these differ from the correctly rounded value by one unit
    for got, ref in ((c, torch.cos(ang)), (s, torch.sin(ang))):
        assert np.array_equal(mimic.f32(got), got)        # values on the fp32 grid
        d = _fp32_ulp_dist(got, ref.numpy())
        assert d.max() <= 1
        assert np.mean(d == 0) >= 0.9


@pytest.mark.parametrize("interleaved", [False, True])
@pytest.mark.parametrize("D", [32, 80, 128])
def test_rope_step_against_torch_ops(D, interleaved):
    x, _ = _rand_rows(200, 3, D, seed=21 + D)
    rng = np.random.default_rng(D)
    pos = rng.integers(0, 256, size=(200, 2)).astype(np.int32)
    got = mimic.norm_rope(wl.bf16_bits(x), pos, 10000.0, None, False, 1e-6, interleaved)
    ref = wl.bf16_bits(_torch_rope(x, pos, 10000.0, interleaved))
    d = _ulp_dist(got, ref)
    assert d.max() <= 1
    assert np.mean(d == 0) >= 0.99


def _derived_bound(ref: np.ndarray, interleaved: bool) -> np.ndarray:
    """2^-6 * r + 1e-5 per element, r the norm of the element's rotation pair (the
    bound the GPU prologue tests use, derived from the roundings modelled here)."""
    D = ref.shape[-1]
    if interleaved:
        r = np.sqrt(ref[..., 0::2] ** 2 + ref[..., 1::2] ** 2)
        r = np.repeat(r, 2, axis=-1)
    else:
        r = np.sqrt(ref[..., : D // 2] ** 2 + ref[..., D // 2:] ** 2)
        r = np.concatenate([r, r], axis=-1)
    return 2.0 ** -6 * r + 1e-5


@pytest.mark.parametrize("interleaved", [False, True])
@pytest.mark.parametrize("idx", [1, 3, 4, 5])
def test_mimic_prologue_within_the_derived_bound(idx, interleaved):
    w = wl.make_config(idx)
    t = w.tensors()
    _, pos = oracle.grid_positions(w.grid_hw)
    T = w.total_tokens
    rows = np.unique(np.linspace(0, T - 1, min(T, 2048)).astype(np.int64))
    nw = None if t["norm_w"] is None else wl.bf16_bits(t["norm_w"])
    for name, wrow in (("q", 0), ("k", 1)):
        x = wl.bf16_bits(t[name])[rows]
        wv = None if nw is None else nw[wrow]
        exact = oracle.norm_rope(x, pos[rows], w.theta, wv, w.qk_norm, w.eps, interleaved)
        got = oracle.widen(mimic.norm_rope(x, pos[rows], w.theta, wv, w.qk_norm, w.eps, interleaved))
        err = np.abs(got - exact)
        assert np.all(err <= _derived_bound(exact, interleaved)), (name, float(err.max()))
        assert err.max() > 0                     # the roundings are really there


# ---------------------------------------------------------------- the attention step

def _torch_segment_attention(q, k, v):
    """q, k, v bf16 [L, H, D] of one segment -> bf16 [L, H, D] with PyTorch CPU ops."""
    D = q.shape[-1]
    qh, kh, vh = (t.transpose(0, 1) for t in (q, k, v))
    s = torch.bmm(qh, kh.transpose(1, 2)) / math.sqrt(D)
    p = torch.softmax(s, dim=-1, dtype=torch.float32).to(torch.bfloat16)
    return torch.bmm(p, vh).transpose(0, 1)


def _torch_dense_attention(q, k, v, cu):
    T, H, D = q.shape
    bias = torch.full((T, T), torch.finfo(torch.bfloat16).min, dtype=torch.bfloat16)
    for i in range(len(cu) - 1):
        bias[cu[i]:cu[i + 1], cu[i]:cu[i + 1]] = 0
    qh, kh, vh = (t.transpose(0, 1) for t in (q, k, v))
    s = torch.bmm(qh, kh.transpose(1, 2)) / math.sqrt(D) + bias
    p = torch.softmax(s, dim=-1, dtype=torch.float32).to(torch.bfloat16)
    return torch.bmm(p, vh).transpose(0, 1)


@pytest.mark.parametrize("D", [32, 80, 128])
def test_attention_step_against_torch_ops(D):
    lengths = [1, 17, 64, 0, 200, 129]
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    T, H = int(cu[-1]), 3
    g = torch.Generator().manual_seed(31 + D)
    q, k, v = (torch.randn((T, H, D), generator=g).to(torch.bfloat16) for _ in range(3))
    got = mimic.attention(*(oracle.widen(wl.bf16_bits(t)) for t in (q, k, v)), cu)
    got_bits = mimic.to_bits(got)
    per_seg = torch.cat([_torch_segment_attention(q[a:b], k[a:b], v[a:b])
                         for a, b in zip(cu[:-1], cu[1:]) if b > a])
    dense = _torch_dense_attention(q, k, v, [int(c) for c in cu])
    # PyTorch's fp32 sums and exp differ from exact-then-rounded in rare near-ties; one flipped
    # rounding of a weight moves an output by a fraction of a unit of |v| ~ 1, which can be a
    # few units of a small output, so the pin counts equal results and bounds the absolute
    # difference. Leaving out any one rounding of the step (scores, scaled scores, weights,
    # output) drops the equal fraction below 0.6 on these inputs.
    for ref in (per_seg, dense):
        assert np.mean(got_bits == wl.bf16_bits(ref)) >= 0.999
        assert np.max(np.abs(got - ref.double().numpy())) <= 2.0 ** -9


def test_attention_rows_subset_and_uncovered():
    lengths = [5, 40, 23]
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    T = int(cu[-1])
    g = torch.Generator().manual_seed(41)
    q, k, v = (oracle.widen(wl.bf16_bits(torch.randn((T + 2, 2, 32), generator=g).to(torch.bfloat16)))
               for _ in range(3))
    full = mimic.attention(q, k, v, cu)
    rows = [67, 0, 44, 45, 4]
    assert np.array_equal(mimic.attention(q, k, v, cu, rows=rows), full[rows])
    assert np.all(np.isnan(full[T:]))            # tokens outside every segment have no value
    assert not np.any(np.isnan(full[:T]))


# ---------------------------------------------------------------- planted mistakes

_MIMIC_MUTANTS = {
    "norm not cast back before the weight": ("y = bf16_round(f32(x * r))", "y = f32(x * r)"),
    "eps outside the square root": ("r = f32(1.0 / np.sqrt(f32(mean + f32(eps))))",
                                    "r = f32(1.0 / np.sqrt(f32(mean)) + eps)"),
    "mean over D - 1": ("mean = f32(ss / D)", "mean = f32(ss / (D - 1))"),
    "weight ignored": ("return bf16_round(y * w)", "return bf16_round(y)"),
    "rotation sign": ("y[..., : D // 2] = f32(f32(a * c) - f32(b * s))",
                      "y[..., : D // 2] = f32(f32(a * c) + f32(b * s))"),
    "row and column swapped": ("[f32(np.outer(pos[:, 0], inv)), f32(np.outer(pos[:, 1], inv))]",
                               "[f32(np.outer(pos[:, 1], inv)), f32(np.outer(pos[:, 0], inv))]"),
    "cos/sin not rounded to fp32": ("return f32(np.cos(a)), f32(np.sin(a))", "return np.cos(a), np.sin(a)"),
    "table for the wrong dim": ("inv = inv_freq_fp32(D // 2, theta)", "inv = inv_freq_fp32(D, theta)[: D // 4]"),
    "scores not rounded": ("s = bf16_round(q[want[rs], h] @ kh.T)", "s = q[want[rs], h] @ kh.T"),
    "scaled scores not rounded": ("s = bf16_round(f32(s / sqrt_d))", "s = f32(s / sqrt_d)"),
    "weights not cast to bf16": ("p = bf16_round(f32(e / f32(e.sum(axis=-1, keepdims=True))))",
                                 "p = f32(e / f32(e.sum(axis=-1, keepdims=True)))"),
    "output not rounded": ("out[rs, h] = bf16_round(p @ vh)", "out[rs, h] = f32(p @ vh)"),
}


@pytest.mark.parametrize("name", sorted(_MIMIC_MUTANTS))
def test_planted_mimic_mistake_fails_a_pin(name, monkeypatch):
    import sys
    import types
    with open(mimic.__file__) as f:
        src = f.read()
    old, new = _MIMIC_MUTANTS[name]
    assert src.count(old) == 1, name
    mod = types.ModuleType("mimic_mutant")
    mod.__dict__["__package__"] = "oracle"
    exec(compile(src.replace(old, new), mimic.__file__, "exec"), mod.__dict__)
    monkeypatch.setattr(sys.modules[__name__], "mimic", mod)
    pins = [(test_norm_step_against_torch_ops, (80, 1.0, 1e-6)),
            (test_norm_step_against_torch_ops, (80, 2.0 ** -10, 1e-6)),
            (test_angle_table_against_torch_fp32, (80,)),
            (test_rope_step_against_torch_ops, (80, False)),
            (test_rope_step_against_torch_ops, (80, True)),
            (test_attention_step_against_torch_ops, (80,))]
    failed = 0
    for fn, args in pins:
        try:
            fn(*args)
        except AssertionError:
            failed += 1
    assert failed > 0, f"the mutant '{name}' passes every pin"
