"""Pins of the fp64 oracle against things other than itself (CPU only).

Each test ties one oracle function to a value worked by hand from the pages
(tests/golden), a closed form, an invariant, a library routine, or brute
force, so that a dropped term, a wrong sign or index, or a transposed operand
in the oracle fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle.dense_ref import dense_block_diag_attention
from vision_encoder_varlen_gb300 import workloads as wl

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def _bits(a):
    """fp64 values that are exact in bf16 -> bf16 bit patterns."""
    t = torch.tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)
    assert np.array_equal(t.float().numpy(), np.asarray(a, dtype=np.float32)), "value not exact in bf16"
    return wl.bf16_bits(t)


# ---------------------------------------------------------------- frequencies / positions

def test_inv_freq_golden(golden_dir):
    g = _load(golden_dir, "rope_inv_freq.json")
    for case in g["cases"]:
        got = oracle.rope_inv_freq(case["dim"], case["theta"])
        assert got.shape == (case["dim"] // 2,)
        if "inv_freq" in case:
            np.testing.assert_allclose(got, case["inv_freq"], rtol=1e-14, atol=0)
        for j, val in case.get("index_value", []):
            assert got[j] == pytest.approx(val, rel=1e-14)


def test_inv_freq_ratio_is_constant():
    # consecutive frequencies differ by the factor theta^(-2/dim): a geometric table
    for dim in (8, 20, 32, 40, 64):
        f = oracle.rope_inv_freq(dim, 10000.0)
        r = f[1:] / f[:-1]
        np.testing.assert_allclose(r, 10000.0 ** (-2.0 / dim), rtol=1e-13)
        assert f[0] == 1.0


def test_grid_positions_golden(golden_dir):
    g = _load(golden_dir, "grid_positions.json")
    cu, pos = oracle.grid_positions(g["grid_hw"])
    assert cu.tolist() == g["cu_seqlens"]
    assert pos.tolist() == g["pos_hw"]


def test_grid_positions_bruteforce_workloads():
    for idx in (1, 3, 5):
        w = wl.make_config(idx)
        cu, pos = oracle.grid_positions(w.grid_hw)
        assert np.array_equal(cu, w.cu_seqlens)
        expect = [(r, c) for (h, ww) in w.grids for r in range(h) for c in range(ww)]
        assert np.array_equal(pos, np.array(expect, dtype=np.int32).reshape(-1, 2))


# ---------------------------------------------------------------- RMSNorm + RoPE

def test_rope_norm_golden(golden_dir):
    g = _load(golden_dir, "rope_norm_cases.json")
    for case in g["cases"]:
        x = np.asarray(case["x"])
        D = x.shape[0]
        xb = _bits(x).reshape(1, 1, D)
        w = None if case["w"] is None else _bits(case["w"])
        pos = np.array([case["pos"]], dtype=np.int32)
        y = oracle.norm_rope(xb, pos, 10000.0, w, case["norm"], case["eps"], case.get("interleaved", False))
        np.testing.assert_allclose(y.reshape(D), case["y"], rtol=0, atol=1e-14, err_msg=case["what"])


def test_rope_matches_complex_rotation():
    # independent formulation: pair (x[m], x[m+D/2]) as the complex number x[m] + i x[m+D/2]
    # multiplied by exp(i a_m) with a_m = row*f_m (m < D/4) or col*f_{m-D/4}
    rng = np.random.default_rng(1)
    D, H, T = 16, 2, 5
    xb = wl.bf16_bits(torch.randn(T, H, D).to(torch.bfloat16))
    x = oracle.widen(xb)
    pos = rng.integers(0, 300, size=(T, 2)).astype(np.int32)
    f = 10000.0 ** (-np.arange(D // 4) * 4.0 / D)        # table of dim D/2: theta^(-2j/(D/2))
    y = oracle.norm_rope(xb, pos)
    for t in range(T):
        ang = np.concatenate([pos[t, 0] * f, pos[t, 1] * f])
        z = (x[t, :, : D // 2] + 1j * x[t, :, D // 2:]) * np.exp(1j * ang)[None]
        np.testing.assert_allclose(y[t, :, : D // 2], z.real, atol=1e-12)
        np.testing.assert_allclose(y[t, :, D // 2:], z.imag, atol=1e-12)


def test_interleaved_rope_matches_complex_rotation():
    # pair (x[2m], x[2m+1]) as the complex number x[2m] + i x[2m+1] multiplied by exp(i a_m)
    rng = np.random.default_rng(2)
    D, H, T = 16, 2, 5
    xb = wl.bf16_bits(torch.randn(T, H, D).to(torch.bfloat16))
    x = oracle.widen(xb)
    pos = rng.integers(0, 300, size=(T, 2)).astype(np.int32)
    f = 10000.0 ** (-np.arange(D // 4) * 4.0 / D)
    y = oracle.norm_rope(xb, pos, interleaved=True)
    for t in range(T):
        ang = np.concatenate([pos[t, 0] * f, pos[t, 1] * f])
        z = (x[t, :, 0::2] + 1j * x[t, :, 1::2]) * np.exp(1j * ang)[None]
        np.testing.assert_allclose(y[t, :, 0::2], z.real, atol=1e-12)
        np.testing.assert_allclose(y[t, :, 1::2], z.imag, atol=1e-12)


def test_interleaved_is_rotate_half_under_a_permutation():
    # moving element 2m to m and 2m+1 to m + D/2 turns one mode into the other, with norm and weight
    torch.manual_seed(13)
    D, H, T = 80, 3, 6
    x = torch.randn(T, H, D).to(torch.bfloat16)
    w = (1 + 0.1 * torch.randn(D)).to(torch.bfloat16)
    perm = np.concatenate([np.arange(0, D, 2), np.arange(1, D, 2)])     # half-layout index -> interleaved index
    pos = np.random.default_rng(4).integers(0, 64, size=(T, 2)).astype(np.int32)
    yi = oracle.norm_rope(wl.bf16_bits(x), pos, w_bits=wl.bf16_bits(w), use_norm=True, eps=1e-6, interleaved=True)
    yh = oracle.norm_rope(wl.bf16_bits(x[..., perm].contiguous()), pos, w_bits=wl.bf16_bits(w[perm].contiguous()),
                          use_norm=True, eps=1e-6)
    np.testing.assert_allclose(yi[..., perm], yh, rtol=0, atol=1e-13)
    assert not np.allclose(yi, oracle.norm_rope(wl.bf16_bits(x), pos, w_bits=wl.bf16_bits(w), use_norm=True,
                                                eps=1e-6))


def test_rope_identity_at_origin_and_pair_norms():
    torch.manual_seed(3)
    D, H, T = 80, 3, 7
    xb = wl.bf16_bits(torch.randn(T, H, D).to(torch.bfloat16))
    x = oracle.widen(xb)
    pos0 = np.zeros((T, 2), dtype=np.int32)
    assert np.array_equal(oracle.norm_rope(xb, pos0), x)
    pos = np.random.default_rng(0).integers(0, 256, size=(T, 2)).astype(np.int32)
    y = oracle.norm_rope(xb, pos)
    n_in = x[..., : D // 2] ** 2 + x[..., D // 2:] ** 2
    n_out = y[..., : D // 2] ** 2 + y[..., D // 2:] ** 2
    np.testing.assert_allclose(n_out, n_in, rtol=1e-12, atol=1e-12)
    # the interleaved mode: identity at the origin, adjacent-pair norms kept elsewhere
    assert np.array_equal(oracle.norm_rope(xb, pos0, interleaved=True), x)
    yi = oracle.norm_rope(xb, pos, interleaved=True)
    np.testing.assert_allclose(yi[..., 0::2] ** 2 + yi[..., 1::2] ** 2, x[..., 0::2] ** 2 + x[..., 1::2] ** 2,
                               rtol=1e-12, atol=1e-12)


def test_rope_relative_offsets_only():
    # <R(p) q, R(p') k> depends only on p' - p (per row and per column offset)
    torch.manual_seed(5)
    D = 32
    qb = wl.bf16_bits(torch.randn(1, 1, D).to(torch.bfloat16))
    kb = wl.bf16_bits(torch.randn(1, 1, D).to(torch.bfloat16))
    rng = np.random.default_rng(7)
    for _ in range(20):
        p = rng.integers(0, 200, 2)
        dp = rng.integers(-50, 50, 2)
        p2 = p + dp
        if (p2 < 0).any():
            continue
        shift = rng.integers(0, 100, 2)
        dots = []
        for a, b in ((p, p2), (p + shift, p2 + shift)):
            qr = oracle.norm_rope(qb, np.array([a], dtype=np.int32))
            kr = oracle.norm_rope(kb, np.array([b], dtype=np.int32))
            dots.append(float(np.sum(qr * kr)))
        assert dots[0] == pytest.approx(dots[1], abs=1e-12)


def test_rope_row_position_moves_first_half_only():
    torch.manual_seed(9)
    D = 80
    xb = wl.bf16_bits(torch.randn(1, 1, D).to(torch.bfloat16))
    x = oracle.widen(xb)
    y = oracle.norm_rope(xb, np.array([[37, 0]], dtype=np.int32))
    q = D // 4
    # the column-angle pairs m in [D/4, D/2) are untouched when col == 0
    np.testing.assert_array_equal(y[0, 0, q:D // 2], x[0, 0, q:D // 2])
    np.testing.assert_array_equal(y[0, 0, D // 2 + q:], x[0, 0, D // 2 + q:])
    assert not np.allclose(y[0, 0, :q], x[0, 0, :q])


def test_rmsnorm_unit_rms_and_scale_invariance():
    torch.manual_seed(11)
    D, H, T = 80, 4, 6
    x = torch.randn(T, H, D).to(torch.bfloat16)
    xb = wl.bf16_bits(x)
    pos0 = np.zeros((T, 2), dtype=np.int32)
    y = oracle.norm_rope(xb, pos0, use_norm=True, eps=0.0)
    rms = np.sqrt(np.mean(y * y, axis=-1))
    np.testing.assert_allclose(rms, 1.0, rtol=1e-14)
    # scaling the input by a power of two (exact in bf16) leaves the eps=0 norm unchanged
    y2 = oracle.norm_rope(wl.bf16_bits(x * 4), pos0, use_norm=True, eps=0.0)
    np.testing.assert_allclose(y2, y, rtol=1e-14, atol=1e-15)
    # the per-element weight multiplies the normalised vector
    wb = wl.bf16_bits(torch.linspace(0.5, 2.0, D).to(torch.bfloat16))
    yw = oracle.norm_rope(xb, pos0, w_bits=wb, use_norm=True, eps=0.0)
    np.testing.assert_allclose(yw, y * oracle.widen(wb)[None, None, :], rtol=1e-14, atol=1e-15)


# ---------------------------------------------------------------- attention

def _rand_qkv(T, H, D, seed):
    g = torch.Generator().manual_seed(seed)
    return [oracle.widen(wl.bf16_bits(torch.randn(T, H, D, generator=g).to(torch.bfloat16))) for _ in range(3)]


def test_attention_worked_example(golden_dir):
    g = _load(golden_dir, "attention_worked.json")
    out = oracle.attention(np.array(g["q"]), np.array(g["k"]), np.array(g["v"]), g["cu_seqlens"], g["scale"])
    np.testing.assert_allclose(out, np.array(g["out"]), rtol=0, atol=1e-14)


def test_form_a_equals_form_b():
    cu = [0, 5, 5, 17, 18, 40]          # includes an empty and a one-token segment
    q, k, v = _rand_qkv(40, 3, 16, 21)
    a = dense_block_diag_attention(q, k, v, cu)
    b = oracle.attention(q, k, v, cu)
    np.testing.assert_allclose(b, a, rtol=0, atol=1e-12)


def test_single_segment_equals_library_sdpa():
    T, H, D = 50, 4, 32
    q, k, v = _rand_qkv(T, H, D, 33)
    b = oracle.attention(q, k, v, [0, T])
    tq, tk, tv = (torch.from_numpy(x).permute(1, 0, 2).unsqueeze(0) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv)     # default scale 1/sqrt(D)
    np.testing.assert_allclose(b, ref[0].permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)
    # an explicit non-default scale goes through the same routine
    b2 = oracle.attention(q, k, v, [0, T], scale=0.37)
    ref2 = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=0.37)
    np.testing.assert_allclose(b2, ref2[0].permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


def test_bruteforce_python_loops():
    cu = [0, 3, 7]
    T, H, D = 7, 2, 4
    q, k, v = _rand_qkv(T, H, D, 44)
    out = oracle.attention(q, k, v, cu)
    scale = 1.0 / math.sqrt(D)
    for s in range(len(cu) - 1):
        for t in range(cu[s], cu[s + 1]):
            for h in range(H):
                sc = [scale * sum(q[t, h, d] * k[u, h, d] for d in range(D)) for u in range(cu[s], cu[s + 1])]
                m = max(sc)
                e = [math.exp(x - m) for x in sc]
                z = sum(e)
                for d in range(D):
                    o = sum(e[i] / z * v[cu[s] + i, h, d] for i in range(len(e)))
                    assert out[t, h, d] == pytest.approx(o, abs=1e-13)


def test_constant_v_and_zero_q():
    cu = [0, 9, 30, 31]
    T, H, D = 31, 2, 8
    q, k, v = _rand_qkv(T, H, D, 55)
    vc = np.broadcast_to(np.arange(1, D + 1, dtype=np.float64), (T, H, D)).copy()
    np.testing.assert_allclose(oracle.attention(q, k, vc, cu), vc, rtol=1e-14)
    out = oracle.attention(np.zeros_like(q), k, v, cu)
    for s in range(len(cu) - 1):
        mean = v[cu[s]:cu[s + 1]].mean(axis=0)
        np.testing.assert_allclose(out[cu[s]:cu[s + 1]], np.broadcast_to(mean, out[cu[s]:cu[s + 1]].shape),
                                   rtol=0, atol=1e-14)


def test_segment_isolation_bitwise():
    cu = [0, 10, 25, 26, 40]
    T, H, D = 40, 2, 16
    q, k, v = _rand_qkv(T, H, D, 66)
    base = oracle.attention(q, k, v, cu)
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    q2[10:25] += 1.0
    k2[10:25] *= -2.0
    v2[10:25] = 0.5
    pert = oracle.attention(q2, k2, v2, cu)
    keep = np.r_[0:10, 25:40]
    assert np.array_equal(pert[keep], base[keep])
    assert not np.allclose(pert[10:25], base[10:25])


def test_rows_subset_is_exact_slice():
    cu = [0, 13, 40]
    q, k, v = _rand_qkv(40, 2, 8, 77)
    full = oracle.attention(q, k, v, cu)
    rows = [0, 12, 13, 39, 5]
    sub = oracle.attention(q, k, v, cu, rows=rows)
    assert np.array_equal(sub, full[rows])


def test_uncovered_token_is_nan():
    q, k, v = _rand_qkv(6, 1, 4, 88)
    out = oracle.attention(q, k, v, [0, 4])
    assert np.isnan(out[4:]).all() and np.isfinite(out[:4]).all()


def test_full_path_composes_steps():
    w = wl.make_config(1)
    t = w.tensors()
    qb, kb, vb = (wl.bf16_bits(t[n]) for n in ("q", "k", "v"))
    out = oracle.full_path(w.grid_hw, qb, kb, vb)
    cu, pos = oracle.grid_positions(w.grid_hw)
    ref = dense_block_diag_attention(oracle.norm_rope(qb, pos), oracle.norm_rope(kb, pos), oracle.widen(vb), cu)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- log-sum-exp output

def test_lse_zero_q_is_log_segment_length():
    # all scores 0: sum of L ones
    cu = [0, 1, 9, 30, 30, 101]
    q, k, v = _rand_qkv(101, 3, 8, 91)
    _, lse = oracle.attention(np.zeros_like(q), k, v, cu, return_lse=True)
    for s in range(len(cu) - 1):
        L = cu[s + 1] - cu[s]
        np.testing.assert_allclose(lse[cu[s]:cu[s + 1]], math.log(L) if L else 0.0, rtol=0, atol=1e-13)


def test_lse_geometric_series_closed_form():
    # q = (c, 0), k_j = (j, 7): scores a*j with a = c*scale, sum_j e^(a j) = (e^(a L) - 1) / (e^a - 1)
    L, c = 37, 0.3
    scale = 1.0 / math.sqrt(2)
    q = np.zeros((L, 1, 2)); q[:, 0, 0] = c
    k = np.zeros((L, 1, 2)); k[:, 0, 0] = np.arange(L); k[:, 0, 1] = 7.0
    v = np.ones((L, 1, 2))
    _, lse = oracle.attention(q, k, v, [0, L], return_lse=True)
    a = c * scale
    np.testing.assert_allclose(lse[:, 0], math.log((math.exp(a * L) - 1.0) / (math.exp(a) - 1.0)), rtol=1e-14)


def test_lse_single_key_is_the_score():
    q, k, v = _rand_qkv(4, 2, 16, 92)
    _, lse = oracle.attention(q, k, v, [0, 1, 2, 3, 4], scale=0.25, return_lse=True)
    np.testing.assert_allclose(lse, 0.25 * np.sum(q * k, axis=-1), rtol=0, atol=1e-13)


def test_lse_equals_library_logsumexp():
    cu = [0, 5, 5, 17, 18, 40]
    q, k, v = _rand_qkv(40, 3, 16, 93)
    out, lse = oracle.attention(q, k, v, cu, scale=0.2, return_lse=True)
    np.testing.assert_array_equal(out, oracle.attention(q, k, v, cu, scale=0.2))
    for s in range(len(cu) - 1):
        a, b = cu[s], cu[s + 1]
        if a == b:
            continue
        tq, tk = torch.from_numpy(q[a:b]), torch.from_numpy(k[a:b])
        sc = torch.einsum("thd,uhd->htu", tq, tk) * 0.2
        ref = torch.logsumexp(sc, dim=-1).transpose(0, 1).numpy()
        np.testing.assert_allclose(lse[a:b], ref, rtol=0, atol=1e-12)


def test_lse_shifts_with_a_common_key_offset():
    # adding one vector u to every key of a segment adds scale*<q, u> to every score of its rows:
    # the lse moves by exactly that, the softmax and the output do not move
    cu = [0, 11, 30]
    q, k, v = _rand_qkv(30, 2, 8, 94)
    out, lse = oracle.attention(q, k, v, cu, return_lse=True)
    u = np.random.default_rng(5).standard_normal((1, 2, 8))
    k2 = k.copy(); k2[11:30] += u
    out2, lse2 = oracle.attention(q, k2, v, cu, return_lse=True)
    scale = 1.0 / math.sqrt(8)
    np.testing.assert_allclose(lse2[11:30], lse[11:30] + scale * np.sum(q[11:30] * u, axis=-1), atol=1e-12)
    assert np.array_equal(lse2[:11], lse[:11])
    np.testing.assert_allclose(out2, out, atol=1e-12)


def test_lse_rows_subset_and_uncovered_token():
    cu = [0, 13, 40]
    q, k, v = _rand_qkv(42, 2, 8, 95)
    _, full = oracle.attention(q, k, v, cu, return_lse=True)
    _, sub = oracle.attention(q, k, v, cu, rows=[0, 39, 12, 13], return_lse=True)
    assert np.array_equal(sub, full[[0, 39, 12, 13]])
    assert np.isnan(full[40:]).all() and np.isfinite(full[:40]).all()
