"""GPU checks of the attention path with the Q prologue fused into the Q load:
the position table against its closed form, the fused path against the
unfused one bit for bit (same arithmetic in the same order), against the fp64
oracle, and the device-side check of token positions."""
import numpy as np
import pytest
import torch

import oracle
import vision_encoder_varlen_gb300 as vit
from vision_encoder_varlen_gb300 import _build
from vision_encoder_varlen_gb300 import workloads as wl
from helpers import assert_close

pytestmark = pytest.mark.gpu

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


def _max_pos(w):
    return int(w.grid_hw.max()) if w.num_segments else 1


def _setup(w, t):
    grid = torch.from_numpy(w.grid_hw.copy()).cuda()
    inv_freq, pos, cu = vit.rope_freqs(grid, w.total_tokens, w.head_dim, w.theta)
    cs = vit.rope_table(inv_freq, w.head_dim, _max_pos(w))
    nw = t["norm_w"].cuda() if t["norm_w"] is not None else None
    return inv_freq, pos, cu, cs, nw


@pytest.mark.parametrize("D", [32, 64, 80, 96, 128])
def test_rope_table_closed_form(D):
    inv_freq = torch.from_numpy(oracle.rope_inv_freq(D // 2)).float().cuda()
    P = 300
    cs = vit.rope_table(inv_freq, D, P).cpu().numpy().astype(np.float64).reshape(P, D // 8, 4)
    f = oracle.rope_inv_freq(D // 2)
    ang = np.arange(P)[:, None] * f[None, :]                       # [P, D/4]
    cos = np.stack([cs[:, :, 0], cs[:, :, 1]], axis=-1).reshape(P, D // 4)
    sin = np.stack([cs[:, :, 2], cs[:, :, 3]], axis=-1).reshape(P, D // 4)
    # fp32 angle (relative 2^-24 of p * f, p < 300) and sincosf (a few ulp): 1e-6 + 3e-7 * angle
    tol = 1e-6 + 3e-7 * ang
    assert np.all(np.abs(cos - np.cos(ang)) <= tol)
    assert np.all(np.abs(sin - np.sin(ang)) <= tol)


def _unfused(w, t, interleaved, lse=True):
    inv_freq, pos, cu, cs, nw = _setup(w, t)
    qr, kr = vit.qk_norm_rope(t["q"].cuda(), t["k"].cuda(), pos, inv_freq, nw, w.eps, interleaved=interleaved)
    return vit.varlen_attn(qr, kr, t["v"].cuda(), cu, w.max_seqlen, return_lse=lse)


def _fused(w, t, interleaved, lse=True, status=None):
    inv_freq, pos, cu, cs, nw = _setup(w, t)
    return vit.encoder_attn(t["q"].cuda(), t["k"].cuda(), t["v"].cuda(), cu, w.max_seqlen, pos, inv_freq, cs, nw,
                            w.eps, interleaved=interleaved, return_lse=lse, status=status)


@pytest.mark.parametrize("interleaved", [False, True])
@pytest.mark.parametrize("idx", [1, 2, 3, 4])
def test_fused_equals_unfused_bitwise(idx, interleaved, split):
    w = wl.make_config(idx)
    t = w.tensors()
    out_u, lse_u = _unfused(w, t, interleaved)
    status = vit.new_status()
    out_f, lse_f = _fused(w, t, interleaved, status=status)
    assert vit.read_status(status) == 0
    assert torch.equal(out_f, out_u), f"{w.name}: fused output differs from the unfused path"
    assert torch.equal(lse_f, lse_u)


@pytest.mark.parametrize("interleaved", [False, True])
def test_fused_equals_unfused_bitwise_mixed_full_size(interleaved):
    w = wl.make_config(5)
    t = w.tensors()
    out_u, lse_u = _unfused(w, t, interleaved)
    out_f, lse_f = _fused(w, t, interleaved)
    assert torch.equal(out_f, out_u)
    assert torch.equal(lse_f, lse_u)


LENGTHS = [
    ([0, 1, 0, 63, 64, 65, 127, 128, 129, 0], 3, 80),
    ([300, 1, 257, 511, 512, 513], 2, 128),
    ([200, 33, 96, 17], 4, 96),
    ([64, 60], 4, 32),
    ([7, 9, 700], 2, 64),
]


@pytest.mark.parametrize("norm", [True, False])
@pytest.mark.parametrize("lengths,H,D", LENGTHS)
def test_fused_strips_bitwise_and_oracle(lengths, H, D, norm, split):
    # 1 x L strips: column positions up to L - 1, row position 0
    w = wl.from_lengths(lengths, H, D, qk_norm=norm, max_seqlen_meta=4096)
    t = w.tensors()
    out_u, lse_u = _unfused(w, t, False)
    out_f, lse_f = _fused(w, t, False)
    assert torch.equal(out_f, out_u)
    assert torch.equal(lse_f, lse_u)
    ref = oracle.full_path(w.grid_hw, *(wl.bf16_bits(t[n]) for n in ("q", "k", "v")),
                           wl.bf16_bits(t["norm_w"]) if norm else None, w.eps, w.theta)
    assert_close(out_f, ref, what=f"fused {lengths}")


def test_fused_packed_qkv_strides():
    w = wl.make_config(3)
    t = w.tensors()
    T, H, D = w.total_tokens, w.heads, w.head_dim
    qkv = torch.stack([t["q"], t["k"], t["v"]], dim=1).cuda()          # [T, 3, H, D]
    q, k, v = qkv[:, 0], qkv[:, 1], qkv[:, 2]
    assert q.stride(0) == 3 * H * D
    inv_freq, pos, cu, cs, nw = _setup(w, t)
    # K pre-stage in place inside the packed buffer, then attention straight from it
    out = vit.encoder_attn(q, k, v, cu, w.max_seqlen, pos, inv_freq, cs, nw, w.eps, k_out=k)
    out_u, _ = _unfused(w, t, False)
    assert torch.equal(out, out_u)


def test_position_outside_table_is_reported():
    w = wl.make_config(3)
    t = w.tensors()
    inv_freq, pos, cu, _, nw = _setup(w, t)
    small = vit.rope_table(inv_freq, w.head_dim, 8)          # every image is wider than 8 patches
    _, kr = vit.qk_norm_rope(None, t["k"].cuda(), pos, inv_freq, nw, w.eps)
    status = vit.new_status()
    vit.varlen_attn_fused_q(t["q"].cuda(), kr, t["v"].cuda(), cu, w.max_seqlen, pos, small, nw[0], w.eps,
                            status=status)
    assert vit.read_status(status) == -15
    # the context is intact: a correct call afterwards succeeds
    status.zero_()
    out = _fused(w, t, False, lse=False, status=status)
    assert vit.read_status(status) == 0
    assert torch.isfinite(out.float()).all()
