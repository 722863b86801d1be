"""The C-ABI library: it builds, loads without a GPU, exports every declared
symbol, and rejects host-detectable bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

import vision_encoder_varlen_gb300 as vit
from vision_encoder_varlen_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "vit_attn.h")


@pytest.fixture(scope="module")
def L():
    _build.build()
    return vit.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(vit_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_three_calls():
    names = declared_functions()
    for n in ("vit_rope_freqs", "vit_qk_norm_rope", "vit_varlen_attn"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, missing


def test_status_strings(L):
    assert vit.status_string(0) == "ok"
    for code in range(-1, -16, -1):
        s = vit.status_string(code)
        assert s and s != "unknown status", code
    assert vit.status_string(-999) == "unknown status"
    assert "sm_103a" in vit.version()


def test_workspace_size_bounds(L):
    # header + one 16-byte item per (head, 64-row block) plus one per segment and head
    assert vit.workspace_size(1024, 16, 1, 80) == 64 + 16 * 16 * (16 + 1)
    assert vit.workspace_size(0, 4, 0, 32) == 64
    assert vit.workspace_size(100, 4, 2, 81) == 0        # bad head_dim
    assert vit.workspace_size(100, 0, 2, 80) == 0        # no heads
    assert vit.workspace_size(100, 4, 8193, 80) == 0     # too many segments
    assert vit.workspace_size(2 ** 31 - 1, 64, 1, 80) == 0   # work list past 2^31 items
    assert vit.workspace_size(2 ** 31 - 1, 63, 1, 80) > 0


def _attn(L, **kw):
    args = dict(q=8, k=8, v=8, T=128, H=2, D=80, qs=160, ks=160, vs=160, cu=16, B=1, max_seqlen=128, scale=0.0,
                out=8, os=160, ws=256, ws_bytes=1 << 20, status=None, stream=None)
    args.update(kw)
    a = args
    p = lambda x: None if x is None else ctypes.c_void_p(x)
    return L.vit_varlen_attn(p(a["q"] * 16 if a["q"] else None), p(a["k"] * 16 if a["k"] else None),
                             p(a["v"] * 16 if a["v"] else None), a["T"], a["H"], a["D"], a["qs"], a["ks"], a["vs"],
                             p(a["cu"]), a["B"], a["max_seqlen"], a["scale"], p(a["out"] * 16 if a["out"] else None),
                             a["os"], p(a["ws"]), a["ws_bytes"], p(a["status"]), p(a["stream"]))


def test_host_validation_without_gpu(L):
    # every case below fails a host check, so nothing reaches the CUDA runtime
    assert _attn(L, D=81) == -2
    assert _attn(L, H=0) == -3
    assert _attn(L, T=-1) == -3
    assert _attn(L, B=9000) == -7
    assert _attn(L, B=0) == -3                      # T > 0 but no segment
    assert _attn(L, qs=100) == -4                   # stride < H*D
    assert _attn(L, ks=164) == -4                   # stride not a multiple of 8
    assert _attn(L, q=0) == -1
    assert _attn(L, ws=0) == -1
    assert _attn(L, ws=264) == -5                   # workspace misaligned
    assert _attn(L, ws_bytes=64) == -6
    assert _attn(L, max_seqlen=-1) == -14            # 0 means "not given" (T bounds it); negative is an error
    assert _attn(L, scale=float("nan")) == -14
    assert _attn(L, cu=0, B=3) == -14               # uniform split needs T % B == 0
    assert _attn(L, T=0, B=0) == 0                  # nothing to do
    # token indices are int32 (cu_seqlens, positions, work items): T must stay below 2^31,
    # including for the uniform split, whose segment starts the scheduler derives from T
    assert _attn(L, T=1 << 31, max_seqlen=1 << 30) == -3
    assert _attn(L, T=1 << 31, cu=0, B=2, max_seqlen=1 << 30) == -3


def test_prologue_and_rope_validation_without_gpu(L):
    p = ctypes.c_void_p
    assert L.vit_qk_norm_rope(p(16), p(16), p(16), p(16), 10, 2, 72, 144, 144, 144, 144, p(16), p(16), None,
                              1e-6, None) == -2
    assert L.vit_qk_norm_rope(None, p(16), p(16), p(16), 10, 2, 80, 160, 160, 160, 160, p(16), p(16), None,
                              1e-6, None) == -1
    assert L.vit_qk_norm_rope(p(16), p(16), p(16), p(16), 10, 2, 80, 160, 160, 160, 160, p(16), p(16), None,
                              -1.0, None) == -14
    assert L.vit_qk_norm_rope(p(16), p(32), p(16), p(16), 10, 2, 80, 160, 160, 168, 160, p(16), p(16), None,
                              1e-6, None) == -4  # in-place k with different strides
    assert L.vit_qk_norm_rope(p(16), p(16), p(16), p(16), 0, 2, 80, 160, 160, 160, 160, None, None, None,
                              1e-6, None) == 0   # empty: nothing to do
    assert L.vit_rope_freqs(3, 10000.0, p(16), 1, 4, p(16), p(16), p(16), None, None) == -14   # odd dim
    assert L.vit_rope_freqs(40, -1.0, p(16), 1, 4, p(16), p(16), p(16), None, None) == -14     # theta <= 0
    assert L.vit_rope_freqs(40, 10000.0, None, 1, 4, p(16), p(16), p(16), None, None) == -1
    assert L.vit_rope_freqs(40, 10000.0, p(16), 9000, 4, p(16), p(16), p(16), None, None) == -7
    assert L.vit_rope_freqs(40, 10000.0, p(16), 1, 4, None, None, None, None, None) == 0
    assert L.vit_rope_freqs(40, 10000.0, p(16), 1, 1 << 31, p(16), p(16), p(16), None, None) == -3
    assert L.vit_qk_norm_rope(p(16), p(16), p(16), p(16), 1 << 31, 2, 80, 160, 160, 160, 160, p(16), p(16),
                              None, 1e-6, None) == -3


def test_extended_calls_validation_without_gpu(L):
    p = ctypes.c_void_p
    ex = L.vit_qk_norm_rope_ex
    good = dict(qi=16, qo=16, ki=16, ko=16, mode=0)

    def call(**kw):
        a = dict(good, **kw)
        return ex(p(a["qi"]) if a["qi"] else None, p(a["qo"]) if a["qo"] else None,
                  p(a["ki"]) if a["ki"] else None, p(a["ko"]) if a["ko"] else None, 10, 2, 80, 160, 160, 160, 160,
                  p(16), p(16), None, 1e-6, a["mode"], None, None)
    assert call(mode=2) == -14                       # unknown rotary pairing
    assert call(mode=-1) == -14
    assert call(qo=0) == -1                          # half a q pair
    assert call(ki=0) == -1                          # half a k pair
    assert call(qi=0, qo=0, ki=0, ko=0) == -1        # nothing to do is a caller error
    # vit_varlen_attn_lse: same checks as vit_varlen_attn plus the lse alignment
    args = [p(16), p(16), p(16), 128, 2, 80, 160, 160, 160, p(16), 1, 128, 0.0, p(16), 160]
    assert L.vit_varlen_attn_lse(*args, p(18), p(256), 1 << 20, None, None) == -5
    args_bad = list(args)
    args_bad[5] = 81
    assert L.vit_varlen_attn_lse(*args_bad, p(16), p(256), 1 << 20, None, None) == -2


def test_fused_q_and_table_validation_without_gpu(L):
    p = ctypes.c_void_p
    assert L.vit_rope_table(p(16), 81, 10, p(16), None) == -2
    assert L.vit_rope_table(p(16), 80, 0, p(16), None) == -14
    assert L.vit_rope_table(None, 80, 10, p(16), None) == -1
    assert L.vit_rope_table(p(16), 80, 10, p(24), None) == -5

    def fused(qr):
        return L.vit_varlen_attn_fused_q(p(16), p(16), p(16), 128, 2, 80, 160, 160, 160,
                                         None if qr is None else ctypes.byref(qr), p(16), 1, 128, 0.0, p(16), 160,
                                         None, p(256), 1 << 20, None, None)
    QR = vit._QRope
    assert fused(None) == -1
    assert fused(QR(16, 16, 64, None, 1e-6, 2)) == -14          # unknown rotary pairing
    assert fused(QR(16, 16, 0, None, 1e-6, 0)) == -14           # empty table
    assert fused(QR(16, 16, 64, None, -1.0, 0)) == -14          # eps < 0
    assert fused(QR(None, 16, 64, None, 1e-6, 0)) == -1
    assert fused(QR(16, 24, 64, None, 1e-6, 0)) == -5           # table not 16-byte aligned
    assert fused(QR(16, 16, 64, 18, 1e-6, 0)) == -5             # weight not 16-byte aligned


def test_padded_call_validation_without_gpu(L):
    p = ctypes.c_void_p

    def padded(B, start, length, D=80):
        return L.vit_varlen_attn_padded(p(16), p(16), p(16), 4096, 2, D, 160, 160, 160,
                                        None if start is None else p(start), None if length is None else p(length),
                                        B, 512, 0.0, p(16), 160, None, None, p(256), 1 << 20, None, None)
    assert padded(0, None, None) == 0              # nothing to compute
    assert padded(2, 16, None) == -1
    assert padded(2, None, 16) == -1
    assert padded(2, 16, 18) == -5                 # seq_len not 4-byte aligned
    assert padded(2, 16, 16, D=81) == -2


def test_general_call_validation_without_gpu(L):
    p = ctypes.c_void_p
    O = vit._AttnOptions

    def ex(cu=16, start=None, length=None, B=1, opts=None, D=80):
        return L.vit_varlen_attn_ex(p(16), p(16), p(16), 4096, 2, D, 160, 160, 160, None if cu is None else p(cu),
                                    None if start is None else p(start), None if length is None else p(length), B,
                                    512, 0.0, p(16), 160, None, None, None if opts is None else ctypes.byref(opts),
                                    p(256), 1 << 20, None, None)
    assert ex(start=16, length=16, B=2) == -14        # both layouts at once
    assert ex(cu=None, start=16, length=None, B=2) == -1
    assert ex(cu=None, start=None, length=16, B=2) == -1
    assert ex(cu=None, start=16, length=16, B=0) == 0  # padded layout with no segments: nothing to do
    assert ex(opts=O(-2)) == -14                       # split below -1
    assert ex(opts=O(-1), D=81) == -2
    assert ex(cu=18) == -5                             # cu_seqlens not 4-byte aligned


def test_release_library_exports_no_test_hook_or_global_setting(L):
    # the failure-path hook lives only in a separate test build, and the kernel split is a
    # per-call option: the shipped library has neither a debug call nor a process-wide knob
    assert not hasattr(L, "vit_debug_stall_long_kernel")
    assert not hasattr(L, "vit_set_short_segment_max")
    assert "vit_debug_stall_long_kernel" not in open(HEADER).read()


def test_test_build_keeps_the_launch_path():
    # the failure-path hook only exists in the test build; that build must still launch the
    # tcgen05 kernel (its call site takes the hook's value), which the object's symbols show
    import shutil
    import subprocess
    lib = _build.build_test_hooks()
    T = ctypes.CDLL(lib)
    assert hasattr(T, "vit_debug_stall_long_kernel")
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm not available")
    syms = subprocess.run([nm, "-C", os.path.join(_build.BUILD, "api.cu.testhooks.o")], capture_output=True,
                          text=True).stdout
    assert "U vit::launch_attn_long(" in syms and "vit_debug_stall_long_kernel" in syms


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import importlib
    monkeypatch.setattr(vit, "_lib", None)
    monkeypatch.setattr(vit, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no fallback"):
        vit.lib()
