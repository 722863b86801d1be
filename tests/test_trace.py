"""NVTX tracing of the library's calls, checked on the CPU.

Every public call opens an NVTX range named after itself in the "vitattn" domain and
closes it on every return, including the early returns of argument validation. A small
NVTX tool (tests/nvtx_recorder.c, loaded through NVTX_INJECTION64_PATH) records the ranges
in a child process, which makes only calls that fail host validation: nothing reaches a
device, with or without a GPU."""
import json
import os
import shutil
import subprocess
import sys

import pytest

from vision_encoder_varlen_gb300 import _build

HERE = os.path.dirname(os.path.abspath(__file__))

_CHILD = r"""
import ctypes, json, sys
L = ctypes.CDLL(sys.argv[1])
rec = ctypes.CDLL(sys.argv[2])
vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
L.vit_rope_freqs.argtypes = [i32, f32, vp, i32, i64, vp, vp, vp, vp, vp]
L.vit_qk_norm_rope.argtypes = [vp, vp, vp, vp, i64, i32, i32, i64, i64, i64, i64, vp, vp, vp, f32, vp]
L.vit_qk_norm_rope_ex.argtypes = [vp, vp, vp, vp, i64, i32, i32, i64, i64, i64, i64, vp, vp, vp, f32, i32, vp, vp]
L.vit_rope_table.argtypes = [vp, i32, i32, vp, vp]
attn = [vp, vp, vp, i64, i32, i32, i64, i64, i64, vp, i32, i32, f32, vp, i64]
L.vit_varlen_attn.argtypes = attn + [vp, sz, vp, vp]
L.vit_varlen_attn_lse.argtypes = attn + [vp, vp, sz, vp, vp]
L.vit_varlen_attn_fused_q.argtypes = [vp, vp, vp, i64, i32, i32, i64, i64, i64, vp, vp, i32, i32, f32, vp, i64,
                                      vp, vp, sz, vp, vp]
L.vit_varlen_attn_padded.argtypes = [vp, vp, vp, i64, i32, i32, i64, i64, i64, vp, vp, i32, i32, f32, vp, i64,
                                     vp, vp, vp, sz, vp, vp]
L.vit_read_status.argtypes = [vp, vp]
rec.nvtx_recorder_ranges.restype = ctypes.c_char_p
p = ctypes.c_void_p
codes = [
    L.vit_rope_freqs(3, 10000.0, p(16), 1, 4, p(16), p(16), p(16), None, None),                  # odd dim
    L.vit_qk_norm_rope(p(16), p(16), p(16), p(16), 10, 2, 72, 144, 144, 144, 144, p(16), p(16), None,
                       1e-6, None),                                                              # head_dim 72
    L.vit_qk_norm_rope_ex(p(16), p(16), p(16), p(16), 10, 2, 80, 160, 160, 160, 160, p(16), p(16), None,
                          1e-6, 2, None, None),                                                  # rotary mode 2
    L.vit_rope_table(p(16), 81, 10, p(16), None),                                                # head_dim 81
    L.vit_varlen_attn(p(128), p(128), p(128), 128, 2, 81, 160, 160, 160, p(16), 1, 128, 0.0, p(128), 160,
                      p(256), 1 << 20, None, None),
    L.vit_varlen_attn_lse(p(128), p(128), p(128), 128, 2, 81, 160, 160, 160, p(16), 1, 128, 0.0, p(128), 160,
                          None, p(256), 1 << 20, None, None),
    L.vit_varlen_attn_fused_q(p(128), p(128), p(128), 128, 2, 80, 160, 160, 160, None, p(16), 1, 128, 0.0,
                              p(128), 160, None, p(256), 1 << 20, None, None),                   # no q_rope
    L.vit_varlen_attn_padded(p(128), p(128), p(128), 128, 2, 81, 160, 160, 160, p(16), p(16), 1, 128, 0.0,
                             p(128), 160, None, None, p(256), 1 << 20, None, None),
    L.vit_read_status(None, None),
]
print(json.dumps({"codes": codes, "ranges": rec.nvtx_recorder_ranges().decode().split(),
                  "pushes": rec.nvtx_recorder_pushes(), "pops": rec.nvtx_recorder_pops(),
                  "min_depth": rec.nvtx_recorder_min_depth()}))
"""


@pytest.fixture(scope="module")
def recorder(tmp_path_factory):
    gcc = shutil.which("gcc")
    try:
        include = os.path.join(os.path.dirname(os.path.dirname(_build._nvcc())), "include")
    except RuntimeError as e:
        pytest.skip(str(e))
    if not gcc or not os.path.exists(os.path.join(include, "nvtx3", "nvToolsExt.h")):
        pytest.skip("gcc or the NVTX 3 headers are missing")
    out = str(tmp_path_factory.mktemp("nvtx") / "libnvtx_recorder.so")
    subprocess.run([gcc, "-O2", "-std=c11", "-shared", "-fPIC", "-I", include,
                    os.path.join(HERE, "nvtx_recorder.c"), "-o", out], check=True, capture_output=True)
    return out


def test_every_public_call_is_one_closed_range(recorder):
    lib = _build.build()
    env = dict(os.environ, NVTX_INJECTION64_PATH=recorder)
    r = subprocess.run([sys.executable, "-c", _CHILD, lib, recorder], env=env, capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0, r.stderr
    got = json.loads(r.stdout.strip().splitlines()[-1])
    assert got["codes"] == [-14, -2, -14, -2, -2, -2, -1, -2, -1]       # all refused on the host
    assert got["ranges"] == ["vitattn/" + n for n in (
        "vit_rope_freqs", "vit_qk_norm_rope", "vit_qk_norm_rope_ex", "vit_rope_table", "vit_varlen_attn",
        "vit_varlen_attn_lse", "vit_varlen_attn_fused_q", "vit_varlen_attn_padded", "vit_read_status")]
    assert got["pushes"] == got["pops"] == 9
    assert got["min_depth"] == 0                                          # no pop without its push
