"""fp64 CPU oracle for varlen ViT encoder attention (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package. The CUDA library never loads it and shares no
code with it. The arithmetic lives in ``vit_oracle.c`` (form B: one plain
softmax attention per packed segment, after RMSNorm and 2D RoPE) and in
``dense_ref.py`` (form A: one dense attention with a block-diagonal additive
mask); see those files for the passages each step follows. ``mimic.py`` repeats
the steps with the roundings of the pages' eager modules; it explains residuals
and never decides a pass or a failure.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "vit_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libvitoracle.so")
_lock = threading.Lock()
_lib = None

_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_i64p = np.ctypeslib.ndpointer(dtype=np.int64, flags="C_CONTIGUOUS")
_u16p = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")


# A prebuilt oracle library to load instead of building vit_oracle.c: the mutation test
# (tests/test_oracle_mutants.py) compiles deliberately broken copies of the source and runs
# the pins against each through this variable.
_OVERRIDE_ENV = "VIT_ORACLE_LIB_OVERRIDE"


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (OpenMP if available). Returns the .so path."""
    override = os.environ.get(_OVERRIDE_ENV)
    if override:
        return override
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.vo_num_threads.restype = ctypes.c_int
            lib.vo_rope_inv_freq.argtypes = [ctypes.c_int, ctypes.c_double, _f64p]
            lib.vo_rope_inv_freq.restype = None
            lib.vo_grid_positions.argtypes = [_i32p, ctypes.c_int, _i32p, ctypes.c_void_p]
            lib.vo_grid_positions.restype = ctypes.c_int64
            lib.vo_norm_rope.argtypes = [_u16p, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                                         _i32p, ctypes.c_double, ctypes.c_void_p, ctypes.c_int,
                                         ctypes.c_double, ctypes.c_int, _f64p]
            lib.vo_norm_rope.restype = None
            lib.vo_attention.argtypes = [_f64p, _f64p, _f64p, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                         _i32p, ctypes.c_int, ctypes.c_double, ctypes.c_void_p,
                                         ctypes.c_int64, _f64p, ctypes.c_void_p]
            lib.vo_attention.restype = None
            _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().vo_num_threads())


def widen(bits: np.ndarray) -> np.ndarray:
    """Exact bf16 -> fp64 of raw uint16 bit patterns."""
    u = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def rope_inv_freq(dim: int, theta: float = 10000.0) -> np.ndarray:
    """1/theta^(2j/dim), j < dim/2 (VisionRotaryEmbedding.__init__, vLLM Dots vision_attention page)."""
    out = np.zeros(max(dim // 2, 1), dtype=np.float64)
    _load().vo_rope_inv_freq(int(dim), float(theta), out)
    return out[: dim // 2]


def grid_positions(grid_hw) -> tuple[np.ndarray, np.ndarray]:
    """(cu_seqlens int32 [n+1], pos_hw int32 [T, 2]) for row-major tokens of each (h, w) image."""
    g = np.ascontiguousarray(np.asarray(grid_hw, dtype=np.int32).reshape(-1, 2))
    n = g.shape[0]
    T = int(np.sum(g[:, 0].astype(np.int64) * g[:, 1]))
    cu = np.zeros(n + 1, dtype=np.int32)
    pos = np.zeros((max(T, 1), 2), dtype=np.int32)
    got = _load().vo_grid_positions(g.reshape(-1), n, cu, pos.ctypes.data)
    assert got == T
    return cu, pos[:T]


def norm_rope(x_bits: np.ndarray, pos: np.ndarray, theta: float = 10000.0, w_bits: np.ndarray | None = None,
              use_norm: bool = False, eps: float = 1e-6, interleaved: bool = False) -> np.ndarray:
    """fp64 RMSNorm (optional) + 2D RoPE of bf16 rows x [T, H, D]: rotate-half pairs (m, m + D/2), or
    adjacent pairs (2m, 2m + 1) with ``interleaved`` (the "complex_rope" mode)."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    T, H, D = x.shape
    assert D % 4 == 0 and D <= 512
    out = np.zeros((T, H, D), dtype=np.float64)
    if T == 0:
        return out
    w = None if w_bits is None else np.ascontiguousarray(w_bits, dtype=np.uint16).reshape(D)
    _load().vo_norm_rope(x.reshape(-1), T, H, D, H * D, np.ascontiguousarray(pos, dtype=np.int32).reshape(-1),
                         float(theta), None if w is None else w.ctypes.data, int(bool(use_norm)), float(eps),
                         int(bool(interleaved)), out.reshape(-1))
    return out


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, cu_seqlens, scale: float | None = None,
              rows=None, return_lse: bool = False):
    """Per-segment softmax(scale q k^T) v in fp64; q, k, v fp64 [T, H, D].

    With ``return_lse`` also returns lse [n, H] = log sum_j exp(scale <q, k_j>) over each row's segment."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    T, H, D = q.shape
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    B = cu.shape[0] - 1
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    if rows is None:
        n, rows_arr = T, None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        n = rows_arr.shape[0]
    out = np.zeros((n, H, D), dtype=np.float64)
    lse = np.zeros((n, H), dtype=np.float64)
    if n == 0 or H == 0:
        return (out, lse) if return_lse else out
    _load().vo_attention(q.reshape(-1), k.reshape(-1), v.reshape(-1), T, H, D, cu, B, float(scale),
                         None if rows_arr is None else rows_arr.ctypes.data, n, out.reshape(-1),
                         lse.ctypes.data if return_lse else None)
    return (out, lse) if return_lse else out


def full_path(grid_hw, q_bits, k_bits, v_bits, norm_w_bits=None, eps: float = 1e-6, theta: float = 10000.0,
              scale: float | None = None, rows=None, interleaved: bool = False, return_lse: bool = False):
    """Positions from the grid, QK-RMSNorm (if weights given) + 2D RoPE, then per-segment attention."""
    cu, pos = grid_positions(grid_hw)
    use_norm = norm_w_bits is not None
    wq = None if norm_w_bits is None else np.asarray(norm_w_bits)[0]
    wk = None if norm_w_bits is None else np.asarray(norm_w_bits)[1]
    qr = norm_rope(q_bits, pos, theta, wq, use_norm, eps, interleaved)
    kr = norm_rope(k_bits, pos, theta, wk, use_norm, eps, interleaved)
    return attention(qr, kr, widen(v_bits), cu, scale, rows, return_lse)
