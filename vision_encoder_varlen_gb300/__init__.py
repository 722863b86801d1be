"""GB300 (sm_103a) varlen ViT encoder attention: thin Python binding of libvitattn.

Argument marshalling only: every step runs in the library's CUDA kernels,
reached through its C ABI (include/vit_attn.h). PyTorch provides device
memory and the current stream. There is no CPU or eager fallback: if the
library is not built, every call raises.

    inv_freq, pos_hw, cu = rope_freqs(grid_hw, T, head_dim)       # 2D RoPE table + positions
    qk_norm_rope(q, k, pos_hw, inv_freq, norm_w, eps, inplace=True)
    out = varlen_attn(q, k, v, cu, max_seqlen)                    # [T, H, D] bf16
"""
from __future__ import annotations

import contextlib
import ctypes
import math
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libvitattn.so")
MAX_SEGMENTS = 8192
HEAD_DIMS = (32, 64, 80, 96, 128)

_lock = threading.Lock()
_lib = None


class VitError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {status_string(code)} (status {code})")


class _QRope(ctypes.Structure):
    _fields_ = [("pos_hw", ctypes.c_void_p), ("cos_sin", ctypes.c_void_p), ("max_pos", ctypes.c_int),
                ("norm_w", ctypes.c_void_p), ("eps", ctypes.c_float), ("rope_mode", ctypes.c_int)]


class _AttnOptions(ctypes.Structure):
    _fields_ = [("short_segment_max", ctypes.c_int)]


class _KernelTime(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char_p), ("launches", ctypes.c_int64), ("total_ms", ctypes.c_double)]


def lib() -> ctypes.CDLL:
    """The loaded libvitattn (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; "
                                   "g.build()'` (needs nvcc); there is no fallback implementation")
            L = ctypes.CDLL(LIB_PATH)
            vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
            L.vit_version.restype = ctypes.c_char_p
            L.vit_status_string.restype = ctypes.c_char_p
            L.vit_status_string.argtypes = [i32]
            L.vit_device_supported.argtypes = [i32]
            L.vit_rope_freqs.argtypes = [i32, f32, vp, i32, i64, vp, vp, vp, vp, vp]
            L.vit_qk_norm_rope.argtypes = [vp, vp, vp, vp, i64, i32, i32, i64, i64, i64, i64, vp, vp, vp, f32, vp]
            L.vit_qk_norm_rope_ex.argtypes = [vp, vp, vp, vp, i64, i32, i32, i64, i64, i64, i64, vp, vp, vp, f32,
                                              i32, vp, vp]
            L.vit_varlen_attn_workspace_size.restype = sz
            L.vit_varlen_attn_workspace_size.argtypes = [i64, i32, i32, i32]
            L.vit_varlen_attn.argtypes = [vp, vp, vp, i64, i32, i32, i64, i64, i64, vp, i32, i32, f32, vp, i64, vp,
                                          sz, vp, vp]
            L.vit_varlen_attn_lse.argtypes = [vp, vp, vp, i64, i32, i32, i64, i64, i64, vp, i32, i32, f32, vp, i64,
                                              vp, vp, sz, vp, vp]
            L.vit_varlen_attn_fused_q.argtypes = [vp, vp, vp, i64, i32, i32, i64, i64, i64, ctypes.POINTER(_QRope),
                                                  vp, i32, i32, f32, vp, i64, vp, vp, sz, vp, vp]
            L.vit_rope_table.argtypes = [vp, i32, i32, vp, vp]
            L.vit_varlen_attn_padded.argtypes = [vp, vp, vp, i64, i32, i32, i64, i64, i64, vp, vp, i32, i32, f32, vp,
                                                 i64, vp, ctypes.POINTER(_QRope), vp, sz, vp, vp]
            L.vit_varlen_attn_ex.argtypes = [vp, vp, vp, i64, i32, i32, i64, i64, i64, vp, vp, vp, i32, i32, f32, vp,
                                             i64, vp, ctypes.POINTER(_QRope), ctypes.POINTER(_AttnOptions), vp, sz,
                                             vp, vp]
            L.vit_read_status.argtypes = [vp, vp]
            L.vit_launch_count.restype = i64
            L.vit_kernel_timing.argtypes = [i32]
            L.vit_kernel_timing_read.argtypes = [ctypes.POINTER(_KernelTime), i32]
            for fn in ("vit_device_supported", "vit_rope_freqs", "vit_qk_norm_rope", "vit_qk_norm_rope_ex",
                       "vit_varlen_attn", "vit_varlen_attn_lse", "vit_varlen_attn_fused_q", "vit_rope_table",
                       "vit_varlen_attn_padded", "vit_varlen_attn_ex",
                       "vit_read_status", "vit_kernel_timing", "vit_kernel_timing_read"):
                getattr(L, fn).restype = i32
            _lib = L
    return _lib


_tls = threading.local()


@contextlib.contextmanager
def kernel_split(short_max: int | None):
    """Within the block, attention calls made by this thread pass ``short_max`` as their kernel
    split (segments longer than min(short_max, 64) run on the tcgen05 kernel, the others on the
    tiny-segment kernel); None restores the library default.
    Per thread, and passed with every call: the library itself keeps no setting between calls."""
    prev = getattr(_tls, "short_max", None)
    _tls.short_max = None if short_max is None else int(short_max)
    try:
        yield
    finally:
        _tls.short_max = prev


def _split(short_max):
    return short_max if short_max is not None else getattr(_tls, "short_max", None)


def status_string(code: int) -> str:
    return lib().vit_status_string(int(code)).decode()


def version() -> str:
    return lib().vit_version().decode()


def _check(code: int, what: str):
    if code != 0:
        raise VitError(code, what)


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _tok_stride(t: torch.Tensor, name: str, H: int, D: int) -> int:
    if t.dim() != 3 or t.shape[1] != H or t.shape[2] != D:
        raise ValueError(f"{name} must be [T, {H}, {D}], got {tuple(t.shape)}")
    if t.dtype != torch.bfloat16 or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA bfloat16 tensor")
    if t.stride(2) != 1 or t.stride(1) != D:
        raise ValueError(f"{name} needs head stride D and unit element stride (got strides {t.stride()})")
    return t.stride(0)


def new_status(device=None) -> torch.Tensor:
    """A zeroed device status word for the device-detected errors of the calls."""
    return torch.zeros(1, dtype=torch.int32, device=device or "cuda")


def read_status(status: torch.Tensor, stream=None) -> int:
    """Synchronise the stream and return the status word (0 = ok)."""
    code = lib().vit_read_status(_ptr(status), _stream(stream))
    return int(code)


def rope_freqs(grid_hw: torch.Tensor, total_tokens: int, head_dim: int, theta: float = 10000.0, *,
               status: torch.Tensor | None = None, stream=None):
    """2D RoPE frequency table (dim = head_dim/2), per-token (row, col) and cu_seqlens from a device grid list."""
    if grid_hw.dtype != torch.int32 or not grid_hw.is_cuda or not grid_hw.is_contiguous():
        raise ValueError("grid_hw must be a contiguous CUDA int32 tensor [n_img, 2]")
    n = grid_hw.numel() // 2
    dev = grid_hw.device
    dim = head_dim // 2
    inv_freq = torch.empty(dim // 2, dtype=torch.float32, device=dev)
    pos = torch.empty((total_tokens, 2), dtype=torch.int32, device=dev)
    cu = torch.empty(n + 1, dtype=torch.int32, device=dev)
    _check(lib().vit_rope_freqs(dim, float(theta), _ptr(grid_hw), n, int(total_tokens), _ptr(inv_freq), _ptr(pos),
                                _ptr(cu), _ptr(status), _stream(stream)), "vit_rope_freqs")
    return inv_freq, pos, cu


def rope_table(inv_freq: torch.Tensor, head_dim: int, max_pos: int, *, stream=None) -> torch.Tensor:
    """cos/sin of p * inv_freq for positions p < max_pos (fp32 [max_pos, head_dim/2]), the table the
    fused-Q attention rotates with."""
    if inv_freq.dtype != torch.float32 or not inv_freq.is_cuda or inv_freq.numel() != head_dim // 4:
        raise ValueError(f"inv_freq must be a CUDA float32 tensor [{head_dim // 4}]")
    cs = torch.empty((int(max_pos), head_dim // 2), dtype=torch.float32, device=inv_freq.device)
    _check(lib().vit_rope_table(_ptr(inv_freq), int(head_dim), int(max_pos), _ptr(cs), _stream(stream)),
           "vit_rope_table")
    return cs


ROPE_ROTATE_HALF = 0    # pairs (m, m + D/2)
ROPE_INTERLEAVED = 1    # pairs (2m, 2m + 1), the "complex_rope" mode


def qk_norm_rope(q: torch.Tensor | None, k: torch.Tensor | None, pos_hw: torch.Tensor, inv_freq: torch.Tensor,
                 norm_w: torch.Tensor | None = None, eps: float = 1e-6, *, q_out: torch.Tensor | None = None,
                 k_out: torch.Tensor | None = None, inplace: bool = False, interleaved: bool = False,
                 status: torch.Tensor | None = None, stream=None):
    """QK-RMSNorm (if norm_w [2, D] is given) + 2D RoPE. Returns (q', k'); a half passed as None is
    skipped and returned as None. ``interleaved`` rotates adjacent pairs instead of (m, m + D/2)."""
    ref = q if q is not None else k
    if ref is None:
        raise ValueError("at least one of q and k is required")
    T, H, D = ref.shape
    qs = _tok_stride(q, "q", H, D) if q is not None else 0
    ks = _tok_stride(k, "k", H, D) if k is not None else 0
    if q is not None and k is not None and q.shape[0] != k.shape[0]:
        raise ValueError("q and k must have the same number of tokens")
    if inplace:
        q_out, k_out = q, k
    if q is not None and q_out is None:
        q_out = torch.empty((T, H, D), dtype=q.dtype, device=q.device)
    if k is not None and k_out is None:
        k_out = torch.empty((T, H, D), dtype=k.dtype, device=k.device)
    if q is None:
        q_out = None
    if k is None:
        k_out = None
    qos = _tok_stride(q_out, "q_out", H, D) if q_out is not None else 0
    kos = _tok_stride(k_out, "k_out", H, D) if k_out is not None else 0
    if norm_w is not None and (norm_w.dtype != torch.bfloat16 or norm_w.numel() != 2 * D
                               or not norm_w.is_contiguous()):
        raise ValueError("norm_w must be a contiguous bfloat16 tensor [2, D]")
    mode = ROPE_INTERLEAVED if interleaved else ROPE_ROTATE_HALF
    _check(lib().vit_qk_norm_rope_ex(_ptr(q), _ptr(q_out), _ptr(k), _ptr(k_out), T, H, D, qs, qos, ks, kos,
                                     _ptr(pos_hw), _ptr(inv_freq), _ptr(norm_w), float(eps), mode, _ptr(status),
                                     _stream(stream)),
           "vit_qk_norm_rope_ex")
    return q_out, k_out


def workspace_size(T: int, H: int, B: int, D: int) -> int:
    return int(lib().vit_varlen_attn_workspace_size(int(T), int(H), int(B), int(D)))


def _max_seqlen(m) -> int:
    """The C convention: 0 = not given (the library bounds the segments by T)."""
    return 0 if m is None else int(m)


def _attn_ex(q, k, v, qs, ks, vs, cu_seqlens, seq_start, seq_len, B, max_seqlen, scale, out, os_, lse, qr,
             short_max, workspace, status, stream, what):
    opts = _AttnOptions(int(short_max))
    _check(lib().vit_varlen_attn_ex(_ptr(q), _ptr(k), _ptr(v), q.shape[0], q.shape[1], q.shape[2], qs, ks, vs,
                                    _ptr(cu_seqlens), _ptr(seq_start), _ptr(seq_len), B, _max_seqlen(max_seqlen),
                                    float(scale) if scale is not None else 0.0, _ptr(out), os_, _ptr(lse),
                                    ctypes.byref(qr) if qr is not None else None, ctypes.byref(opts),
                                    _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(status),
                                    _stream(stream)), what)


def varlen_attn(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_seqlens: torch.Tensor | None,
                max_seqlen: int | None = None, scale: float | None = None, *, num_segments: int | None = None,
                out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                status: torch.Tensor | None = None, return_lse: bool = False, lse: torch.Tensor | None = None,
                short_max: int | None = None, stream=None):
    """Non-causal attention inside each packed segment. q, k, v [T, H, D] bf16 -> out [T, H, D] bf16.

    ``max_seqlen`` bounds the segment lengths (a padded bucket is fine); None leaves the bound
    to the library (T), so nothing is read back to the host. With ``return_lse`` (or an ``lse``
    buffer) also returns lse [T, H] fp32, the natural-log sum of exp(scale * q.k) over each
    row's segment: (out, lse). ``short_max`` is this call's kernel split (see kernel_split)."""
    T, H, D = q.shape
    qs, ks, vs = _tok_stride(q, "q", H, D), _tok_stride(k, "k", H, D), _tok_stride(v, "v", H, D)
    if cu_seqlens is not None:
        if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda or not cu_seqlens.is_contiguous():
            raise ValueError("cu_seqlens must be a contiguous CUDA int32 tensor [B + 1]")
        B = cu_seqlens.numel() - 1
    else:
        if num_segments is None:
            raise ValueError("num_segments is required when cu_seqlens is None")
        B = int(num_segments)
    if out is None:
        out = torch.empty((T, H, D), dtype=q.dtype, device=q.device)
    os_ = _tok_stride(out, "out", H, D)
    need = workspace_size(T, H, B, D)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    sc = float(scale) if scale is not None else 0.0
    ws_bytes = workspace.numel() * workspace.element_size()
    short_max = _split(short_max)
    if return_lse and lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=q.device)
    if lse is not None and (lse.dtype != torch.float32 or tuple(lse.shape) != (T, H) or not lse.is_contiguous()
                            or not lse.is_cuda):
        raise ValueError(f"lse must be a contiguous CUDA float32 tensor [{T}, {H}]")
    if short_max is not None:
        _attn_ex(q, k, v, qs, ks, vs, cu_seqlens, None, None, B, max_seqlen, scale, out, os_, lse, None, short_max,
                 workspace, status, stream, "vit_varlen_attn_ex")
        return (out, lse) if lse is not None else out
    if lse is None:
        _check(lib().vit_varlen_attn(_ptr(q), _ptr(k), _ptr(v), T, H, D, qs, ks, vs, _ptr(cu_seqlens), B,
                                     _max_seqlen(max_seqlen), sc, _ptr(out), os_, _ptr(workspace), ws_bytes,
                                     _ptr(status), _stream(stream)), "vit_varlen_attn")
        return out
    _check(lib().vit_varlen_attn_lse(_ptr(q), _ptr(k), _ptr(v), T, H, D, qs, ks, vs, _ptr(cu_seqlens), B,
                                     _max_seqlen(max_seqlen), sc, _ptr(out), os_, _ptr(lse), _ptr(workspace), ws_bytes,
                                     _ptr(status), _stream(stream)), "vit_varlen_attn_lse")
    return out, lse


def varlen_attn_fused_q(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_seqlens: torch.Tensor | None,
                        max_seqlen: int | None, pos_hw: torch.Tensor, cos_sin: torch.Tensor,
                        q_norm_w: torch.Tensor | None = None, eps: float = 1e-6, scale: float | None = None, *,
                        interleaved: bool = False, num_segments: int | None = None,
                        out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                        status: torch.Tensor | None = None, return_lse: bool = False,
                        lse: torch.Tensor | None = None, short_max: int | None = None, stream=None):
    """varlen_attn on raw q: the kernels normalise (q_norm_w [D], or None) and rotate every Q tile
    after loading it. k must already be normalised and rotated (qk_norm_rope(None, k, ...))."""
    T, H, D = q.shape
    qs, ks, vs = _tok_stride(q, "q", H, D), _tok_stride(k, "k", H, D), _tok_stride(v, "v", H, D)
    if cu_seqlens is not None:
        if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda or not cu_seqlens.is_contiguous():
            raise ValueError("cu_seqlens must be a contiguous CUDA int32 tensor [B + 1]")
        B = cu_seqlens.numel() - 1
    else:
        if num_segments is None:
            raise ValueError("num_segments is required when cu_seqlens is None")
        B = int(num_segments)
    if cos_sin.dtype != torch.float32 or cos_sin.dim() != 2 or cos_sin.shape[1] != D // 2 \
            or not cos_sin.is_contiguous():
        raise ValueError(f"cos_sin must be the contiguous float32 [max_pos, {D // 2}] table of rope_table")
    if q_norm_w is not None and (q_norm_w.dtype != torch.bfloat16 or q_norm_w.numel() != D
                                 or not q_norm_w.is_contiguous()):
        raise ValueError("q_norm_w must be a contiguous bfloat16 tensor [D]")
    if out is None:
        out = torch.empty((T, H, D), dtype=q.dtype, device=q.device)
    os_ = _tok_stride(out, "out", H, D)
    if workspace is None:
        workspace = torch.empty(max(workspace_size(T, H, B, D), 16), dtype=torch.uint8, device=q.device)
    if return_lse and lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=q.device)
    if lse is not None and (lse.dtype != torch.float32 or tuple(lse.shape) != (T, H) or not lse.is_contiguous()):
        raise ValueError(f"lse must be a contiguous CUDA float32 tensor [{T}, {H}]")
    qr = _QRope(pos_hw.data_ptr(), cos_sin.data_ptr(), int(cos_sin.shape[0]),
                q_norm_w.data_ptr() if q_norm_w is not None else None, float(eps),
                ROPE_INTERLEAVED if interleaved else ROPE_ROTATE_HALF)
    short_max = _split(short_max)
    if short_max is not None:
        _attn_ex(q, k, v, qs, ks, vs, cu_seqlens, None, None, B, max_seqlen, scale, out, os_, lse, qr, short_max,
                 workspace, status, stream, "vit_varlen_attn_ex")
        return (out, lse) if lse is not None else out
    _check(lib().vit_varlen_attn_fused_q(_ptr(q), _ptr(k), _ptr(v), T, H, D, qs, ks, vs, ctypes.byref(qr),
                                         _ptr(cu_seqlens), B, _max_seqlen(max_seqlen),
                                         float(scale) if scale is not None else 0.0, _ptr(out), os_, _ptr(lse),
                                         _ptr(workspace), workspace.numel() * workspace.element_size(),
                                         _ptr(status), _stream(stream)), "vit_varlen_attn_fused_q")
    return (out, lse) if lse is not None else out


def varlen_attn_padded(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, seq_start: torch.Tensor,
                       seq_len: torch.Tensor, max_seqlen: int | None = None, scale: float | None = None, *,
                       out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                       status: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                       short_max: int | None = None, stream=None):
    """Attention over a padded layout: segment i is rows [seq_start[i], seq_start[i] + seq_len[i]) of
    q, k, v and out (ascending, not overlapping); rows between segments are left untouched. Nothing
    on the host depends on the lengths, so the call can be captured in a CUDA graph and replayed
    after new starts/lengths are written into the same device tensors."""
    T, H, D = q.shape
    qs, ks, vs = _tok_stride(q, "q", H, D), _tok_stride(k, "k", H, D), _tok_stride(v, "v", H, D)
    for name, t in (("seq_start", seq_start), ("seq_len", seq_len)):
        if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA int32 tensor [B]")
    B = seq_len.numel()
    if seq_start.numel() != B:
        raise ValueError("seq_start and seq_len must have the same length")
    if out is None:
        out = torch.empty((T, H, D), dtype=q.dtype, device=q.device)
    os_ = _tok_stride(out, "out", H, D)
    if workspace is None:
        workspace = torch.empty(max(workspace_size(T, H, B, D), 16), dtype=torch.uint8, device=q.device)
    if lse is not None and (lse.dtype != torch.float32 or tuple(lse.shape) != (T, H) or not lse.is_contiguous()):
        raise ValueError(f"lse must be a contiguous CUDA float32 tensor [{T}, {H}]")
    short_max = _split(short_max)
    if short_max is not None:
        _attn_ex(q, k, v, qs, ks, vs, None, seq_start, seq_len, B, max_seqlen, scale, out, os_, lse, None, short_max,
                 workspace, status, stream, "vit_varlen_attn_ex")
        return out
    _check(lib().vit_varlen_attn_padded(_ptr(q), _ptr(k), _ptr(v), T, H, D, qs, ks, vs, _ptr(seq_start),
                                        _ptr(seq_len), B, _max_seqlen(max_seqlen),
                                        float(scale) if scale is not None else 0.0, _ptr(out), os_, _ptr(lse), None,
                                        _ptr(workspace),
                                        workspace.numel() * workspace.element_size(), _ptr(status), _stream(stream)),
           "vit_varlen_attn_padded")
    return out


def encoder_attn(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_seqlens: torch.Tensor,
                 max_seqlen: int | None,
                 pos_hw: torch.Tensor, inv_freq: torch.Tensor, cos_sin: torch.Tensor,
                 norm_w: torch.Tensor | None = None, eps: float = 1e-6, *, interleaved: bool = False,
                 k_out: torch.Tensor | None = None, **kw):
    """The whole hot path with the Q prologue fused into attention: a one-tensor K pre-stage
    (norm_w row 1, written to k_out, or in place when k_out is k), then attention on raw q with
    norm_w row 0 applied as Q tiles load."""
    _, kr = qk_norm_rope(None, k, pos_hw, inv_freq, norm_w, eps, k_out=k_out, interleaved=interleaved,
                         stream=kw.get("stream"))
    q_w = norm_w.reshape(2, -1)[0] if norm_w is not None else None
    return varlen_attn_fused_q(q, kr, v, cu_seqlens, max_seqlen, pos_hw, cos_sin, q_w, eps,
                               interleaved=interleaved, **kw)


DEFAULT_SHORT_MAX = 64   # the library's kernel split when a call passes none


def launch_count() -> int:
    return int(lib().vit_launch_count())


def kernel_timing(enable: bool) -> bool:
    return bool(lib().vit_kernel_timing(1 if enable else 0))


def kernel_timing_read(max_entries: int = 32) -> dict:
    """{kernel name: (launches, total ms)} for launches timed since the last read (synchronises)."""
    arr = (_KernelTime * max_entries)()
    n = lib().vit_kernel_timing_read(arr, max_entries)
    if n < 0:
        raise VitError(-8, "vit_kernel_timing_read")
    return {arr[i].name.decode(): (int(arr[i].launches), float(arr[i].total_ms)) for i in range(n)}


def default_scale(head_dim: int) -> float:
    return 1.0 / math.sqrt(head_dim)
