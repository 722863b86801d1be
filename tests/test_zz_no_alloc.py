"""vit_varlen_attn_noalloc: the attention call for callers that cannot allocate
device memory (frozen memory pools, plugins that only receive input/output
pointers, C callers without an allocator). It is called here through the C ABI
and must give the same output as vit_varlen_attn with a caller workspace, on
two calls in a row that share the library's fixed scratch array.

Kept in its own file, named to be collected last."""
import ctypes

import pytest
import torch

import vision_encoder_varlen_gb300 as vit
from vision_encoder_varlen_gb300 import _build
from vision_encoder_varlen_gb300 import workloads as wl
from helpers import MAX_ABS, MEAN_ABS

pytestmark = pytest.mark.gpu

VIT_ERR_WORKSPACE_TOO_SMALL = -6
NOALLOC_BYTES = 4 << 20


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    lib = vit.lib()
    vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    lib.vit_varlen_attn_noalloc.argtypes = [vp, vp, vp, i64, i32, i32, i64, i64, i64, vp, i32, i32, f32, vp, i64,
                                            vp, vp]
    lib.vit_varlen_attn_noalloc.restype = i32
    return lib


def _call_noalloc(L, q, k, v, cu, max_seqlen, out, status):
    T, H, D = q.shape
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return L.vit_varlen_attn_noalloc(p(q), p(k), p(v), T, H, D, q.stride(0), k.stride(0), v.stride(0), p(cu),
                                     cu.numel() - 1, max_seqlen, 0.0, p(out), out.stride(0), p(status), stream)


def _case(lengths, H, D, seed):
    w = wl.from_lengths(lengths, H, D, seed=wl.SEED_BASE + seed, max_seqlen_meta=131072)
    t = w.tensors()
    return w, torch.from_numpy(w.cu_seqlens).cuda(), [t[n].cuda() for n in ("q", "k", "v")]


def test_noalloc_matches_workspace_call_on_two_calls_in_a_row(L):
    # two different problems back to back: the second call finds the first call's
    # work list still in the shared array and must not be affected by it
    cases = [([700, 5, 64, 2000, 129], 4, 80, 11), ([300, 1, 513], 2, 128, 12)]
    for lengths, H, D, seed in cases:
        w, cu, (q, k, v) = _case(lengths, H, D, seed)
        ref = vit.varlen_attn(q, k, v, cu, w.max_seqlen)
        out = torch.full_like(q, 5.0)
        status = vit.new_status()
        rc = _call_noalloc(L, q, k, v, cu, w.max_seqlen, out, status)
        assert rc == 0, vit.status_string(rc)
        assert vit.read_status(status) == 0
        err = (out.float() - ref.float()).abs()
        assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS, (lengths, err.max().item())


def test_noalloc_refuses_sizes_beyond_its_scratch(L):
    H, D, B = 16, 80, 8
    T = 1 << 21                                    # work list of ~524k items > 4 MiB
    assert vit.workspace_size(T, H, B, D) > NOALLOC_BYTES
    p = ctypes.c_void_p(16)
    cu = ctypes.c_void_p(16)
    rc = L.vit_varlen_attn_noalloc(p, p, p, T, H, D, H * D, H * D, H * D, cu, B, T, 0.0, p, H * D, None, None)
    assert rc == VIT_ERR_WORKSPACE_TOO_SMALL
