"""vit_varlen_attn_noalloc: the attention call for callers that cannot allocate
device memory (frozen memory pools, plugins that only receive input/output
pointers, C callers without an allocator). It is called here through the C ABI.

It runs the same scheduler and kernels as vit_varlen_attn, only on a work list
kept in the library's fixed device array, so its output must be bit-identical
to vit_varlen_attn with a caller workspace, on two calls in a row that share
that array; it is also held to the oracle. The calls must not allocate, and a
call that would have to look the array up while a stream is being captured is
refused rather than breaking the capture.

Kept in its own file, named to be collected last."""
import ctypes
import os
import subprocess
import sys
import textwrap

import pytest
import torch

import oracle
import vision_encoder_varlen_gb300 as vit
from vision_encoder_varlen_gb300 import _build
from vision_encoder_varlen_gb300 import workloads as wl
from helpers import assert_close

pytestmark = pytest.mark.gpu

VIT_ERR_WORKSPACE_TOO_SMALL = -6
VIT_ERR_BAD_ARGUMENT = -14
NOALLOC_BYTES = 4 << 20
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declare(lib):
    vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    lib.vit_varlen_attn_noalloc.argtypes = [vp, vp, vp, i64, i32, i32, i64, i64, i64, vp, i32, i32, f32, vp, i64,
                                            vp, vp]
    lib.vit_varlen_attn_noalloc.restype = i32
    return lib


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    return _declare(vit.lib())


def _call_noalloc(L, q, k, v, cu, max_seqlen, out, status, stream=None):
    T, H, D = q.shape
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    s = torch.cuda.current_stream() if stream is None else stream
    return L.vit_varlen_attn_noalloc(p(q), p(k), p(v), T, H, D, q.stride(0), k.stride(0), v.stride(0), p(cu),
                                     cu.numel() - 1, max_seqlen, 0.0, p(out), out.stride(0),
                                     None if status is None else p(status), ctypes.c_void_p(s.cuda_stream))


def _case(lengths, H, D, seed):
    w = wl.from_lengths(lengths, H, D, seed=wl.SEED_BASE + seed, max_seqlen_meta=131072)
    t = w.tensors()
    return w, t, torch.from_numpy(w.cu_seqlens).cuda(), [t[n].cuda() for n in ("q", "k", "v")]


def _free_device_bytes():
    free, _ = torch.cuda.mem_get_info()
    return free


def test_noalloc_matches_workspace_call_bitwise_on_two_calls_in_a_row(L):
    # two different problems back to back: the second call finds the first call's work list
    # still in the shared array and must not be affected by it
    cases = [([700, 5, 64, 2000, 129], 4, 80, 11), ([300, 1, 513], 2, 128, 12)]
    prepared = []
    for lengths, H, D, seed in cases:
        w, t, cu, (q, k, v) = _case(lengths, H, D, seed)
        ref = vit.varlen_attn(q, k, v, cu, w.max_seqlen)
        out = torch.full_like(q, 5.0)
        prepared.append((w, t, cu, q, k, v, ref, out, vit.new_status()))
    # the first call in a process looks the array up; with CUDA's lazy module loading that is also
    # when the array is placed in device memory (4 MiB), so the allocation check starts after it
    w0, _, cu0, (q0, k0, v0) = _case([100, 300], 2, 80, 10)
    assert _call_noalloc(L, q0, k0, v0, cu0, w0.max_seqlen, torch.empty_like(q0), None) == 0
    torch.cuda.synchronize()
    torch_before, free_before = torch.cuda.memory_allocated(), _free_device_bytes()
    for w, t, cu, q, k, v, ref, out, status in prepared:
        rc = _call_noalloc(L, q, k, v, cu, w.max_seqlen, out, status)
        assert rc == 0, vit.status_string(rc)
    torch.cuda.synchronize()
    # nothing was allocated by the calls: not through torch, not behind its back
    assert torch.cuda.memory_allocated() == torch_before
    assert _free_device_bytes() == free_before
    for w, t, cu, q, k, v, ref, out, status in prepared:
        assert vit.read_status(status) == 0
        assert torch.equal(out, ref), w.lengths
        exact = oracle.attention(*(oracle.widen(wl.bf16_bits(t[n])) for n in ("q", "k", "v")), w.cu_seqlens)
        assert_close(out, exact, what=f"noalloc {w.lengths.tolist()}")


def test_noalloc_replays_in_a_cuda_graph_after_its_first_call(L):
    w, t, cu, (q, k, v) = _case([400, 70, 1100], 4, 80, 13)
    ref = vit.varlen_attn(q, k, v, cu, w.max_seqlen)
    out = torch.zeros_like(q)
    assert _call_noalloc(L, q, k, v, cu, w.max_seqlen, out, None) == 0       # the lookup, outside capture
    torch.cuda.synchronize()
    out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        rc = _call_noalloc(L, q, k, v, cu, w.max_seqlen, out, None)
    assert rc == 0
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref)


def test_noalloc_refuses_the_first_lookup_during_capture():
    """In a fresh process the first call needs the array's address; made while its stream is
    being captured, it is refused and the capture itself stays valid."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    script = textwrap.dedent(f"""
        import ctypes, sys, torch
        sys.path.insert(0, {ROOT!r}); sys.path.insert(0, {os.path.join(ROOT, "tests")!r})
        import vision_encoder_varlen_gb300 as vit
        import test_zz_no_alloc as t
        L = t._declare(vit.lib())
        q = torch.zeros((256, 2, 80), dtype=torch.bfloat16, device="cuda")
        cu = torch.tensor([0, 256], dtype=torch.int32, device="cuda")
        out = torch.empty_like(q)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            rc = t._call_noalloc(L, q, q, q, cu, 256, out, None)
        g.replay()
        torch.cuda.synchronize()
        rc2 = t._call_noalloc(L, q, q, q, cu, 256, out, None)     # outside capture: looks it up
        torch.cuda.synchronize()
        print(rc, rc2)
    """)
    r = subprocess.run([sys.executable, "-c", script], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.split() == [str(VIT_ERR_BAD_ARGUMENT), "0"], r.stdout


def test_noalloc_refuses_sizes_beyond_its_scratch(L):
    H, D, B = 16, 80, 8
    T = 1 << 21                                    # work list of ~524k items > 4 MiB
    assert vit.workspace_size(T, H, B, D) > NOALLOC_BYTES
    p = ctypes.c_void_p(16)
    cu = ctypes.c_void_p(16)
    rc = L.vit_varlen_attn_noalloc(p, p, p, T, H, D, H * D, H * D, H * D, cu, B, T, 0.0, p, H * D, None, None)
    assert rc == VIT_ERR_WORKSPACE_TOO_SMALL
    # the other arguments are checked first, as vit_varlen_attn checks them
    rc = L.vit_varlen_attn_noalloc(p, p, p, T, H, 81, H * D, H * D, H * D, cu, B, T, 0.0, p, H * D, None, None)
    assert rc == -2
