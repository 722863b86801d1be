"""GPU edge cases: bitwise segment isolation, determinism, strided and uniform
inputs, and device-detected errors that leave the outputs untouched."""
import numpy as np
import pytest
import torch

import oracle
import vision_encoder_varlen_gb300 as vit
from vision_encoder_varlen_gb300 import _build
from vision_encoder_varlen_gb300 import workloads as wl
from helpers import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()


# "default" passes no option (the plain entry points, the library's own split); the others pass
# their split with every call
SPLITS = {"default": None, "all_long": 0, "split_32": 32}


@pytest.fixture(params=list(SPLITS))
def split(request):
    with vit.kernel_split(SPLITS[request.param]):
        yield request.param


def _inputs(lengths, H, D, seed=0):
    w = wl.from_lengths(lengths, H, D, seed=wl.SEED_BASE + seed, max_seqlen_meta=131072)
    t = w.tensors()
    return w, t, torch.from_numpy(w.cu_seqlens).cuda(), [t[n].cuda() for n in ("q", "k", "v")]


@pytest.mark.parametrize("D", [80, 128])
def test_segment_isolation_bitwise(D, split):
    lengths = [130, 1, 700, 64, 255]
    w, t, cu, (q, k, v) = _inputs(lengths, 2, D)
    base = vit.varlen_attn(q, k, v, cu, w.max_seqlen).clone()
    cuh = w.cu_seqlens
    for seg in range(len(lengths)):
        a, b = int(cuh[seg]), int(cuh[seg + 1])
        q2, k2, v2 = q.clone(), k.clone(), v.clone()
        q2[a:b] = torch.randn_like(q2[a:b].float()).to(torch.bfloat16)
        k2[a:b] *= -2
        v2[a:b] += 1
        pert = vit.varlen_attn(q2, k2, v2, cu, w.max_seqlen)
        keep = torch.ones(w.total_tokens, dtype=torch.bool, device="cuda")
        keep[a:b] = False
        assert torch.equal(pert[keep].view(torch.int16), base[keep].view(torch.int16)), f"segment {seg} leaked"
        assert not torch.equal(pert[a:b], base[a:b])


def test_segment_isolation_bitwise_beside_a_65536_token_image(split):
    """The headline layout: one 256x256 image (65536 tokens) packed with short images, and
    max_seqlen padded to the 131072 bucket. Perturbing any one segment leaves every byte of
    every other segment's output unchanged, the long neighbour included."""
    lengths = [65536, 100, 1, 513, 64, 257]
    w, t, cu, (q, k, v) = _inputs(lengths, 2, 80, seed=9)
    assert w.max_seqlen == 131072
    base = vit.varlen_attn(q, k, v, cu, w.max_seqlen).clone()
    cuh = w.cu_seqlens
    for seg in (0, 1, 3, 5):
        a, b = int(cuh[seg]), int(cuh[seg + 1])
        q2, k2, v2 = q.clone(), k.clone(), v.clone()
        k2[a:b] *= -2
        v2[a:b] += 1
        pert = vit.varlen_attn(q2, k2, v2, cu, w.max_seqlen)
        keep = torch.ones(w.total_tokens, dtype=torch.bool, device="cuda")
        keep[a:b] = False
        assert torch.equal(pert[keep].view(torch.int16), base[keep].view(torch.int16)), f"segment {seg} leaked"
        assert not torch.equal(pert[a:b], base[a:b])


def test_deterministic_bitwise(split):
    w, t, cu, (q, k, v) = _inputs([3000, 17, 900], 4, 80, seed=3)
    ws = torch.empty(vit.workspace_size(w.total_tokens, 4, 3, 80), dtype=torch.uint8, device="cuda")
    a = vit.varlen_attn(q, k, v, cu, w.max_seqlen, workspace=ws).clone()
    for _ in range(3):
        b = vit.varlen_attn(q, k, v, cu, w.max_seqlen, workspace=ws)
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_strided_packed_qkv_and_strided_out(split):
    lengths = [100, 300]
    H, D = 3, 80
    w, t, cu, _ = _inputs(lengths, H, D, seed=4)
    T = w.total_tokens
    qkv = torch.stack([t["q"], t["k"], t["v"]], dim=1).cuda()        # [T, 3, H, D]
    q, k, v = qkv[:, 0], qkv[:, 1], qkv[:, 2]
    assert q.stride(0) == 3 * H * D
    big = torch.full((T, H + 2, D), 7.0, dtype=torch.bfloat16, device="cuda")
    out = big[:, 1:H + 1]                                             # token stride (H+2)*D, offset D
    vit.varlen_attn(q, k, v, cu, w.max_seqlen, out=out)
    ref = oracle.attention(*(oracle.widen(wl.bf16_bits(t[n])) for n in ("q", "k", "v")), w.cu_seqlens)
    assert_close(out, ref, what="strided")
    assert torch.all(big[:, 0] == 7.0) and torch.all(big[:, H + 1] == 7.0)


def test_uniform_segments_without_cu_seqlens(split):
    H, D, B, L = 2, 64, 4, 96
    w, t, cu, (q, k, v) = _inputs([L] * B, H, D, seed=5)
    out = vit.varlen_attn(q, k, v, None, L, num_segments=B)
    ref = oracle.attention(*(oracle.widen(wl.bf16_bits(t[n])) for n in ("q", "k", "v")), w.cu_seqlens)
    assert_close(out, ref, what="uniform")


def test_max_seqlen_not_given(split):
    # None (0 in the C ABI): T bounds the segments; the work items and so the results are those
    # of a call given the exact maximum, bit for bit, for packed, uniform and padded layouts
    lengths = [1, 300, 0, 64, 65, 129]
    w, t, cu, (q, k, v) = _inputs(lengths, 2, 80, seed=9)
    bits = lambda x: x.view(torch.int16)                 # noqa: E731
    status = vit.new_status()
    got = vit.varlen_attn(q, k, v, cu, None, status=status)
    assert vit.read_status(status) == 0
    assert torch.equal(bits(got), bits(vit.varlen_attn(q, k, v, cu, 300)))
    q4, k4, v4 = q[:120], k[:120], v[:120]
    assert torch.equal(bits(vit.varlen_attn(q4, k4, v4, None, None, num_segments=4)),
                       bits(vit.varlen_attn(q4, k4, v4, None, 30, num_segments=4)))
    start, length = cu[:-1].contiguous(), (cu[1:] - cu[:-1]).contiguous()
    assert torch.equal(bits(vit.varlen_attn_padded(q, k, v, start, length, None)), bits(got))


def test_in_place_prologue_matches_out_of_place():
    w = wl.make_config(3)
    t = w.tensors()
    grid = torch.from_numpy(w.grid_hw.copy()).cuda()
    inv_freq, pos, cu = vit.rope_freqs(grid, w.total_tokens, w.head_dim)
    q, k = t["q"].cuda(), t["k"].cuda()
    nw = t["norm_w"].cuda()
    qo, ko = vit.qk_norm_rope(q, k, pos, inv_freq, nw, w.eps)
    vit.qk_norm_rope(q, k, pos, inv_freq, nw, w.eps, inplace=True)
    assert torch.equal(qo.view(torch.int16), q.view(torch.int16))
    assert torch.equal(ko.view(torch.int16), k.view(torch.int16))


@pytest.mark.parametrize("cu_list,max_seqlen,code", [
    ([0, 10, 5, 20], 100, -10),      # decreasing
    ([1, 10, 20], 100, -10),         # does not start at 0
    ([0, 10, 19], 100, -10),         # does not end at T
    ([0, 10, 20], 9, -11),           # a segment longer than max_seqlen
])
def test_device_detected_bad_seqlens_leave_output_untouched(cu_list, max_seqlen, code, split):
    T, H, D = 20, 2, 80
    g = torch.Generator().manual_seed(0)
    q, k, v = (torch.randn(T, H, D, generator=g).to(torch.bfloat16).cuda() for _ in range(3))
    out = torch.full((T, H, D), 3.0, dtype=torch.bfloat16, device="cuda")
    status = vit.new_status()
    cu = torch.tensor(cu_list, dtype=torch.int32, device="cuda")
    vit.varlen_attn(q, k, v, cu, max_seqlen, out=out, status=status)
    assert vit.read_status(status) == code
    assert torch.all(out == 3.0)
    # a good call afterwards works again and does not clear the sticky error word
    good = torch.tensor([0, 10, 20], dtype=torch.int32, device="cuda")
    vit.varlen_attn(q, k, v, good, 10, out=out, status=status)
    assert vit.read_status(status) == code
    assert not torch.all(out == 3.0)


def test_grid_mismatch_detected_on_device():
    grid = torch.tensor([[4, 4], [2, 3]], dtype=torch.int32, device="cuda")
    status = vit.new_status()
    inv_freq, pos, cu = vit.rope_freqs(grid, 21, 80, status=status)   # 16 + 6 = 22 != 21
    assert vit.read_status(status) == -12
    grid_neg = torch.tensor([[4, -4]], dtype=torch.int32, device="cuda")
    status2 = vit.new_status()
    vit.rope_freqs(grid_neg, 0, 80, status=status2)
    assert vit.read_status(status2) == -12


def test_empty_inputs():
    H, D = 2, 80
    q = torch.empty((0, H, D), dtype=torch.bfloat16, device="cuda")
    cu = torch.zeros(3, dtype=torch.int32, device="cuda")
    status = vit.new_status()
    out = vit.varlen_attn(q, q, q, cu, 1, status=status)
    assert out.shape == (0, H, D) and vit.read_status(status) == 0
    grid = torch.zeros((2, 2), dtype=torch.int32, device="cuda")
    inv_freq, pos, cu2 = vit.rope_freqs(grid, 0, D, status=status)
    assert vit.read_status(status) == 0 and cu2.tolist() == [0, 0, 0]


def test_launches_are_counted_and_timed():
    w, t, cu, (q, k, v) = _inputs([500, 20], 2, 80, seed=6)
    n0 = vit.launch_count()
    vit.kernel_timing(True)
    try:
        vit.varlen_attn(q, k, v, cu, w.max_seqlen)
        rec = vit.kernel_timing_read()
    finally:
        vit.kernel_timing(False)
    assert vit.launch_count() - n0 >= 2
    assert "schedule" in rec and all(ms >= 0 for _, ms in rec.values())


_STALL_SCRIPT = """
import ctypes, json, sys
import numpy as np
import torch
sys.path[:0] = [{root!r}, {tests!r}]
import oracle
import vision_encoder_varlen_gb300 as vit
from vision_encoder_varlen_gb300 import workloads as wl
from helpers import assert_close
vit.LIB_PATH = {lib!r}                 # this process loads the test build only
L = vit.lib()
L.vit_debug_stall_long_kernel.argtypes = [ctypes.c_int]
L.vit_debug_stall_long_kernel.restype = ctypes.c_int
w = wl.from_lengths([600, 300], 2, 80, seed=wl.SEED_BASE + 7, max_seqlen_meta=131072)
t = w.tensors()
q, k, v = (t[n].cuda() for n in ("q", "k", "v"))
cu = torch.from_numpy(w.cu_seqlens).cuda()
vit.varlen_attn(q, k, v, cu, w.max_seqlen, short_max=0)      # every kernel loaded before the stall
torch.cuda.synchronize()
status = vit.new_status()
L.vit_debug_stall_long_kernel(1)
try:
    vit.varlen_attn(q, k, v, cu, w.max_seqlen, status=status, short_max=0)
    code = vit.read_status(status)
finally:
    L.vit_debug_stall_long_kernel(0)
status2 = vit.new_status()
out = vit.varlen_attn(q, k, v, cu, w.max_seqlen, status=status2, short_max=0)
code2 = vit.read_status(status2)
ref = oracle.attention(*(oracle.widen(wl.bf16_bits(t[n])) for n in ("q", "k", "v")), w.cu_seqlens)
mx, mean = assert_close(out, ref, what="after timeout")
print("RESULT " + json.dumps([code, code2, mx]))
"""


def test_long_kernel_bounded_wait_reports_timeout_and_context_survives():
    """A wait that can never complete (V is never loaded) must end in VIT_ERR_TIMEOUT within its
    clock budget; afterwards the same process computes correct results again. The hook exists
    only in a test build of the library (the release library exports no debug call), which a
    separate process loads alone; a first call there loads every kernel the stalled call uses."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    script = _STALL_SCRIPT.format(root=root, tests=os.path.join(root, "tests"), lib=_build.build_test_hooks())
    r = subprocess.run([sys.executable, "-c", script], capture_output=True, text=True, timeout=240)
    assert r.returncode == 0, r.stderr[-3000:]
    line = [x for x in r.stdout.splitlines() if x.startswith("RESULT ")][-1]
    code, code2, _ = __import__("json").loads(line[len("RESULT "):])
    assert code == -13 and code2 == 0


def test_threads_with_different_splits_get_their_own_results():
    """The kernel split is a per-call option: two host threads that keep issuing the same
    attention with different splits, on their own streams, each get exactly the bits their own
    split gives when run alone. The short segments run on the tiny kernel under one split and on
    the tcgen05 kernel under the other; their fp32 log-sum-exp rows differ between the two
    kernels (other summation orders), so a leaked setting shows."""
    import threading
    w, t, cu, (q, k, v) = _inputs([700, 40, 64, 300, 17, 129, 50], 8, 80, seed=8)
    splits = (0, 64)

    def call(sm):
        out, lse = vit.varlen_attn(q, k, v, cu, w.max_seqlen, short_max=sm, return_lse=True)
        return out, lse

    alone = {sm: call(sm) for sm in splits}
    torch.cuda.synchronize()
    assert not torch.equal(alone[0][1], alone[64][1])
    bad = []

    def worker(sm):
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            outs = [call(sm) for _ in range(30)]
        s.synchronize()
        bad.extend(sm for o, l in outs if not (torch.equal(o, alone[sm][0]) and torch.equal(l, alone[sm][1])))

    th = [threading.Thread(target=worker, args=(sm,)) for sm in splits]
    for x in th:
        x.start()
    for x in th:
        x.join()
    assert not bad
