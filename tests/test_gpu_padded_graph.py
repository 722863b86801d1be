"""GPU checks of the padded layout (per-segment start and real length, padding
rows between segments that nothing reads into a result or writes), of segment
isolation against non-finite values outside a segment, and of CUDA-graph
capture: one graph captured for a bucket of sizes, replayed after new starts
and lengths are written on the device."""
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
NAN_BF16 = 0x7FC0
SENTINEL = 0x1234


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


def _layout(lengths, align=128, gap=5):
    """starts of segments padded up to `align` rows plus `gap` rows of padding after each"""
    starts, t = [], 3                                  # leading padding too
    for L in lengths:
        starts.append(t)
        t += (L + align - 1) // align * align + gap
    return np.array(starts, dtype=np.int32), np.array(lengths, dtype=np.int32), t


def _padded_inputs(lengths, H, D, seed, pad_value=NAN_BF16):
    starts, lens, T = _layout(lengths)
    g = torch.Generator().manual_seed(seed)
    qkv = [torch.randn((T, H, D), generator=g).to(torch.bfloat16) for _ in range(3)]
    pad = np.ones(T, dtype=bool)
    for a, L in zip(starts, lens):
        pad[a:a + L] = False
    for t in qkv:
        t.view(torch.int16)[torch.from_numpy(pad)] = np.int16(pad_value)
    return starts, lens, T, qkv, pad


def _oracle_padded(qkv, starts, lens, scale=None):
    rows = np.concatenate([np.arange(a, a + L) for a, L in zip(starts, lens)]) if len(lens) else np.zeros(0, int)
    cu = np.zeros(len(lens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lens)
    widened = [oracle.widen(wl.bf16_bits(t))[rows] for t in qkv]
    out, lse = oracle.attention(*widened, cu, scale=scale, return_lse=True)
    return rows, out, lse


@pytest.mark.parametrize("lengths,H,D", [
    ([130, 0, 64, 1, 300, 17, 257], 2, 80),
    ([513, 100, 128], 2, 128),
    ([40, 41, 1000], 3, 64),
    ([9, 600, 200], 2, 96),
    ([64, 3, 100], 4, 32),
])
def test_padded_layout_parity_and_padding_untouched(lengths, H, D, split):
    starts, lens, T, qkv, pad = _padded_inputs(lengths, H, D, seed=sum(lengths) + D)
    q, k, v = (t.cuda() for t in qkv)
    out = torch.full((T, H, D), 0, dtype=torch.int16, device="cuda").fill_(SENTINEL).view(torch.bfloat16)
    lse = torch.full((T, H), -7.0, device="cuda")
    status = vit.new_status()
    vit.varlen_attn_padded(q, k, v, torch.from_numpy(starts).cuda(), torch.from_numpy(lens).cuda(), 4096,
                           out=out, lse=lse, status=status)
    assert vit.read_status(status) == 0
    rows, ref, ref_lse = _oracle_padded(qkv, starts, lens)
    idx = torch.from_numpy(rows).cuda()
    assert_close(out[idx], ref, what=f"padded {lengths}")
    g = lse[idx].cpu().numpy().astype(np.float64)
    assert np.max(np.abs(g - ref_lse)) <= 1e-3
    # padding rows: neither results nor lse were written
    pad_idx = torch.from_numpy(np.nonzero(pad)[0]).cuda()
    assert torch.all(out[pad_idx].view(torch.int16) == SENTINEL)
    assert torch.all(lse[pad_idx] == -7.0)


def test_padded_equals_packed_bitwise(split):
    lengths, H, D = [300, 1, 257, 64, 65, 129], 2, 80
    starts, lens, T, qkv, _ = _padded_inputs(lengths, H, D, seed=3)
    q, k, v = (t.cuda() for t in qkv)
    out = vit.varlen_attn_padded(q, k, v, torch.from_numpy(starts).cuda(), torch.from_numpy(lens).cuda(), 512)
    rows = np.concatenate([np.arange(a, a + L) for a, L in zip(starts, lens)])
    idx = torch.from_numpy(rows).cuda()
    cu = torch.from_numpy(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)).cuda()
    packed = vit.varlen_attn(q[idx].contiguous(), k[idx].contiguous(), v[idx].contiguous(), cu, 512)
    assert torch.equal(out[idx], packed)


@pytest.mark.parametrize("which", ["v", "k", "q"])
def test_non_finite_neighbour_does_not_leak(which, split):
    # contiguous packing: Inf/NaN in the middle segment must not reach the other two
    w = wl.from_lengths([300, 200, 129], 2, 80)
    t = w.tensors()
    q, k, v = (t[n].cuda() for n in ("q", "k", "v"))
    cu = torch.from_numpy(w.cu_seqlens).cuda()
    base = vit.varlen_attn(q, k, v, cu, w.max_seqlen)
    bad = {"q": q.clone(), "k": k.clone(), "v": v.clone()}
    seg = bad[which][300:500].view(torch.int16)
    seg[::2] = np.int16(NAN_BF16)
    seg[1::2] = np.int16(0x7F80)                         # +Inf
    out = vit.varlen_attn(bad["q"], bad["k"], bad["v"], cu, w.max_seqlen)
    keep = torch.cat([torch.arange(0, 300), torch.arange(500, 629)]).cuda()
    assert torch.equal(out[keep], base[keep])


def test_graph_capture_and_replay_with_new_lengths():
    H, D, T, B = 2, 80, 4096, 6
    g = torch.Generator().manual_seed(11)
    q, k, v = (torch.randn((T, H, D), generator=g).to(torch.bfloat16).cuda() for _ in range(3))
    starts = torch.zeros(B, dtype=torch.int32, device="cuda")
    lens = torch.zeros(B, dtype=torch.int32, device="cuda")
    out = torch.zeros((T, H, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((T, H), dtype=torch.float32, device="cuda")
    ws = torch.empty(vit.workspace_size(T, H, B, D), dtype=torch.uint8, device="cuda")
    status = vit.new_status()

    def set_layout(lengths):
        st, ln, _ = _layout(lengths, align=256, gap=7)
        starts.copy_(torch.from_numpy(st))
        lens.copy_(torch.from_numpy(ln))
        return st, ln

    def call():
        vit.varlen_attn_padded(q, k, v, starts, lens, 1024, out=out, lse=lse, workspace=ws, status=status)

    layout_a = [300, 17, 256, 1, 600, 90]
    layout_b = [5, 700, 0, 129, 64, 400]
    set_layout(layout_a)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):                         # warm-up outside the capture
        call()
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    for lengths in (layout_a, layout_b, layout_a):
        st, ln = set_layout(lengths)
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert vit.read_status(status) == 0
        got, got_lse = out.clone(), lse.clone()
        out.zero_()
        call()                                         # the same call, eagerly
        torch.cuda.synchronize()
        rows = np.concatenate([np.arange(a, a + L) for a, L in zip(st, ln)])
        idx = torch.from_numpy(rows).cuda()
        assert torch.equal(got[idx], out[idx]) and torch.equal(got_lse[idx], lse[idx])
        # and against the oracle
        cu = np.zeros(B + 1, dtype=np.int32)
        cu[1:] = np.cumsum(ln)
        ref = oracle.attention(*(oracle.widen(wl.bf16_bits(t.cpu()))[rows] for t in (q, k, v)), cu)
        assert_close(got[idx], ref, what=f"graph replay {lengths}")


@pytest.mark.parametrize("starts,lens,code", [
    ([0, 100], [120, 50], -10),        # overlap
    ([0, 4000], [10, 200], -10),       # past T
    ([-1, 100], [10, 10], -10),        # negative start
    ([0, 100], [10, -3], -10),         # negative length
    ([0, 1000], [10, 900], -11),       # longer than max_seqlen
])
def test_padded_layout_validation(starts, lens, code):
    H, D, T = 2, 80, 4096
    q = torch.randn((T, H, D)).to(torch.bfloat16).cuda()
    out = torch.full((T, H, D), 0, dtype=torch.int16, device="cuda").fill_(SENTINEL).view(torch.bfloat16)
    status = vit.new_status()
    vit.varlen_attn_padded(q, q, q, torch.tensor(starts, dtype=torch.int32).cuda(),
                           torch.tensor(lens, dtype=torch.int32).cuda(), 512, out=out, status=status)
    assert vit.read_status(status) == code
    assert torch.all(out.view(torch.int16) == SENTINEL)


def test_padded_empty_batch_is_a_no_op():
    q = torch.randn((64, 2, 80)).to(torch.bfloat16).cuda()
    out = torch.zeros_like(q)
    e = torch.zeros(0, dtype=torch.int32, device="cuda")
    vit.varlen_attn_padded(q, q, q, e, e, 64, out=out)
    assert torch.count_nonzero(out.float()) == 0
