"""The device scheduler's work list, bit for bit against a host recomputation.

After a call, the workspace holds a 64-byte header (int32: long items, short
items, rows per long item, rows per short item, error, tiny items) and the
items (int4: segment start, segment length, first query row, head). The host
recomputes the same list from the segment lengths alone: segments longer than
the split go to the tcgen05 kernel in 256-row blocks, longest first (ties by
index); the rest in index order, those of at most min(split, 64) tokens last,
one item per head; heads outer, query blocks inner within a segment."""
import numpy as np
import pytest
import torch

import vision_encoder_varlen_gb300 as vit
from vision_encoder_varlen_gb300 import _build

pytestmark = pytest.mark.gpu

BM_LONG, BM_SHORT, TINY = 256, 128, 64


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()


def expected(lengths, starts, H, short_max):
    tiny_max = min(short_max, TINY)
    idx = range(len(lengths))
    long_s = sorted((i for i in idx if lengths[i] > short_max), key=lambda i: (-lengths[i], i))
    short_s = [i for i in idx if tiny_max < lengths[i] <= short_max]
    tiny_s = [i for i in idx if lengths[i] <= tiny_max]
    items, counts = [], []
    for group, bm in ((long_s, BM_LONG), (short_s, BM_SHORT), (tiny_s, BM_SHORT)):
        n0 = len(items)
        for seg in group:
            L, a = int(lengths[seg]), int(starts[seg])
            nq = (L + bm - 1) // bm
            for h in range(H):
                for qb in range(nq):
                    items.append((a, L, a + qb * bm, h))
        counts.append(len(items) - n0)
    return counts, np.array(items, dtype=np.int32).reshape(-1, 4)


def run(lengths, H, D, short_max, padded=False):
    lengths = np.asarray(lengths, dtype=np.int64)
    if padded:
        starts = np.zeros(len(lengths), dtype=np.int64)
        t = 5
        for i, L in enumerate(lengths):
            starts[i] = t
            t += L + 3
        T = int(t)
    else:
        starts = np.concatenate([[0], np.cumsum(lengths)[:-1]]).astype(np.int64)
        T = int(lengths.sum())
    B = len(lengths)
    q = torch.zeros((max(T, 1), H, D), dtype=torch.bfloat16, device="cuda")[:T]
    ws = torch.zeros(vit.workspace_size(T, H, B, D), dtype=torch.uint8, device="cuda")
    prev = vit.set_short_segment_max(short_max)
    try:
        status = vit.new_status()
        if padded:
            vit.varlen_attn_padded(q, q, q, torch.from_numpy(starts.astype(np.int32)).cuda(),
                                   torch.from_numpy(lengths.astype(np.int32)).cuda(), int(lengths.max()),
                                   workspace=ws, status=status)
        else:
            cu = torch.from_numpy(np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)).cuda()
            vit.varlen_attn(q, q, q, cu, max(int(lengths.max()), 1), workspace=ws, status=status)
        assert vit.read_status(status) == 0
    finally:
        vit.set_short_segment_max(prev)
    raw = ws.cpu().numpy()
    hdr = raw[:64].view(np.int32)
    return hdr, raw[64:].view(np.int32).reshape(-1, 4), starts


CASES = [
    ([300, 1, 0, 64, 65, 2000, 129, 128, 17, 0, 700], 3),
    ([5, 4096, 4096, 4095, 1], 2),
    ([64] * 50 + [65] * 7 + [1000] * 3, 1),
]


@pytest.mark.parametrize("padded", [False, True])
@pytest.mark.parametrize("short_max", [64, 0, 2 ** 31 - 1, 100])
@pytest.mark.parametrize("lengths,H", CASES)
def test_work_list_matches_host_recomputation(lengths, H, short_max, padded):
    hdr, items, starts = run(lengths, H, 80, short_max, padded)
    counts, ref = expected(np.asarray(lengths), starts, H, short_max)
    n = sum(counts)
    assert hdr[4] == 0                                     # no error
    assert (hdr[0], hdr[1], hdr[5]) == tuple(counts)
    assert (hdr[2], hdr[3]) == (BM_LONG, BM_SHORT)
    assert np.array_equal(items[:n], ref)


def test_work_list_many_segments():
    rng = np.random.default_rng(4)
    lengths = rng.integers(0, 300, size=3000)
    lengths[rng.choice(3000, 20, replace=False)] = rng.integers(1000, 5000, size=20)
    hdr, items, starts = run(lengths, 2, 64, 64)
    counts, ref = expected(lengths, starts, 2, 64)
    assert (hdr[0], hdr[1], hdr[5]) == tuple(counts)
    assert np.array_equal(items[:sum(counts)], ref)
