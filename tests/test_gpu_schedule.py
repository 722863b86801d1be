"""The device scheduler's work list, bit for bit against a host recomputation.

After a call, the workspace holds a 64-byte header (int32: long items, 0, rows
per long item, the tiny bound, error, tiny items, whether every long item is
split) and the items (int4: segment start, segment length, first query row,
head | split flag). The host recomputes the same list from the segment lengths
and the SM count alone: segments longer than min(split, 64) go to the tcgen05
kernel in 256-row blocks, longest first (ties by index), a last block of at
most 128 rows flagged as split; when that would give at most SMs / 2 long
items, every long segment goes in 128-row blocks instead, all flagged. The
rest (tiny segments) follow in index order, one item per head; heads outer,
query blocks inner within a segment."""
import numpy as np
import pytest
import torch

import vision_encoder_varlen_gb300 as vit
from vision_encoder_varlen_gb300 import _build

pytestmark = pytest.mark.gpu

BM_LONG, TINY = 256, 64
SPLIT = 1 << 30


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()


def expected(lengths, starts, H, short_max, num_sms):
    tiny_max = min(short_max, TINY)
    idx = range(len(lengths))
    long_s = sorted((i for i in idx if lengths[i] > tiny_max), key=lambda i: (-lengths[i], i))
    tiny_s = [i for i in idx if lengths[i] <= tiny_max]
    full_items = sum(H * -(-int(lengths[i]) // BM_LONG) for i in long_s)
    all_split = 2 * full_items <= num_sms
    bm_long = BM_LONG // 2 if all_split else BM_LONG
    items, counts = [], []
    for group, bm in ((long_s, bm_long), (tiny_s, TINY)):
        n0 = len(items)
        for seg in group:
            L, a = int(lengths[seg]), int(starts[seg])
            if L == 0:
                continue
            nq = (L + bm - 1) // bm
            for h in range(H):
                for qb in range(nq):
                    last_rows = L - qb * bm
                    split = group is long_s and (all_split or (qb == nq - 1 and 2 * last_rows <= BM_LONG))
                    items.append((a, L, a + qb * bm, h | (SPLIT if split else 0)))
        counts.append(len(items) - n0)
    return counts, np.array(items, dtype=np.int32).reshape(-1, 4), bm_long, all_split


def _num_sms():
    return torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count


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
    with vit.kernel_split(short_max):
        status = vit.new_status()
        if padded:
            vit.varlen_attn_padded(q, q, q, torch.from_numpy(starts.astype(np.int32)).cuda(),
                                   torch.from_numpy(lengths.astype(np.int32)).cuda(), int(lengths.max()),
                                   workspace=ws, status=status)
        else:
            cu = torch.from_numpy(np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)).cuda()
            vit.varlen_attn(q, q, q, cu, max(int(lengths.max()), 1), workspace=ws, status=status)
        assert vit.read_status(status) == 0
    raw = ws.cpu().numpy()
    hdr = raw[:64].view(np.int32)
    return hdr, raw[64:].view(np.int32).reshape(-1, 4), starts


CASES = [
    ([300, 1, 0, 64, 65, 2000, 129, 128, 17, 0, 700], 3),
    ([5, 4096, 4096, 4095, 1], 2),
    ([64] * 50 + [65] * 7 + [1000] * 3, 1),
    ([1024], 16),                                   # one 32x32 image: few items, all split
    ([1000, 129, 300], 8),                          # exactly at the all-split threshold region
    ([200, 90, 65], 1),
]


@pytest.mark.parametrize("padded", [False, True])
@pytest.mark.parametrize("short_max", [64, 0, 2 ** 31 - 1, 100, 32])
@pytest.mark.parametrize("lengths,H", CASES)
def test_work_list_matches_host_recomputation(lengths, H, short_max, padded):
    hdr, items, starts = run(lengths, H, 80, short_max, padded)
    counts, ref, bm_long, all_split = expected(np.asarray(lengths), starts, H, short_max, _num_sms())
    n = sum(counts)
    assert hdr[4] == 0                                     # no error
    assert (hdr[0], hdr[1], hdr[5]) == (counts[0], 0, counts[1])
    if counts[0]:
        assert hdr[2] == bm_long and hdr[6] == int(all_split)
    assert hdr[3] == min(short_max, TINY)
    assert np.array_equal(items[:n], ref)


def test_small_batches_are_cut_into_split_items():
    # 16 heads of one 1024-token image: 64 two-tile items would leave most SMs idle, so the
    # scheduler cuts 128 split items of 128 rows instead (up to 152 SMs)
    if _num_sms() < 128:
        pytest.skip("needs at least 128 SMs")
    hdr, items, _ = run([1024], 16, 80, 64)
    assert hdr[0] == 128 and hdr[2] == 128 and hdr[6] == 1
    assert np.all(items[:128, 3] & SPLIT)


def test_work_list_many_segments():
    rng = np.random.default_rng(4)
    lengths = rng.integers(0, 300, size=3000)
    lengths[rng.choice(3000, 20, replace=False)] = rng.integers(1000, 5000, size=20)
    hdr, items, starts = run(lengths, 2, 64, 64)
    counts, ref, _, _ = expected(lengths, starts, 2, 64, _num_sms())
    assert (hdr[0], hdr[1], hdr[5]) == (counts[0], 0, counts[1])
    assert np.array_equal(items[:sum(counts)], ref)
