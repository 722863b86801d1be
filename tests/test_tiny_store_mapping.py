"""CPU model of the tiny-segment kernel's output stores (no GPU).

The m16n8k16 accumulator gives lane (g, t) of a warp, g = lane / 4 and t = lane % 4, the two
columns 2t and 2t + 1 of every 8-column block for rows g and g + 8. The kernel stores wider
pieces: the four lanes of a quad transpose one word (two bf16 columns) of each of four blocks
in two shuffle stages (partners two apart, then neighbours), so lane t holds the whole block
j + t of its row for one 16-byte store; a trailing pair of blocks (head_dim 80: ten blocks)
swaps one word between neighbours for 8-byte stores. This model replays those exchanges on
symbolic words, one per (row, column pair), and checks that every (row, column) of a 16-row
unit is written exactly once, with its own value, at aligned offsets, for the head dims and
chunk widths the kernel compiles with wide stores (head_dim 128 keeps 4-byte stores). Planted
mistakes in the exchange fail it."""
import pytest


def sel(c, a, b):
    return a if c else b


def transpose4(xs, mistake=None):
    """xs[lane] = that lane's words of blocks j..j+3; returns each lane's words of block j + t
    in column order, exchanging values only as the kernel's shuffles do."""
    p2 = 1 if mistake == "stage1_neighbour" else 2
    kept, send2 = {}, {}
    for ln, x in xs.items():
        hi = ln & 2
        kept[ln] = (sel(hi, x[2], x[0]), sel(hi, x[3], x[1]))
        send2[ln] = (sel(hi, x[0], x[2]), sel(hi, x[1], x[3]))
    send1, own = {}, {}
    for ln in xs:
        lo = ln & 1
        (k0, k1), (g0, g1) = kept[ln], send2[ln ^ p2]
        send1[ln] = (sel(lo, k0, k1), sel(lo, g0, g1))
        own[ln] = (sel(lo, k1, k0), sel(lo, g1, g0))
    out = {}
    for ln in xs:
        lo, hi = ln & 1, ln & 2
        z0, z2 = own[ln]
        z1, z3 = send1[ln ^ 1]
        if mistake == "no_reorder":
            out[ln] = (z0, z1, z2, z3)
            continue
        w = (sel(lo, z1, z0), sel(lo, z0, z1), sel(lo, z3, z2), sel(lo, z2, z3))
        out[ln] = (w[2], w[3], w[0], w[1]) if hi else w
    return out


def run_unit(D, NC, mistake=None):
    DN = D // 8
    written = {}

    def put(row, col, words, align):
        assert (col * 2) % align == 0, f"column {col} not {align}-byte aligned"
        for e, wd in enumerate(words):
            for h in range(2):
                key = (row, col + 2 * e + h)
                assert key not in written, f"{key} written twice"
                written[key] = wd[h]

    for c0 in range(0, DN, NC):
        for rs in (0, 1):                      # accumulator rows g and g + 8
            def word(lane, blk):
                r, t = (lane >> 2) + 8 * rs, lane & 3
                return ((r, blk * 8 + 2 * t), (r, blk * 8 + 2 * t + 1))

            for j in range(0, NC - 3, 4):
                ys = transpose4({ln: [word(ln, c0 + j + i) for i in range(4)] for ln in range(32)}, mistake)
                for ln, y in ys.items():
                    put((ln >> 2) + 8 * rs, (c0 + j + (ln & 3)) * 8, y, 16)
            if NC % 4 == 2:                    # the trailing pair of blocks
                j = NC - 2
                for ln in range(32):
                    lo = ln & 1
                    p = ln ^ 1
                    got = sel(p & 1, word(p, c0 + j), word(p, c0 + j + 1))
                    a, b = word(ln, c0 + j), word(ln, c0 + j + 1)
                    put((ln >> 2) + 8 * rs, (c0 + j + lo) * 8 + (ln & 2) * 2, (got, b) if lo else (a, got), 8)
    assert len(written) == 16 * D
    for key, val in written.items():
        assert key == val, f"{key} holds {val}"


# (head_dim, 8-column blocks per P.V chunk) of every variant with 16- or 8-byte stores
VARIANTS = [(32, 4), (64, 8), (80, 10), (96, 12), (96, 4)]


@pytest.mark.parametrize("D,NC", VARIANTS)
def test_every_output_element_written_once_in_place(D, NC):
    run_unit(D, NC)


@pytest.mark.parametrize("mistake", ["stage1_neighbour", "no_reorder"])
def test_planted_exchange_mistakes_are_caught(mistake):
    with pytest.raises(AssertionError):
        run_unit(80, 10, mistake)
