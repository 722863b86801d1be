"""Model check of the tiny-segment kernel's item ring (csrc/attn_tiny.cu), CPU only.

The kernel's producer warp places each item's Q, K and V tiles (ceil16(L) rows of HG heads
each, every tile rounded up to 1024 bytes) at the next free bytes of a shared-memory ring,
wrapping to the ring start when the item would cross its end, and frees items strictly in
item order by waiting for the oldest item's release until the item fits or the ring is
empty (an empty ring takes any item not larger than it); a 32-entry descriptor ring bounds
the items in the ring. Consumer groups take the items in turn and release them in any order
relative to each other.

This replays that allocation rule against consumers that finish in random order and
checks that an item is never placed over the bytes of an item that its consumers have
not released, that no item crosses the ring's end, and that the producer never waits for
an item it has not issued (a deadlock)."""
import random

import pytest

TM = 64
SLOTS = 32
GROUPS = 3
RING = 220 * 1024


def tile_bytes(D, n16, HG=1):
    return (16 * n16 * HG * D * 2 + 1023) // 1024 * 1024


def simulate(lengths, D, seed, mistake=None, HG=1):
    rng = random.Random(seed)
    head = freed = 0
    released_view = 0                      # items the producer has seen released (in order)
    live = {}                              # item -> (offset, size), not yet released by its consumers
    done = set()
    end_of = {}
    pending = list(range(len(lengths)))    # items the producer still has to place

    def consumer_step():
        # the oldest not-yet-released item of a random group may finish now
        g = rng.randrange(GROUPS)
        mine = [m for m in sorted(live) if m % GROUPS == g]
        if mine:
            del live[mine[0]]              # a group finishes its items in order
            done.add(mine[0])
            return True
        return False

    while pending or live:
        if not (pending and rng.random() < 0.5):
            consumer_step()
            continue
        n = pending[0]
        sz = 3 * tile_bytes(D, (lengths[n] + 15) // 16, HG)
        start = head
        if start % RING + sz > RING and mistake != "no_wrap":
            start += RING - start % RING
        blocked = False
        while n - released_view >= SLOTS or (released_view < n and start + sz > freed + RING):
            if released_view not in done and mistake != "free_without_wait":
                blocked = True             # the wait on the oldest item's release
                break
            freed = end_of[released_view]
            released_view += 1
        if blocked:
            if not consumer_step():
                for _ in range(GROUPS * 4):
                    if consumer_step():
                        break
            continue
        if released_view == n and mistake != "keep_stale_freed":
            freed = start                  # empty ring: all of it is free
        off = start % RING
        assert off + sz <= RING, "item crosses the ring end"
        for m, (o, s) in live.items():
            assert off + sz <= o or o + s <= off, f"item {n} placed over live item {m}"
        live[n] = (off, sz)
        end_of[n] = start + sz
        head = start + sz
        pending.pop(0)


@pytest.mark.parametrize("D,HG", [(32, 1), (32, 2), (64, 1), (80, 1), (80, 2), (80, 4), (96, 1), (96, 2), (128, 1)])
def test_ring_never_overlaps_live_items(D, HG):
    rng = random.Random(D * 8 + HG)
    for seed in range(60):
        kind = seed % 3
        if kind == 0:
            lengths = [rng.randint(1, TM) for _ in range(300)]
        elif kind == 1:
            lengths = [rng.choice([1, 16, 17, 63, 64]) for _ in range(300)]
        else:
            lengths = [TM] * 200
        simulate(lengths, D, seed, HG=HG)


def test_largest_item_fits_the_empty_ring():
    for D, HG in [(32, 2), (64, 1), (80, 2), (80, 4), (96, 2), (128, 1)]:
        assert 3 * tile_bytes(D, TM // 16, HG) <= RING


@pytest.mark.parametrize("mistake", ["free_without_wait", "no_wrap"])
def test_planted_ring_mistakes_are_caught(mistake):
    with pytest.raises(AssertionError):
        for seed in range(50):
            simulate([TM] * 100, 80, seed, mistake=mistake, HG=2)
