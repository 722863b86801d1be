"""Model check of the tcgen05 long-segment kernel's barrier protocol (one CTA, CPU only).

The kernel's roles talk only through mbarriers: the TMA producer (Q per item, each
tile's K, then the previous tile's V), the item ring it feeds, two MMA issuers
(two-tile items, and split items whose key tiles alternate between them), eight
softmax warps (two groups; split items end with a two-phase merge; at head_dim 128 a
two-tile item's output is written after the group has stored the first P of its next
item, at the other head dims at once) and warp 3. This
module replays exactly those waits and arrivals as Python generators under a random
scheduler with random completion latencies for the asynchronous copies and MMAs,
and checks on every run:

* no deadlock;
* every parity wait passes exactly when the phase it means has completed: never on
  an older phase of the same parity (a waiter two phases behind), and never while
  the barrier is already past it;
* every buffer is read only when it holds what the reader expects (Q of the item,
  K and V of the tile, S and P of the tile, O accumulated over exactly the tiles of
  the item or of its half), and is written only after its previous readers finished.

It mirrors the waits and arrivals of csrc/attn_long.cu: a change to the kernel's
protocol is a change to this model. Planted mistakes (switches of the model) show
that the checks catch the failures they are meant to catch."""
import random

import pytest


class Bar:
    """mbarrier: an arrival count per phase, a transaction count, the completed-phase count."""

    def __init__(self, name, count):
        self.name, self.count = name, count
        self.k = 0
        self.arr = 0
        self.tx = 0

    def _check(self):
        if self.arr == self.count and self.tx == 0:
            self.k += 1
            self.arr = 0

    def arrive(self, tx=0):
        self.arr += 1
        self.tx += tx
        assert self.arr <= self.count, f"{self.name}: too many arrivals"
        self._check()

    def complete_tx(self, n):
        self.tx -= n
        assert self.tx >= 0
        self._check()

    def passes(self, intended):
        """try_wait.parity: true when the current phase's parity differs from the waited one."""
        if self.name == "always":
            return True
        ok = (self.k & 1) != (intended & 1)
        if ok:
            assert self.k == intended + 1, f"{self.name}: wait for phase {intended} passed at {self.k} phases"
        else:
            assert self.k <= intended, f"{self.name}: waiter two phases behind (phase {intended}, {self.k} done)"
        return ok


class Model:
    """One CTA's roles over a list of items (index, (segment length, split))."""

    def __init__(self, items, ST, QBUF, BN, seed, mistake=None, defer=False):
        self.rng = random.Random(seed)
        self.defer = defer
        self.items, self.ST, self.QBUF, self.BN, self.mistake = items, ST, QBUF, BN, mistake
        B = lambda n, c: [Bar(f"{n}{i}", c) for i in range(max(ST, 2))]
        self.q_full, self.q_empty = B("q_full", 1), B("q_empty", 2)
        self.k_full, self.v_full = B("k_full", 1), B("v_full", 1)
        self.k_empty, self.v_empty = B("k_empty", 2), B("v_empty", 2)
        self.s_full, self.s_free = B("s_full", 1), B("s_free", 4)
        self.p_full, self.pv_done, self.o_free = B("p_full", 4), B("pv_done", 1), B("o_free", 4)
        self.merge = Bar("merge", 8)
        self.R = 4
        self.item_full = [Bar(f"item_full{i}", 1) for i in range(self.R)]
        self.item_empty = [Bar(f"item_empty{i}", 11) for i in range(self.R)]
        self.ring = [None] * self.R
        self.always = Bar("always", 1)
        self.events = []
        self.time = 0
        self.qbuf = [None] * QBUF
        self.kst, self.vst = [None] * ST, [None] * ST
        self.k_readers, self.v_readers = [0] * ST, [0] * ST
        self.S, self.P, self.O = [None, None], [None, None], [None, None]
        self.O_readers = [0, 0]
        self.mma_q = [[], []]
        self.s_reads, self.p_writes, self.merges = {}, {}, {}

    def later(self, fn):
        self.events.append((self.time + self.rng.randint(1, 30), fn))

    def take(self, k, out):
        slot = k % self.R
        yield (self.item_full[slot], k // self.R)
        out.append(self.ring[slot])
        self.item_empty[slot].arrive()

    def items_taken(self):
        """The generator protocol of a consumer of the item ring: yields waits, returns items."""
        k = 0
        while True:
            got = []
            yield from self.take(k, got)
            if got[0] is None:
                return
            yield ("item", k, got[0])
            k += 1

    # ------------------------------------------------------------ producer
    def producer(self):
        ST, QBUF, BN = self.ST, self.QBUF, self.BN
        g, k_pub, pend_v = 0, 0, None

        def load_v(gv, idx, j):
            st = gv % ST
            if gv >= ST:
                yield (self.v_empty[st], gv // ST - 1)
            assert self.v_readers[st] == 0, "V half refilled while a P.V reads it"
            self.v_full[st].arrive(tx=1)

            def land(st=st, v=(idx, j)):
                self.vst[st] = v
                self.v_full[st].complete_tx(1)
            self.later(land)

        def publish(x):
            nonlocal k_pub
            slot = k_pub % self.R
            if k_pub >= self.R:
                yield (self.item_empty[slot], k_pub // self.R - 1)
            self.ring[slot] = x
            self.item_full[slot].arrive()
            k_pub += 1

        for q_it, (idx, (L, split)) in enumerate(self.items):
            yield from publish((idx, (L, split)))
            qb, qn = q_it % QBUF, q_it // QBUF
            if qn > 0:
                yield (self.q_empty[qb], qn - 1)
            self.q_full[qb].arrive(tx=1)

            def land_q(qb=qb, idx=idx):
                self.qbuf[qb] = idx
                self.q_full[qb].complete_tx(1)
            self.later(land_q)
            for j in range(-(-L // BN)):
                st = g % ST
                if g >= ST:
                    yield (self.k_empty[st], g // ST - 1)
                assert self.k_readers[st] == 0, "K half refilled while a QK reads it"
                self.k_full[st].arrive(tx=1)

                def land_k(st=st, v=(idx, j)):
                    self.kst[st] = v
                    self.k_full[st].complete_tx(1)
                self.later(land_k)
                if pend_v is not None:          # each tile's V goes out after the next tile's K
                    yield from load_v(*pend_v)
                pend_v = (g, idx, j)
                g += 1
        if pend_v is not None:
            yield from load_v(*pend_v)
        yield from publish(None)

    # ------------------------------------------------------------ MMA issuers
    def _mma(self, ti, start, done):
        start()
        q = self.mma_q[ti]
        t = max(q[-1] if q else self.time, self.time) + self.rng.randint(1, 20)
        q.append(t)                             # an issuer's MMAs complete in order
        self.events.append((t, done))

    def _commit(self, ti, bar):
        q = self.mma_q[ti]
        t = max(q[-1] if q else self.time, self.time) + 1
        q.append(t)
        self.events.append((t, bar.arrive))

    def issuer(self, ti):
        ST, QBUF, BN = self.ST, self.QBUF, self.BN
        t = c = 0
        for ev in self.items_taken():
            if ev[0] != "item":
                yield ev
                continue
            _, item_cnt, (idx, (L, split)) = ev
            n_kv = -(-L // BN)
            qb = item_cnt % QBUF
            yield (self.q_full[qb], item_cnt // QBUF)

            def qk(j, st, idx=idx, qb=qb):
                def start():
                    assert self.qbuf[qb] == idx, "Q not loaded"
                    assert self.kst[st] == (idx, j), f"K slot holds {self.kst[st]}, want {(idx, j)}"
                    assert self.S[ti] in (None, "free"), "S overwritten before it was read"
                    self.k_readers[st] += 1
                    self.S[ti] = "busy"

                def done(idx=idx, j=j, st=st):
                    self.k_readers[st] -= 1
                    self.S[ti] = (idx, j)
                self._mma(ti, start, done)
                self._commit(ti, self.s_full[ti])

            def pv(j, st, first, idx=idx):
                def start():
                    assert self.vst[st] == (idx, j), "V slot"
                    assert self.P[ti] == (idx, j), f"P holds {self.P[ti]}, want {(idx, j)}"
                    assert self.O_readers[ti] == 0, "O written while it is read"
                    if first:
                        self.O[ti] = (idx, frozenset())
                    self.v_readers[st] += 1

                def done(j=j, idx=idx, st=st):
                    self.v_readers[st] -= 1
                    assert self.O[ti][0] == idx
                    self.O[ti] = (idx, self.O[ti][1] | {j})
                    self.P[ti] = "consumed"
                self._mma(ti, start, done)
                self._commit(ti, self.pv_done[ti])

            if not split:
                # two-tile item: QK of the next tile before P.V of this one
                st = t % ST
                yield (self.k_full[st], t // ST)
                if c > 0:
                    yield (self.s_free[ti], c - 1)
                qk(0, st)
                self._commit(ti, self.k_empty[st])
                if n_kv == 1:
                    self._commit(ti, self.q_empty[qb])
                for j in range(n_kv):
                    u, st, st1 = c + j, (t + j) % ST, (t + j + 1) % ST
                    if j + 1 < n_kv:
                        yield (self.k_full[st1], (t + j + 1) // ST)
                        yield (self.s_free[ti], u)
                        qk(j + 1, st1)
                        self._commit(ti, self.k_empty[st1])
                        if j + 2 == n_kv:
                            self._commit(ti, self.q_empty[qb])
                    yield (self.v_full[st], (t + j) // ST)
                    if j == 0 and item_cnt > 0:
                        yield (self.o_free[ti], item_cnt - 1)
                    yield (self.p_full[ti], u)
                    pv(j, st, j == 0)
                    self._commit(ti, self.v_empty[st])
                t += n_kv
                c += n_kv
                continue
            # split item: tiles j = ti, ti + 2, ...; the other issuer's tiles are passed and released
            prev, first_pv, skip = None, [True], [None]

            def pv_of_prev(prev):
                pj, pst, puse, pc = prev
                yield (self.v_full[pst], puse)
                if first_pv[0] and item_cnt > 0:
                    yield (self.o_free[ti], item_cnt - 1)
                yield (self.p_full[ti], pc)
                pv(pj, pst, first_pv[0])
                self._commit(ti, self.v_empty[pst])
                first_pv[0] = False

            def pass_skipped_v():
                if skip[0] is not None:
                    sst, suse = skip[0]
                    yield (self.v_full[sst], suse)
                    self.v_empty[sst].arrive()
                    skip[0] = None

            for j in range(n_kv):
                st, use = (t + j) % ST, (t + j) // ST
                if (j & 1) != ti:
                    if self.mistake != "skip_no_k_wait":
                        yield (self.k_full[st], use)
                    self.k_empty[st].arrive()
                    skip[0] = (st, use)
                    continue
                yield (self.k_full[st], use)
                if c > 0:
                    yield (self.s_free[ti], c - 1)
                qk(j, st)
                self._commit(ti, self.k_empty[st])
                if j + 2 >= n_kv:
                    self._commit(ti, self.q_empty[qb])
                yield from pass_skipped_v()
                if prev is not None:
                    yield from pv_of_prev(prev)
                prev = (j, st, use, c)
                c += 1
            if prev is None and self.mistake != "q_release_after_skipped_v":
                self.q_empty[qb].arrive()
            yield from pass_skipped_v()
            if prev is None and self.mistake == "q_release_after_skipped_v":
                self.q_empty[qb].arrive()
            if prev is not None:
                yield from pv_of_prev(prev)
            elif item_cnt > 0:
                yield (self.o_free[ti], item_cnt - 1)
            t += n_kv

    # ------------------------------------------------------------ softmax warps and warp 3
    def _write_out(self, grp, idx, n_kv):
        """A two-tile item's output: O read (it must hold every tile of the item), then o_free."""
        self.O_readers[grp] += 1
        assert self.O[grp] == (idx, frozenset(range(n_kv))), f"O {self.O[grp]}"
        yield (self.always, 0)                  # the epilogue's reads take time
        assert self.O[grp] == (idx, frozenset(range(n_kv))), f"O changed while read {self.O[grp]}"
        self.O_readers[grp] -= 1
        self.o_free[grp].arrive()

    def softmax(self, grp, warp):
        BN = self.BN
        p_cnt = 0
        pend = None                             # a two-tile item whose output is not written yet
        for ev in self.items_taken():
            if ev[0] != "item":
                yield ev
                continue
            _, item_cnt, (idx, (L, split)) = ev
            n_kv = -(-L // BN)
            j, dj = (grp, 2) if split else (0, 1)
            while j < n_kv:
                yield (self.s_full[grp], p_cnt)
                assert self.S[grp] == (idx, j), f"S holds {self.S[grp]}, want {(idx, j)}"
                key = (grp, idx, j)
                self.s_reads[key] = self.s_reads.get(key, 0) + 1
                if self.s_reads[key] == 4:
                    self.S[grp] = "free"
                self.s_free[grp].arrive()
                if p_cnt > 0:
                    yield (self.pv_done[grp], p_cnt - 1)
                self.p_writes[key] = self.p_writes.get(key, 0) + 1
                if self.p_writes[key] == 4:
                    assert self.P[grp] in (None, "consumed"), f"P overwritten: {self.P[grp]}"
                    self.P[grp] = (idx, j)
                self.p_full[grp].arrive()
                p_cnt += 1
                # the previous item's output, after the first P of this one (its last P.V is done)
                if pend is not None:
                    yield from self._write_out(grp, *pend)
                    pend = None
                j += dj
            if not split:
                if self.defer:                  # head_dim 128: written after the next item's first P
                    pend = (idx, n_kv)
                else:                           # other head dims: written at once
                    yield (self.pv_done[grp], p_cnt - 1)
                    yield from self._write_out(grp, idx, n_kv)
                continue
            if pend is not None:                # a split item without a tile of this group
                yield (self.pv_done[grp], p_cnt - 1)
                yield from self._write_out(grp, *pend)
                pend = None
            n1 = n_kv >> 1
            if grp == 0 or n1 > 0:
                yield (self.pv_done[grp], p_cnt - 1)
            ph = self.merges.get((grp, warp), 0)     # merge phases this warp has waited for
            self.merge.arrive()
            yield (self.merge, ph)
            halves = [(0, frozenset(range(0, n_kv, 2)))] + ([(1, frozenset(range(1, n_kv, 2)))] if n1 else [])
            for h, want in halves:
                self.O_readers[h] += 1
                assert self.O[h] == (idx, want), f"O{h} {self.O[h]}"
            yield (self.always, 0)              # the merge's reads take time
            for h, want in halves:
                assert self.O[h] == (idx, want), f"O{h} changed while read {self.O[h]}"
                self.O_readers[h] -= 1
            if self.mistake != "merge_one_meeting":
                self.merge.arrive()
                yield (self.merge, ph + 1)
                self.merges[(grp, warp)] = ph + 2
            else:
                self.merges[(grp, warp)] = ph + 1
            self.o_free[grp].arrive()
        if pend is not None:                    # the last item's output
            yield (self.pv_done[grp], p_cnt - 1)
            yield from self._write_out(grp, *pend)

    def warp3(self):
        for ev in self.items_taken():
            if ev[0] != "item":
                yield ev

    # ------------------------------------------------------------ scheduler
    def run(self):
        roles = [self.producer(), self.issuer(0), self.issuer(1), self.warp3()]
        roles += [self.softmax(g, w) for g in (0, 1) for w in range(4)]
        pending = [None] * len(roles)
        alive = set(range(len(roles)))
        for _ in range(2_000_000):
            if not alive and not self.events:
                return
            progressed = False
            order = list(alive)
            self.rng.shuffle(order)
            for i in order:
                w = pending[i]
                if w is not None and not w[0].passes(w[1]):
                    continue
                try:
                    pending[i] = next(roles[i])
                except StopIteration:
                    alive.discard(i)
                    pending[i] = None
                progressed = True
                break
            if progressed and self.rng.random() < 0.7:
                continue
            if self.events:
                self.events.sort(key=lambda e: e[0])
                self.time = max(self.time, self.events[0][0])
                due = [e for e in self.events if e[0] <= self.time]
                self.events = [e for e in self.events if e[0] > self.time]
                self.rng.shuffle(due)
                for _, fn in due:
                    fn()
                continue
            if not progressed:
                stuck = {i: (pending[i][0].name, pending[i][1], pending[i][0].k) for i in alive}
                raise AssertionError(f"deadlock: {stuck}")
        raise AssertionError("no progress bound")


def random_case(seed):
    rng = random.Random(seed)
    ST, QBUF, BN = rng.choice([2, 3, 4]), rng.choice([1, 2]), rng.choice([80, 112, 128])
    items = []
    for i in range(rng.randint(1, 7)):
        L = rng.choice([65, 100, 128, 129, 200, 257, 300, 700, 1000, BN, BN + 1, 2 * BN, 2 * BN + 5])
        items.append((i, (L, rng.random() < 0.5)))
    return items, ST, QBUF, BN


@pytest.mark.parametrize("defer", [False, True])
def test_protocol_holds_over_random_layouts_and_timings(defer):
    for seed in range(400):
        items, ST, QBUF, BN = random_case(seed)
        Model(items, ST, QBUF, BN, seed, defer=defer).run()


@pytest.mark.parametrize("mistake,expect", [
    ("skip_no_k_wait", "two phases behind|passed at|refilled"),  # a skipped tile's K phase not taken
    ("q_release_after_skipped_v", "deadlock"),                   # Q buffer released after the lagging V
    ("merge_one_meeting", "changed while read|written while|O"),   # merge without its second meeting
])
def test_planted_protocol_mistakes_are_caught(mistake, expect):
    import re
    caught = None
    for seed in range(600):
        items, ST, QBUF, BN = random_case(seed)
        try:
            Model(items, ST, QBUF, BN, seed, mistake=mistake).run()
        except AssertionError as e:
            caught = str(e)
            break
    assert caught is not None, f"{mistake} not caught"
    assert re.search(expect, caught), caught
