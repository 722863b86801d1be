"""Race check of the benchmark's end-to-end pipeline, on the CPU.

bench.E2EPipeline overlaps host->device uploads, the compute and device->host downloads
on three CUDA streams over two sets of device buffers, ordered only by events. Here
torch's streams, events and tensors are replaced by recording fakes, the pipeline runs
a few steps, and every pair of accesses to one buffer where at least one writes must be
ordered by happens-before: program order within a stream, plus an edge from each event
record to every wait on it. A control run with one of the pipeline's waits removed must
be reported as a race, so the check itself is known to work."""
import contextlib
import itertools

import pytest
import torch

import bench
from vision_encoder_varlen_gb300 import workloads as wl


class _Recorder:
    def __init__(self):
        self.nodes = []                      # (stream id, kind, payload)
        self.streams = {}
        self.stack = []
        self.default = self.new_stream()

    def new_stream(self):
        s = _Stream(self, len(self.streams))
        self.streams[s.sid] = s
        return s

    def current(self):
        return self.stack[-1] if self.stack else self.default

    def op(self, stream, kind, payload=None):
        node = len(self.nodes)
        self.nodes.append((stream.sid, kind, payload))
        stream.ops.append(node)
        return node


class _Stream:
    def __init__(self, rec, sid):
        self.rec, self.sid, self.ops = rec, sid, []

    def wait_event(self, ev):
        self.rec.op(self, "wait", ev.node)   # the record this wait observes (None: never recorded)


class _Event:
    def __init__(self, rec):
        self.rec, self.node = rec, None

    def record(self, stream=None):
        self.node = self.rec.op(stream or self.rec.current(), "record")


class _Tensor:
    _ids = itertools.count()

    def __init__(self, rec, name):
        self.rec, self.name = rec, f"{name}#{next(self._ids)}"

    def copy_(self, src, non_blocking=False):
        s = self.rec.current()
        self.rec.op(s, "read", src.name)
        self.rec.op(s, "write", self.name)
        return self

    def numel(self):
        return 1


class _Vit:
    """The three calls of a step, as buffer reads and writes on the current stream."""

    def __init__(self, rec):
        self.rec = rec

    def _touch(self, reads, writes):
        s = self.rec.current()
        for t in reads:
            if t is not None:
                self.rec.op(s, "read", t.name)
        for t in writes:
            self.rec.op(s, "write", t.name)

    def workspace_size(self, *a):
        return 16

    def rope_freqs(self, grid, *a, **k):
        outs = [_Tensor(self.rec, n) for n in ("inv_freq", "pos", "cu")]
        self._touch([grid], outs)
        return tuple(outs)

    def qk_norm_rope(self, q, k, pos, inv_freq, nw, eps, inplace=False, **kw):
        assert inplace
        self._touch([q, k, pos, inv_freq, nw], [q, k])

    def varlen_attn(self, q, k, v, cu, max_seqlen, out=None, workspace=None, **kw):
        self._touch([q, k, v, cu], [workspace])
        self._touch([workspace], [out])


def _happens_before(rec):
    succ = {i: set() for i in range(len(rec.nodes))}
    for s in rec.streams.values():
        for a, b in zip(s.ops, s.ops[1:]):
            succ[a].add(b)
    for i, (_, kind, payload) in enumerate(rec.nodes):
        if kind == "wait" and payload is not None:
            succ[payload].add(i)
    reach = {}
    for i in reversed(range(len(rec.nodes))):      # edges only go to later nodes
        r = set()
        for j in succ[i]:
            r.add(j)
            r |= reach[j]
        reach[i] = r
    return reach


def _races(rec):
    reach = _happens_before(rec)
    by_buf = {}
    for i, (_, kind, name) in enumerate(rec.nodes):
        if kind in ("read", "write"):
            by_buf.setdefault(name, []).append((i, kind))
    found = []
    for name, acc in by_buf.items():
        for (i, ki), (j, kj) in itertools.combinations(acc, 2):
            if "write" in (ki, kj) and j not in reach[i] and i not in reach[j]:
                found.append((name, i, j))
    return found


def _run_pipeline(monkeypatch, steps=5, drop=None):
    rec = _Recorder()
    monkeypatch.setattr(torch.cuda, "Stream", lambda *a, **k: rec.new_stream())
    monkeypatch.setattr(torch.cuda, "Event", lambda *a, **k: _Event(rec))
    monkeypatch.setattr(torch.cuda, "current_stream", lambda *a, **k: rec.current())

    @contextlib.contextmanager
    def stream_ctx(s):
        rec.stack.append(s)
        try:
            yield
        finally:
            rec.stack.pop()

    monkeypatch.setattr(torch.cuda, "stream", stream_ctx)
    monkeypatch.setattr(torch, "empty", lambda *a, **k: _Tensor(rec, "dev"))
    monkeypatch.setattr(torch, "empty_like", lambda *a, **k: _Tensor(rec, "dev"))
    if drop is not None:
        real = _Stream.wait_event

        def wait_event(self, ev):
            if ev is not None and ev in drop(pipe):
                return
            real(self, ev)
        monkeypatch.setattr(_Stream, "wait_event", wait_event)
    w = wl.make_config(3)
    host = {n: _Tensor(rec, "host_" + n) for n in ("grid", "q", "k", "v", "nw", "out")}
    pipe = bench.E2EPipeline(_Vit(rec), w, host, device="cuda")
    start = _Event(rec)
    start.record(rec.default)
    pipe.run(3)                                        # warm-up, as the benchmark does
    pipe.run(steps, start_event=start)
    return rec


def test_pipeline_has_no_unordered_conflicting_accesses(monkeypatch):
    rec = _run_pipeline(monkeypatch)
    assert sum(1 for n in rec.nodes if n[1] == "write") > 50
    assert _races(rec) == []


@pytest.mark.parametrize("which", ["downloaded", "consumed", "uploaded"])
def test_a_missing_wait_is_reported(monkeypatch, which):
    # drop every wait on one kind of event of buffer set 0: the check must find a race
    rec = _run_pipeline(monkeypatch, drop=lambda pipe: {pipe.bufs[0][which]})
    assert _races(rec), which
