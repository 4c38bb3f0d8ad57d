"""The end-to-end timing schedule of bench.py, on CPU with stand-ins for CUDA
streams and events.

The pipelined schedule runs each step's three phases (indexer + top-k, the
forward, the backward) on one stream and every copy on a second, over two
device buffer sets.  The stand-ins record
every copy and every library call with the buffers it reads and writes, and
vector clocks give the happens-before order that stream order and event
waits establish.  The check: every two accesses to one buffer, at least one
of them a write, are ordered -- no buffer is overwritten while an earlier
step still reads it, and nothing is read before it is written."""
import types

import pytest
import torch

import bench


class _Rec:
    """Issued operations with their vector clocks."""

    def __init__(self):
        self.ops = []           # (kind, stream, reads, writes, clock)
        self.clocks = {}        # stream -> vector clock (dict stream -> count)
        self.current = None     # stream of the innermost torch.cuda.stream context

    def _vc(self, stream):
        return self.clocks.setdefault(stream, {})

    def op(self, kind, stream, reads=(), writes=()):
        vc = self._vc(stream)
        vc[stream] = vc.get(stream, 0) + 1
        self.ops.append((kind, stream, frozenset(reads), frozenset(writes), dict(vc)))

    def record(self, stream):
        self.op("record", stream)
        return dict(self._vc(stream))

    def wait(self, stream, snapshot):
        vc = self._vc(stream)
        for s, c in snapshot.items():
            vc[s] = max(vc.get(s, 0), c)
        self.op("wait", stream)


def _happens_before(a, b):
    """a's own tick on its stream is visible in b's clock."""
    return a[4][a[1]] <= b[4].get(a[1], 0)


def _install(monkeypatch, rec):
    class Event:
        def __init__(self, enable_timing=False):
            self.snapshot = None
            self.at = None

        def record(self, stream=None):
            name = getattr(stream, "name", "default")
            self.snapshot = rec.record(name)
            self.at = len(rec.ops)

        def elapsed_time(self, other):
            return float(other.at - self.at)

    class Stream:
        count = 0

        def __init__(self, device=None):
            Stream.count += 1
            self.name = f"s{Stream.count}"

        def wait_event(self, ev):
            rec.wait(self.name, ev.snapshot)

    class StreamCtx:
        def __init__(self, s):
            self.s = s

        def __enter__(self):
            rec.current = self.s.name

        def __exit__(self, *exc):
            rec.current = None

    monkeypatch.setattr(torch.cuda, "Event", Event)
    monkeypatch.setattr(torch.cuda, "Stream", Stream)
    monkeypatch.setattr(torch.cuda, "stream", lambda s: StreamCtx(s))
    monkeypatch.setattr(torch.cuda, "synchronize", lambda device=None: None)
    real_empty = torch.empty

    def empty(*a, pin_memory=False, **kw):    # no pinned memory without a GPU
        return real_empty(*a, **kw)

    monkeypatch.setattr(bench.torch, "empty", empty)
    real_copy = torch.Tensor.copy_

    def copy_(self, src, non_blocking=False):
        rec.op("copy", rec.current or "default", reads={id(src)}, writes={id(self)})
        return real_copy(self, src)

    monkeypatch.setattr(torch.Tensor, "copy_", copy_)


class _Lib:
    """The library calls end_to_end makes, recorded with what they read and write."""

    def __init__(self, rec):
        self.rec = rec

    def _op(self, kind, stream, reads, writes):
        self.rec.op(kind, getattr(stream, "name", "default"), {id(t) for t in reads if t is not None},
                    {id(t) for t in writes if t is not None})

    def pool_keys(self, dims, k_I, kpool, stream=None):
        self._op("pool", stream, [k_I], [kpool])

    def indexer_topk(self, dims, q_I, kpool, w, q0, n, idx, ws, ws_bytes=None, stream=None):
        self._op("select", stream, [q_I, kpool, w], [idx, ws])

    def sparse_attn_fwd(self, dims, Q, K, V, idx, o, lse, stream=None, o_acc=None):
        self._op("fwd", stream, [Q, K, V, idx], [o, lse, o_acc])

    def layer_bwd(self, dims, Q, K, V, idx, o, lse, dO, dq, dk, dv, ws=None, ws_bytes=None, stream=None,
                  o_acc=None):
        self._op("bwd", stream, [Q, K, V, idx, lse, dO, o_acc, ws], [dq, dk, dv])

    def sparse_attn_bwd_det(self, dims, Q, K, V, idx, o, lse, dO, dq, dk, dv, ws, ws_bytes=None, stream=None,
                            o_acc=None):
        self._op("bwd", stream, [Q, K, V, idx, lse, dO, o_acc], [dq, dk, dv, ws])


def _run(monkeypatch, with_bwd, steps, det=False, q_chunk=400):
    rec = _Rec()
    _install(monkeypatch, rec)
    names = ["Q", "K", "V", "q_I", "k_I", "w"] + (["dO"] if with_bwd else [])
    host = {n: torch.randn(4, 3) for n in names}
    d_in = {n: torch.zeros(4, 3) for n in names}
    bufs = types.SimpleNamespace(o=torch.zeros(4, 3), lse=torch.zeros(4), idx=torch.zeros(5), kpool=torch.zeros(6),
                                 ws=torch.zeros(7), o_acc=torch.zeros(4, 3) if with_bwd else None)
    grads = (torch.zeros(4, 3), torch.zeros(4), torch.zeros(4)) if with_bwd else (None, None, None)
    bws = torch.zeros(8) if det else None
    # the copy-rate measurement after the pipelined run is not part of the schedule
    monkeypatch.setattr(bench, "copy_bandwidth", lambda *a, **kw: {})
    dims = types.SimpleNamespace(q_chunk=q_chunk)
    r = bench.end_to_end(_Lib(rec), dims, types.SimpleNamespace(L=1000), host, d_in, bufs, *grads, bws,
                         torch.cuda.Stream(), types.SimpleNamespace(steps=steps, e2e_steps=steps), with_bwd, 1, "cpu",
                         det=det)
    return rec, r, host, d_in, names


@pytest.mark.parametrize("with_bwd,det", [(True, False), (True, True), (False, False)])
@pytest.mark.parametrize("steps", [1, 2, 3, 5])
def test_pipelined_schedule_orders_every_conflicting_access(monkeypatch, with_bwd, det, steps):
    rec, r, host, d_in, names = _run(monkeypatch, with_bwd, steps, det)
    assert r["mode"].startswith("pipelined")
    assert r["steps"] == steps
    assert r["h2d_bytes_per_step"] == sum(t.numel() * t.element_size() for t in host.values())
    assert all(torch.equal(d_in[n], host[n]) for n in names)

    # every step runs its phases once, in order, on one stream: pool keys, the
    # indexer + top-k per query chunk (1000 queries in chunks of 400: 3), the
    # forward, the backward
    kinds = [op[0] for op in rec.ops if op[0] in ("pool", "select", "fwd", "bwd")]
    per_step = ["pool", "select", "select", "select", "fwd"] + (["bwd"] if with_bwd else [])
    assert kinds == per_step * steps
    assert len({op[1] for op in rec.ops if op[0] in ("pool", "select", "fwd", "bwd")}) == 1

    # the two buffer sets alternate
    fwd_writes = [op[3] for op in rec.ops if op[0] == "fwd"]
    if steps >= 3:
        assert fwd_writes[0] != fwd_writes[1] and fwd_writes[0] == fwd_writes[2]

    # happens-before for every conflicting pair of accesses
    accesses = [op for op in rec.ops if op[2] or op[3]]
    for i, a in enumerate(accesses):
        for b in accesses[i + 1:]:
            if (a[3] & (b[2] | b[3])) or (b[3] & a[2]):
                assert _happens_before(a, b), (a[:2], b[:2])

    # copies in and out share one stream of their own, apart from the phases,
    # so two copies never run at once
    copy_streams = {op[1] for op in rec.ops if op[0] == "copy"}
    run_stream = next(op[1] for op in rec.ops if op[0] == "fwd")
    assert run_stream not in copy_streams and len(copy_streams) == 1

    # the next step's inputs are queued before this step's outputs
    copies = [op for op in rec.ops if op[0] == "copy"]
    if steps >= 2:
        host_ids = {id(t) for t in host.values()}
        h2d = [k for k, op in enumerate(copies) if op[2] & host_ids]
        first_out = next(k for k, op in enumerate(copies) if op[2] & fwd_writes[0])
        assert all(k < first_out for k in h2d[len(names):2 * len(names)])

    ov = r["overlap"]
    assert set(ov) == {"layer_ms_mean", "layer_ms_max", "run_stream_wait_ms_mean", "fill_ms", "drain_ms"}
    assert ov["layer_ms_max"] >= ov["layer_ms_mean"] > 0
    assert ov["run_stream_wait_ms_mean"] >= 0 and ov["fill_ms"] > 0 and ov["drain_ms"] > 0


def test_outputs_of_the_forward_leave_before_the_backward_ends(monkeypatch):
    """O and LSE are copied out as soon as the forward is done: their copy
    waits for the forward, not for the backward of the same step."""
    rec, _, _, _, _ = _run(monkeypatch, True, 3)
    fwd = [op for op in rec.ops if op[0] == "fwd"]
    bwd = [op for op in rec.ops if op[0] == "bwd"]
    for f, b in zip(fwd, bwd):
        outs = [op for op in rec.ops if op[0] == "copy" and op[2] & f[3] and _happens_before(f, op)]
        assert outs and not _happens_before(b, outs[0])


def test_the_check_is_not_vacuous(monkeypatch):
    """The same operations replayed without their event waits (stream order
    only) leave conflicting accesses on different streams unordered, so the
    happens-before check above can fail."""
    rec, _, _, _, _ = _run(monkeypatch, True, 3)
    replay = _Rec()
    for kind, stream, reads, writes, _ in rec.ops:
        if kind != "wait":
            replay.op(kind, stream, reads, writes)
    accesses = [op for op in replay.ops if op[2] or op[3]]
    unordered = sum(1 for i, a in enumerate(accesses) for b in accesses[i + 1:]
                    if ((a[3] & (b[2] | b[3])) or (b[3] & a[2])) and not _happens_before(a, b))
    assert unordered > 0


def test_serial_schedule_runs_every_step(monkeypatch):
    rec = _Rec()
    _install(monkeypatch, rec)
    host = {"Q": torch.randn(3)}
    d_in = {"Q": torch.zeros(3)}
    calls = []
    phases = [(["Q"], lambda d, o, s: calls.append(("a", s.name)), []),
              ([], lambda d, o, s: calls.append(("b", s.name)), [0, 1])]
    ms = bench._e2e_serial(host, ["Q"], d_in, [torch.zeros(2), torch.zeros(1)], phases, 3, torch.cuda.Stream(), "cpu")
    assert [c[0] for c in calls] == ["a", "b"] * 4         # one warm-up step, three timed
    assert len({c[1] for c in calls}) == 1
    assert ms == 0.0 or ms > 0
    assert torch.equal(d_in["Q"], host["Q"])
