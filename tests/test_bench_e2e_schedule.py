"""The end-to-end timing schedule of bench.py, on CPU with stand-ins for CUDA
streams and events: two device buffer sets over three streams.  Every step's
input copy, layer and output copy must be ordered so that no buffer set is
overwritten while an earlier step still uses it."""
import types

import pytest
import torch

import bench


class _Rec:
    def __init__(self):
        self.ops = []           # (kind, stream, payload) in issue order
        self.current = None     # stream of the innermost torch.cuda.stream context


def _install(monkeypatch, rec):
    class Event:
        count = 0

        def __init__(self, enable_timing=False):
            Event.count += 1
            self.id = Event.count
            self.at = None

        def record(self, stream=None):
            self.at = len(rec.ops)
            rec.ops.append(("record", getattr(stream, "name", "default"), self.id))

        def elapsed_time(self, other):
            return float(other.at - self.at)

    class Stream:
        count = 0

        def __init__(self, device=None):
            Stream.count += 1
            self.name = f"s{Stream.count}"

        def wait_event(self, ev):
            rec.ops.append(("wait", self.name, ev.id))

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


class _Lib:
    def __init__(self, rec):
        self.rec = rec

    def layer_fwd(self, dims, Q, K, V, qI, kI, w, o, lse, idx, kpool, ws, stream=None, o_acc=None):
        self.rec.ops.append(("fwd", getattr(stream, "name", "default"), id(o)))

    def layer_bwd(self, dims, Q, K, V, idx, o, lse, dO, dq, dk, dv, ws, stream=None, o_acc=None):
        self.rec.ops.append(("bwd", getattr(stream, "name", "default"), id(dq)))


@pytest.mark.parametrize("with_bwd", [True, False])
@pytest.mark.parametrize("steps", [1, 2, 5])
def test_pipelined_schedule_orders_every_buffer_reuse(monkeypatch, with_bwd, steps):
    rec = _Rec()
    _install(monkeypatch, rec)
    names = ["Q", "K", "V", "q_I", "k_I", "w"] + (["dO"] if with_bwd else [])
    host = {n: torch.randn(4, 3) for n in names}
    d_in = {n: torch.zeros(4, 3) for n in names}
    bufs = types.SimpleNamespace(o=torch.zeros(4, 3), lse=torch.zeros(4), idx=None, kpool=None, ws=None, o_acc=None)
    grads = (torch.zeros(4, 3), torch.zeros(4), torch.zeros(4)) if with_bwd else (None, None, None)
    # the copy-rate measurement after the pipelined run is not part of the schedule
    monkeypatch.setattr(bench, "copy_bandwidth", lambda *a, **kw: {})
    r = bench.end_to_end(_Lib(rec), None, types.SimpleNamespace(L=1000), host, d_in, bufs, *grads, None,
                         torch.cuda.Stream(), types.SimpleNamespace(steps=steps, e2e_steps=steps), with_bwd, 1, "cpu")
    assert r["mode"].startswith("pipelined")
    assert r["steps"] == steps
    ov = r["overlap"]
    assert set(ov) == {"layer_ms_mean", "layer_ms_max", "run_stream_wait_ms_mean", "fill_ms", "drain_ms"}
    assert ov["layer_ms_max"] >= ov["layer_ms_mean"] > 0
    assert (ov["run_stream_wait_ms_mean"] is None) == (steps == 1)
    if steps > 1:
        assert ov["run_stream_wait_ms_mean"] >= 0
    assert r["h2d_bytes_per_step"] == sum(t.numel() * t.element_size() for t in host.values())
    assert all(torch.equal(d_in[n], host[n]) for n in names)

    # The three streams, identified by what is issued on them: input copies are
    # recorded on one stream (plus the start event), layers on another, output
    # copies on the third; on each stream the events come in step order.
    layers = [op for op in rec.ops if op[0] == "fwd"]
    assert len(layers) == steps
    run_stream = layers[0][1]
    records = [op for op in rec.ops if op[0] == "record"]
    start = records[0]
    by_stream = {}
    for op in records[1:]:
        by_stream.setdefault(op[1], []).append(op)
    assert run_stream in by_stream and len(by_stream) == 3
    in_stream = start[1]
    out_stream = next(st for st in by_stream if st not in (in_stream, run_stream))
    in_done = [op[2] for op in by_stream[in_stream]]
    run_done = [op[2] for op in by_stream[run_stream]]
    out_done = [op[2] for op in by_stream[out_stream]]
    assert len(in_done) == len(run_done) == len(out_done) == steps
    if steps >= 3:
        # the two buffer sets alternate
        assert layers[0][2] != layers[1][2] and layers[0][2] == layers[2][2]

    def waits_before(event_id):
        """Waits issued on the event's stream between its previous record and this one."""
        pos = next(i for i, op in enumerate(rec.ops) if op[0] == "record" and op[2] == event_id)
        stream = rec.ops[pos][1]
        out = []
        for op in reversed(rec.ops[:pos]):
            if op[0] == "record" and op[1] == stream:
                break
            if op[0] == "wait" and op[1] == stream:
                out.append(op[2])
        return set(out)

    for i in range(steps):
        w_in, w_run, w_out = waits_before(in_done[i]), waits_before(run_done[i]), waits_before(out_done[i])
        assert in_done[i] in w_run                       # the layer waits for its inputs
        assert run_done[i] in w_out                      # the copy-out waits for the layer
        if i >= 2:
            assert run_done[i - 2] in w_in               # inputs of set i%2 free again
            assert out_done[i - 2] in w_run              # outputs of set i%2 copied out
        else:
            assert not w_in


def test_serial_schedule_runs_every_step(monkeypatch):
    rec = _Rec()
    _install(monkeypatch, rec)
    names = ["Q"]
    host = {"Q": torch.randn(3)}
    d_in = {"Q": torch.zeros(3)}
    calls = []
    ms = bench._e2e_serial(host, names, d_in, [torch.zeros(2), torch.zeros(1)],
                           lambda d, o, lse, g, s: calls.append(s.name), 3, torch.cuda.Stream(), "cpu")
    assert len(calls) == 4                               # one warm-up step, three timed
    assert ms == 0.0 or ms > 0
    assert torch.equal(d_in["Q"], host["Q"])
