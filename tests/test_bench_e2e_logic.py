"""Host logic of bench.py's end-to-end leg, on the CPU with stand-ins for CUDA streams and events.

Checks what the timed region copies per step (bytes host->device and device->host), that each
prefill waits for its own layer's copies, and that the decode launches of a step are preceded by
one copy of the step's decode inputs on a stream of their own, with no copy on the compute stream
between decode launches."""
import contextlib
import types

import pytest

import synth

torch = pytest.importorskip("torch")


class _Event:
    def __init__(self, log, enable_timing=False):
        self.log, self.recorded_on = log, None

    def record(self, stream=None):
        self.recorded_on = stream
        self.log.append(("record", id(self), stream.name if stream is not None else None))

    def elapsed_time(self, other):
        return 10.0


class _Stream:
    def __init__(self, log, name):
        self.log, self.name = log, name

    def wait_event(self, ev):
        self.log.append(("wait", self.name, id(ev)))


@pytest.fixture
def cpu_cuda(monkeypatch):
    log = []
    current = [None]
    counter = [0]

    def make_stream(dev=None):
        counter[0] += 1
        return _Stream(log, f"s{counter[0]}")

    @contextlib.contextmanager
    def stream_ctx(s):
        old, current[0] = current[0], s
        try:
            yield
        finally:
            current[0] = old

    empty_like, empty, copy = torch.empty_like, torch.empty, torch.Tensor.copy_

    def copy_(self, src, non_blocking=False):
        log.append(("copy", current[0].name if current[0] is not None else None, src.nbytes))
        return copy(self, src)

    monkeypatch.setattr(torch.cuda, "Stream", make_stream)
    monkeypatch.setattr(torch.cuda, "Event", lambda enable_timing=False: _Event(log, enable_timing))
    monkeypatch.setattr(torch.cuda, "stream", stream_ctx)
    monkeypatch.setattr(torch.cuda, "synchronize", lambda *a, **k: None)
    monkeypatch.setattr(torch.Tensor, "pin_memory", lambda self: self)
    monkeypatch.setattr(torch, "empty_like", lambda x, **k: empty_like(x, **{a: b for a, b in k.items() if a != "device"}))
    monkeypatch.setattr(torch, "empty", lambda *a, **k: empty(*a, **{x: y for x, y in k.items() if x != "device"}))
    monkeypatch.setattr(torch.Tensor, "copy_", copy_)
    return log, make_stream


class _Cache:
    def __init__(self, w, layer, log):
        self.w, self.layer, self.log = w, layer, log

    def reset(self):
        pass

    def prefill_quantize(self, k, v, stream=None):
        w = self.w
        assert tuple(k.shape) == (w.batch, w.kv_heads, w.prefill_tokens, w.head_dim) and v.shape == k.shape
        self.log.append(("prefill", self.layer, stream.name))

    def decode_step(self, kn, vn, q, out, stream=None):
        w = self.w
        assert tuple(kn.shape) == (w.batch, w.kv_heads, w.head_dim) and vn.shape == kn.shape
        assert tuple(q.shape) == (w.batch, w.q_heads, w.head_dim) and out.shape == q.shape
        self.log.append(("decode", self.layer, stream.name))


class _Dist:
    local_rank, rank, world = 0, 0, 1

    def barrier(self):
        pass

    def max(self, x):
        return x

    def sum(self, x):
        return x


@pytest.mark.parametrize("batch", [1, 6])
def test_e2e_copies_and_their_order(cpu_cuda, batch):
    import bench
    log, make_stream = cpu_cuda
    w = synth.WORKLOADS[0].scaled(batch=batch, kv_heads=2, q_heads=4, prefill_tokens=256, decode_steps=3)
    L = 3
    compute = make_stream()
    res = bench.run_e2e(types.SimpleNamespace(e2e_steps=2), w, _Dist(), [_Cache(w, l, log) for l in range(L)],
                        compute)
    D, T0, S = w.head_dim, w.prefill_tokens, w.decode_steps
    prompt = 2 * w.batch * w.kv_heads * T0 * D * 2
    decode_inputs = S * w.batch * (2 * w.kv_heads + w.q_heads) * D * 2
    assert res["h2d_bytes_per_step"] == L * prompt + decode_inputs
    assert res["d2h_bytes_per_step"] == L * S * w.batch * w.q_heads * D * 2
    # each prefill follows the copies of its own prompt, made on streams other than the compute stream
    prefills = [i for i, x in enumerate(log) if x[0] == "prefill"]
    assert len(prefills) == 3 * L  # the untimed first step and the two timed ones
    prev = 0
    for i in prefills:
        copies = [x for x in log[prev:i] if x[0] == "copy"]
        prompt_copies = [x for x in copies if x[1] != compute.name]
        assert sum(x[2] for x in prompt_copies) >= prompt
        prev = i
    # a step's decode launches: preceded by one copy of its decode inputs on a stream of their own,
    # with nothing copied between the first and the last launch
    decodes = [i for i, x in enumerate(log) if x[0] == "decode"]
    assert len(decodes) == 3 * L * S
    for k in range(0, len(decodes), L * S):
        first, last = decodes[k], decodes[k + L * S - 1]
        assert not any(x[0] == "copy" for x in log[first:last + 1])
        assert all(log[i][2] == compute.name for i in decodes[k:k + L * S])
        before = [x for x in log[:first] if x[0] == "copy"][-3:]
        assert all(x[1] not in (None, compute.name) for x in before)
        assert sum(x[2] for x in before) == decode_inputs
