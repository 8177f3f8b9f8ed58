"""The forward-shape latency table and the three-phase replay (host logic;
the GPU measurement itself is covered in the gpu-marked tests)."""
import pytest

from chunked_prefill_extend_gb300 import cpe
from chunked_prefill_extend_gb300.latency import ForwardLatencyRecord, ForwardShapeKey, KernelLatencyTable, \
    simulate_with_table


class FakeTable(KernelLatencyTable):
    """Deterministic 'measurements' and a settable amount of free memory."""

    def __init__(self, free=1 << 50, **kw):
        super().__init__(32, 8, 128, device="cpu", **kw)
        self.free = free
        self.calls = []

    def free_bytes(self):
        return self.free

    def _measure(self, k):
        self.calls.append(k)
        self.measured += 1
        ms = (0.3 + 1e-5 * k.model_concurrency * k.seq_len) if k.is_decode else \
             (0.6 + 1e-8 * k.model_concurrency * k.query_len * k.seq_len)
        return ForwardLatencyRecord(ms, self.bytes_needed(k), 3)


def _plan(n, c):
    chunks, _, _ = cpe.cpe_plan_chunks(n, 0.0, c)
    return [(x.query_len, x.seq_len) for x in chunks]


@pytest.mark.parametrize("n,c,N,O", [(32768, 4096, 16, 64), (4000, 512, 8, 20), (10000, 4096, 1, 1),
                                     (131072, 1024, 3, 5)])
def test_replay_equals_step_by_step_calls(n, c, N, O):
    """Dry run, prefetch, replay gives the same result as asking the latency
    model at every step, and measures each unique shape once."""
    t1 = FakeTable()
    a = simulate_with_table(t1, _plan(n, c), N, O, c)
    t2 = FakeTable()
    b = cpe.cpe_simulate_requests(_plan(n, c), N, O, c, lambda *x: t2._measure(t2.key(*x)).latency_ms)
    for k in ("ttft", "tpot", "makespan", "steps", "first_token_time", "finish_time"):
        assert a[k] == b[k]
    assert t1.measured == len(set(t1.calls)) == a["forward_shapes"]
    assert len(t2.calls) == a["forward_calls"] >= a["forward_shapes"]


def test_long_prompt_has_one_prefill_shape_per_chunk():
    """A 128k prompt in 1k chunks: 128 prefill shapes, however many requests
    (the table section's 128 * concurrency -> 128 example)."""
    t = FakeTable()
    simulate_with_table(t, _plan(131072, 1024), 8, 1, 1024)
    pre = [k for k in t.records if not k.is_decode]
    assert len(pre) == 128 and {k.model_concurrency for k in pre} == {1}


def test_keys_separate_lengths_and_bucket_decode_context():
    t = FakeTable()
    assert t.key(False, 2, 1024, 5000) == ForwardShapeKey(False, 2, 1024, 5000)
    assert t.key(False, 2, 1024, 5000) != t.key(False, 2, 512, 5000) != t.key(False, 2, 1024, 5001)
    assert t.key(True, 7, 1, 2049) == t.key(True, 7, 1, 4096) == ForwardShapeKey(True, 7, 1, 4096)
    assert t.key(True, 7, 1, 4097) == ForwardShapeKey(True, 7, 1, 6144)


def test_prefetch_stops_at_the_first_shape_that_does_not_fit():
    t = FakeTable()
    keys = [ForwardShapeKey(False, 1, 1024, 2048), ForwardShapeKey(False, 64, 4096, 1 << 20),
            ForwardShapeKey(False, 1, 1024, 4096)]
    t.free = t.bytes_needed(keys[0]) + t.memory_reserve_bytes + 1
    t.prefetch(keys)
    assert t.calls == [keys[0]] and t.memory_exceeded_key == keys[1]
    with pytest.raises(RuntimeError):
        t.get(keys[1])
