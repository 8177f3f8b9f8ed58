"""The latency table measured with the library's kernels on the GPU, and the
simulation driver end to end."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from chunked_prefill_extend_gb300 import cpe
    return cpe


def test_table_measures_each_shape_once(lib):
    from chunked_prefill_extend_gb300.latency import KernelLatencyTable
    t = KernelLatencyTable(32, 8, 128, reps=3, warmup=1)
    pre = t.key(False, 2, 1024, 8192)
    dec = t.key(True, 64, 1, 5000)
    t.prefetch([pre, dec, pre])
    assert t.measured == 2
    n0 = lib.cpe_launch_count()
    ms_pre, ms_dec = t(False, 2, 1024, 8192), t(True, 64, 1, 4500)  # same decode bucket
    assert lib.cpe_launch_count() == n0 and t.measured == 2  # replayed, not re-run
    assert ms_pre > 0 and ms_dec > 0
    assert t.records[pre].launches >= 3 and t.records[dec].launches >= 2
    st, _ = lib.cpe_get_device_status()
    assert st == lib.CPE_OK


def test_simulate_driver(lib):
    from chunked_prefill_extend_gb300 import simulate
    out = simulate.main(["--input-len", "8192", "--chunk", "2048", "--output-len", "8", "--concurrency", "4",
                         "--reps", "2"])
    assert out["prefill_num_chunks"] == 4 and out["measured_shapes"] == out["forward_shapes"]
    assert 0 < out["ttft_ms"] <= out["makespan_ms"] and out["tpot_ms"] > 0
    assert out["output_throughput"] == pytest.approx(1000.0 * 4 * 8 / out["makespan_ms"])
