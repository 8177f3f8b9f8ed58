"""Host-side pieces of the benchmark (no GPU): the algorithmic-work formula,
the code hash and traffic lookup behind `roofline.traffic`, the L2 rule and
the config keys the main line and the reference arm share."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from chunked_prefill_extend_gb300 import workloads as W  # noqa: E402
import oracle  # noqa: E402


@pytest.mark.parametrize("n,c", [(4000, 512), (131072, 1024), (517, 128), (1, 16)])
def test_chunk_flops_sum_to_one_shot_causal_work(n, c):
    """Summed over a request's rounds, E_t P_t + E_t (E_t + 1) / 2 counts every
    (query, key) pair with key <= query once: N (N + 1) / 2, the one-shot
    causal prefill (SGLang article, resumable extends: the rounds compute the
    same o_i as one prefill)."""
    d, h = 128, 32
    total = sum(bench.chunk_flops(d, h, ch.prefix_len, ch.query_len) for ch in oracle.plan_chunks(n, 0.0, c))
    assert total == pytest.approx(4.0 * d * h * n * (n + 1) / 2.0, rel=1e-12)


def test_code_hash_ignores_comments_and_blank_lines(tmp_path):
    a = tmp_path / "a.cu"
    a.write_text("int f() {  // one\n  return 1;\n}\n")
    b = tmp_path / "b.cu"
    b.write_text("// a new comment\nint f() {  // two\n\n  return 1;   \n}\n")
    c = tmp_path / "c.cu"
    c.write_text("int f() {\n  return 2;\n}\n")
    assert bench.code_hash(str(a)) == bench.code_hash(str(b))
    assert bench.code_hash(str(a)) != bench.code_hash(str(c))


def _fake_tree(tmp_path, kernel_text, recorded_hash):
    csrc = tmp_path / "chunked_prefill_extend_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "extend_tc.cu").write_text(kernel_text)
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "extend_tc_kernel_prefill-128k-c1024.md").write_text(
        "summary\n\ntraffic-bytes-per-launch: 400 | captured-launch-flops: 1000 | "
        f"extend_tc.cu-code-sha256-16: {recorded_hash}\n")
    return csrc / "extend_tc.cu"


def test_profiled_traffic_scales_by_work_and_turns_null_when_the_kernel_changed(tmp_path, monkeypatch):
    kernel = _fake_tree(tmp_path, "void k() {}\n", "0" * 16)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic(500.0) is None  # recorded hash is not the file's
    h = bench.code_hash(str(kernel))
    (tmp_path / "profiles" / "extend_tc_kernel_prefill-128k-c1024.md").write_text(
        f"traffic-bytes-per-launch: 400 | captured-launch-flops: 1000 | extend_tc.cu-code-sha256-16: {h}\n")
    assert bench.profiled_traffic(500.0) == pytest.approx(200.0)
    kernel.write_text("void k() { return; }\n")  # a code change: the counters no longer apply
    assert bench.profiled_traffic(500.0) is None


def test_l2_rule():
    assert bench.l2_text(W.CONFIGS["prefill-4000-c512"]).startswith("flushed")
    assert bench.l2_text(W.CONFIGS["fp32-512"]).startswith("flushed")
    assert bench.l2_text(W.CONFIGS["prefill-128k-c1024"]).startswith("inputs larger than L2")
    assert bench.l2_text(W.CONFIGS["prefill-32k-hit50"]).startswith("inputs larger than L2")


class _Args:
    input_len = 0
    decode_rows = 0
    rounds = ""


@pytest.mark.parametrize("name", sorted(W.CONFIGS))
def test_workload_config_keys(name):
    """The main line and the reference arm both build `config` with this
    function, so the two lines carry the same keys and values."""
    cfg = bench.workload_config(name, _Args(), 1)
    assert set(cfg) == {"workload", "l2", "parallelism"}
    assert cfg["workload"].startswith(name + ": ")
    assert cfg["parallelism"] == "replicas x1"
