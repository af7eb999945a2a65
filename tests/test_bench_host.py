"""Host-side pieces of bench.py that need no GPU: the oracle arm's JSON line and
the CPU-baseline sample, which must never credit the oracle with more tokens
than the batch holds."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from sparse_mixture_experts_topk_gb300 import workloads as W  # noqa: E402


@pytest.mark.parametrize("T", [1, 3, 64, 100])
def test_cpu_baseline_counts_only_the_batch(T):
    w = W.small("cb", T=T, H=64, E=4, K=2, F=32, dtype=W.F32)
    inp = W.generate(w)
    cb = bench.cpu_baseline(inp, 0.05)
    n = int(cb["sample"].split("first ")[1].split(" of ")[0])
    assert 0 < n <= T
    assert f"of {T} tokens" in cb["sample"]
    assert cb["kind"] == "oracle" and cb["unit"] == "tokens/s" and cb["value"] > 0


def test_oracle_rate_rejects_more_tokens_than_the_batch():
    w = W.small("cb", T=2, H=64, E=4, K=2, F=32, dtype=W.F32)
    inp = W.generate(w)
    with pytest.raises(AssertionError):
        bench.oracle_rate(inp, bench.widen_inputs(inp), 3)


def test_reference_arm_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny", "--steps", "3", "--warmup", "3"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["steps"] == 3 and d["warmup"] == 3
    assert d["higher_is_better"] is True and d["unit"] == "tokens/s" and d["value"] > 0
    n = int(d["cpu_baseline"]["sample"].split("first ")[1].split(" of ")[0])
    assert 0 < n <= W.WORKLOADS["tiny"].T
    # the same config keys and values the GPU arm prints for this workload
    w = W.WORKLOADS["tiny"]
    assert d["config"] == bench.config_of(w, 1, w.T * w.K, w.E, "auto")
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]


def test_ncu_traffic_follows_the_kernel_sources():
    """Measured DRAM bytes are reported only for the kernel sources they were
    taken on: an entry is keyed by the hash of its kernel's files."""
    assert bench.ncu_traffic("no such workload") is None
    stream = bench.ncu_traffic("decode8", bench.STREAM_SOURCES)
    if stream is not None:
        assert stream["ffn"] > 0
        # the same entry checked against the tensor-core GEMM's files does not match
        assert bench.ncu_traffic("decode8", bench.GEMM_SOURCES) is None
    gemm = bench.ncu_traffic("prefill", bench.GEMM_SOURCES)
    if gemm is not None:
        assert bench.ncu_traffic("prefill", bench.STREAM_SOURCES) is None


def test_tensor_peak_follows_the_clock_record():
    """Burst peak when no power cap was seen; burst scaled by the sampled SM
    clock when it was."""
    p, why = bench.tensor_peak(1900.0, 1700.0, 2000.0, {"reasons": [], "sm_mhz": 2000.0}, "measured")
    assert p == 1900.0 and "burst" in why
    p, why = bench.tensor_peak(1900.0, 1700.0, 2000.0, {"reasons": ["sw_power_cap"], "sm_mhz": 1800.0}, "measured")
    assert p == pytest.approx(1710.0) and "1800" in why
    p, _ = bench.tensor_peak(1900.0, 1700.0, 2000.0, {"reasons": ["sw_power_cap"], "sm_mhz": None}, "measured")
    assert p == 1700.0
    p, _ = bench.tensor_peak(1900.0, 1700.0, 2000.0, None, "measured")
    assert p == 1900.0
