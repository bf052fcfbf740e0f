"""Host logic of bench.py that needs no GPU: the committed ncu counters are used
only while the kernel source they were taken from is unchanged, and the
reference arm's sample sizing stays inside its time budget."""
import importlib.util
import json
from pathlib import Path


ROOT = Path(__file__).resolve().parent.parent


def _bench():
    spec = importlib.util.spec_from_file_location("bench_host_mod", ROOT / "bench.py")
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def test_committed_counters_match_current_sources():
    """Every committed counter is keyed by the hash of the source it was taken
    from; the files in the tree must still hash to those keys (otherwise the
    bench would report null traffic / no ALU roofline)."""
    b = _bench()
    traffic = json.loads((ROOT / "profiles" / "ncu_traffic.json").read_text())
    for e in traffic["entries"]:
        assert e["kernel_source_sha256"] == b.kernel_source_sha()
        assert b.ncu_traffic(e["workload"], e["layout"]) == e["dram_bytes_per_launch"]
    inst = json.loads((ROOT / "profiles" / "ncu_inst.json").read_text())
    for e in inst["entries"]:
        assert e["header_sha256"] == b.header_sha(e["header"]), e["kernel"]
    assert b.ncu_inst("lookup_decode_reduce_kernel", 196608, 1024, 4, 24) is not None
    assert b.ncu_encoder_inst_per_row(1024, 4) is not None


def test_counters_ignored_for_other_shapes_or_sources(monkeypatch):
    b = _bench()
    assert b.ncu_traffic("no_such_workload", "aos") is None
    assert b.ncu_inst("lookup_decode_reduce_kernel", 1000, 1024, 4, 24) is None
    assert b.ncu_encoder_inst_per_row(256, 4) is None
    # a source that no longer hashes to the committed key disables the counter
    monkeypatch.setattr(b, "header_sha", lambda name: "0" * 64)
    assert b.ncu_inst("lookup_decode_reduce_kernel", 196608, 1024, 4, 24) is None
    assert b.ncu_encoder_inst_per_row(1024, 4) is None


def test_roofline_arithmetic():
    """achieved / peak for the HBM line: bytes per lookup x lookups / time."""
    b = _bench()
    from trellis_row_decode_gb300 import synth
    w = synth.WORKLOADS["deepseek_prefill"]
    assert w.algorithmic_bytes_per_lookup() == 258 + 2 * 1024 + 8
    assert w.n_lookups == 196608
    assert abs(b.ISSUE_PEAK_WARP_INST_S - 152 * 4 * 2.07e9) < 1.0
    peak, kind = b.measured_peaks()
    assert peak > 0 and kind in ("measured", "fallback")


def test_oracle_sample_size_bounds():
    """The calibrated prefix never exceeds the replay and never falls below the
    calibration prefix; it scales with the time budget."""
    b = _bench()
    calls = []

    def run(m):                                   # 1 microsecond per lookup
        calls.append(m)
        return m * 1e-6

    assert b.oracle_sample_size(run, 196608, 0.01, 2048) == 10000
    assert b.oracle_sample_size(run, 196608, 100.0, 2048) == 196608
    assert b.oracle_sample_size(run, 196608, 1e-6, 2048) == 2048
    assert b.oracle_sample_size(run, 100, 1.0, 2048) == 100
    assert calls[0] == 2048
