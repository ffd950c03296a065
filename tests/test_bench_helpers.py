"""bench.py's host-side helpers on the CPU: the clock record that rejects a
measurement, and the source hash that keeps a recorded ncu traffic figure
only while the attention kernels' code is the one it was taken on."""

import importlib.util
import os
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _clk(sm, smax, reasons):
    return {"sm_mhz": sm, "sm_max_mhz": smax, "reasons": reasons, "samples": 10}


def test_clocks_bad(bench):
    assert not bench.clocks_bad(None)
    assert not bench.clocks_bad(_clk(2070, 2070, []))
    assert not bench.clocks_bad(_clk(1900, 2070, ["sw_power_cap"]))      # kept and noted
    for r in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"):
        assert bench.clocks_bad(_clk(2070, 2070, [r]))
    assert bench.clocks_bad(_clk(1200, 2070, []))                        # stuck low with no reason
    assert not bench.clocks_bad(_clk(1900, 2070, []))                    # within 10 %


def _tree(tmp_path):
    csrc = tmp_path / "stream_speculative_decode_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name in ("attn.cu", "attn_tc.cu", "attn_item.cuh", "tc_ptx.cuh", "tf_internal.cuh"):
        shutil.copy(os.path.join(ROOT, "stream_speculative_decode_gb300", "csrc", name), csrc / name)
    return csrc


def test_source_hash_ignores_comments_only(bench, tmp_path, monkeypatch):
    csrc = _tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_hash()
    with open(csrc / "attn.cu", "a") as f:
        f.write("\n// a comment\n/* and a block\n   comment */\n")
    assert bench.kernel_source_hash() == h0
    with open(csrc / "attn_tc.cu", "a") as f:
        f.write("\nstatic int added_code = 1;\n")
    assert bench.kernel_source_hash() != h0


def test_recorded_traffic_follows_the_hash(bench, tmp_path, monkeypatch):
    _tree(tmp_path)
    (tmp_path / "profiles").mkdir()
    shutil.copy(os.path.join(ROOT, "profiles", "attn_partials_traffic.json"), tmp_path / "profiles")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    # the committed record names the committed sources
    assert bench.recorded_traffic(2) is not None and bench.recorded_traffic(2) > 0
    assert bench.recorded_traffic(1) is None                             # no record for this workload
    with open(tmp_path / "stream_speculative_decode_gb300" / "csrc" / "tf_internal.cuh", "a") as f:
        f.write("\nstatic int changed = 2;\n")
    assert bench.recorded_traffic(2) is None
