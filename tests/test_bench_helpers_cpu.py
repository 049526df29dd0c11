"""bench.py's host-side helpers: the kernel-source hash that keeps a recorded
DRAM-traffic figure tied to the code it was measured on, and the summary of
the clock samples taken during the timed region."""
import json
import os
import shutil

import pytest

import bench


@pytest.fixture
def tree(tmp_path, monkeypatch):
    """A copy of the kernel sources and the traffic record under a temporary root."""
    src = os.path.join(bench.ROOT, "mla_latent_kv_05_gb300", "csrc")
    dst = tmp_path / "mla_latent_kv_05_gb300" / "csrc"
    dst.mkdir(parents=True)
    for name in bench.KERNEL_SOURCES:
        shutil.copy(os.path.join(src, name), dst / name)
    (tmp_path / "profiles").mkdir()
    shutil.copy(os.path.join(bench.ROOT, "profiles", "decode_dram_traffic.json"), tmp_path / "profiles")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return tmp_path


def test_comment_edits_keep_the_hash_and_code_edits_change_it(tree):
    h0 = bench.kernel_source_hash()
    f = tree / "mla_latent_kv_05_gb300" / "csrc" / "decode.cu"
    text = f.read_text()
    f.write_text("// a new comment line\n" + text.replace("\n", "  // trailing note\n", 3) + "\n\n")
    assert bench.kernel_source_hash() == h0
    edited = text.replace("kModeF16<kMode> ? 15.0f : 16.0f", "kModeF16<kMode> ? 15.0f : 17.0f")
    assert edited != text
    f.write_text(edited)
    assert bench.kernel_source_hash() != h0
    assert bench.recorded_traffic(3, "bf16") is None           # stale counters are not reported


def test_recorded_traffic_is_per_workload_and_kind(tree):
    assert bench.recorded_traffic(3, "bf16") is not None
    assert bench.recorded_traffic(3, "fp8") is None              # no such record
    assert bench.recorded_traffic(42, "bf16") is None
    os.unlink(tree / "profiles" / "decode_dram_traffic.json")
    assert bench.recorded_traffic(3, "bf16") is None


def _summary(tmp_path, lines):
    s = bench.ClockSampler(0)
    s.proc = object()                                            # as if nvidia-smi had run
    s.path = str(tmp_path / "clocks.csv")
    with open(s.path, "w") as f:
        f.write("\n".join(lines) + "\n")
    return s.summary()


def test_clock_summary_takes_the_median_under_load_and_names_active_reasons(tmp_path):
    idle = "0, 345, 2070, 120.5, 0x0, Not Active, Not Active, Not Active, Not Active"
    busy = "0, {}, 2070, 900.0, 0x4, Not Active, Not Active, Not Active, {}"
    got = _summary(tmp_path, [idle, busy.format(2070, "Not Active"), busy.format(1980, "Active"),
                              busy.format(2070, "Not Active"), "garbage line", idle])
    assert got["sm_mhz"] == 2070.0 and got["sm_max_mhz"] == 2070.0
    assert got["reasons"] == ["sw_power_cap"]
    assert got["samples"] == 5 and got["samples_under_load"] == 3


def test_clock_summary_flags_thermal_slowdown_and_handles_no_samples(tmp_path):
    hot = "0, 1500, 2070, 1300.0, 0x40, Not Active, Active, Not Active, Not Active"
    assert _summary(tmp_path, [hot])["reasons"] == ["hw_thermal_slowdown"]
    assert _summary(tmp_path, ["no data"])["reasons"] == ["no samples"]
    s = bench.ClockSampler(0)
    assert s.summary()["reasons"] == ["nvidia-smi unavailable"]
