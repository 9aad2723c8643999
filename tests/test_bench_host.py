"""Host-side pieces of bench.py that need no GPU: the clock record taken
during the timed region, and the ncu traffic record lookup (a record whose
source hash no longer matches its kernel's sources is not used)."""
import hashlib
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_clock_summary_median_max_and_reasons():
    c = bench.ClockSampler("0")
    c.lines = [
        "0, 2070, 2070, 812.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2070, 1390.1, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 905.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, [N/A], 2070, 905.0, 0x0, Not Active, Not Active, Not Active, Not Active",  # unreadable: skipped
        "garbage",
    ]
    s = c.summary()
    assert s == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}


def test_clock_summary_flags_thermal_and_empty_record():
    c = bench.ClockSampler("0")
    c.lines = ["0, 1500, 2070, 1400.0, 0x48, Active, Not Active, Active, Not Active"]
    assert c.summary()["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    c.lines = []
    assert c.summary() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}


def test_recorded_traffic_requires_matching_source_hash(tmp_path, monkeypatch):
    src = tmp_path / "k.cu"
    src.write_bytes(b"__global__ void k() {}\n")
    h = hashlib.sha256(src.read_bytes()).hexdigest()
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "k.txt").write_text(f"# k\nsource_sha256: {h}\nkernel: k\ndram_bytes_per_launch: 12345\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench._recorded_traffic("k", [str(src)]) == 12345.0
    src.write_bytes(b"__global__ void k() { }\n")  # the kernel changed since the counters were taken
    assert bench._recorded_traffic("k", [str(src)]) is None
    assert bench._recorded_traffic("missing", [str(src)]) is None


def test_all_cores_oracle_timing_spawns_one_process_per_core():
    """The all-cores CPU baseline: one spawned process per usable core, each
    timing whole layer decodes of the oracle; the per-decode time is the wall
    time of all of them divided by the decodes."""
    s, n_proc, n_dec = bench.time_oracle_all_cores(0.1, reps=1, n_layers=1)
    assert n_proc == len(os.sched_getaffinity(0)) and n_dec == n_proc
    assert 0 < s < 60


def test_union_fractions_by_hand():
    """Two routed experts (one 64-neuron group each, top-1), one shared
    group: expert 0 has tokens 0, 1, 2 (live neurons {0,1}, {1,2}, {40}),
    expert 1 has token 3 (live {63}); the shared group's tokens have live
    sets {0}, {0}, {5}, {6}.  Tiles of 2 tokens: expert 0's tiles have
    unions {0,1,2} and {40}, expert 1's {63}: (3 + 1 + 1) / 3 / 64; the
    shared tiles {0} and {5,6}: (1 + 2) / 2 / 64.  Tiles of 128: one tile
    per expert: (4 + 1) / 2 / 64 routed, 3 / 64 shared."""
    import numpy as np
    idx = np.array([[0], [0], [0], [1]], dtype=np.int32)
    bit = lambda *ns: sum(1 << n for n in ns)
    shared = [bit(0), bit(0), bit(5), bit(6)]
    routed = [bit(0, 1), bit(1, 2), bit(40), bit(63)]
    words = np.array([[s, r] for s, r in zip(shared, routed)], dtype=np.uint64).view(np.int64)
    out = bench.union_fractions(idx, words, 64, 64, tiles=(2, 128))
    assert out["tile2"]["routed"] == round((3 + 1 + 1) / 3 / 64, 4)
    assert out["tile2"]["shared"] == round((1 + 2) / 2 / 64, 4)
    assert out["tile128"]["routed"] == round((4 + 1) / 2 / 64, 4)
    assert out["tile128"]["shared"] == round(3 / 64, 4)
