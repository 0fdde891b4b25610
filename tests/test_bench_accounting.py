"""Host-side accounting of bench.py, on CPU: the algorithmic bytes behind every
roofline figure, the rotating input sets, the config object both arms print,
the lookup of committed ncu traffic and the parsing of the clock samples.

The byte counts are worked out by hand from the definitions (read each token
row once, write every live copy; read every live row and write each token
row once; the routing arrays), so a change in bench.py's formulas shows here.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads as W  # noqa: E402

# Every copy is live in the five workloads: no masked ids, and in the decode
# capacity buffer no expert gets more than its 128 rows (8 distinct experts a
# token, 128 tokens).
EXPECTED = {
    # tiny: T=128 H=1024 k=4, bf16.  128*1024*2 + 512*1024*2; 512*1024*2 + 128*1024*2 + 128*4*8
    "tiny": dict(dispatch=1_310_720, combine=1_314_816),
    # decode: T=128 H=7168 k=8, fp8.  128*7168*2 + 1024*7168 + 1024*56*4; 1024*7168*2 + 128*7168*2 + 128*8*8;
    # layout 2*4*1024 + 8*32768 + 4*(2*256 + 2*32 + 2)
    "decode": dict(layout=272_648, dispatch=9_404_416, combine=16_523_264),
    # prefill: T=4096 H=7168 k=8, bf16
    "prefill": dict(dispatch=528_482_304, combine=528_744_448),
    # skewed: T=8192 H=7168 k=8, fp8
    "skewed": dict(dispatch=601_882_624, combine=1_057_488_896),
    # group-limited: T=16384 H=4096 k=8, bf16; layout 2*4*131072 + 8*131072 + 4*(2*128 + 2*8 + 2)
    "grouped": dict(layout=2_098_248, dispatch=1_207_959_552, combine=1_209_008_128),
    # unbalanced: the skewed shape with milder routing, so the same bytes
    "unbalanced": dict(dispatch=601_882_624, combine=1_057_488_896),
}


@pytest.mark.parametrize("name", sorted(EXPECTED))
def test_algorithmic_bytes_by_hand(name):
    wl = W.WORKLOADS[name]
    got = bench.algorithmic_bytes(wl, wl.T * wl.k)
    for stage, want in EXPECTED[name].items():
        assert got[stage] == want, (name, stage, got[stage], want)


@pytest.mark.parametrize("name,n_sets", [("tiny", 196), ("decode", 20), ("prefill", 1), ("skewed", 1),
                                         ("grouped", 1), ("unbalanced", 1)])
def test_rotating_sets_cover_four_l2(name, n_sets):
    wl = W.WORKLOADS[name]
    step = sum(bench.algorithmic_bytes(wl, wl.T * wl.k).values())
    n = bench.n_rotating_sets(step)
    assert n == n_sets
    assert n * step >= 4 * bench.L2_BYTES


@pytest.mark.parametrize("name,partition,expert", [("skewed", 4.06, 29.7), ("unbalanced", 1.50, 5.59)])
def test_skewed_routing_imbalance(name, partition, expert):
    """The two Zipf workloads' imbalance with seed 0: max/mean copies per
    partition and per expert."""
    d = W.make(name)
    st = W.load_stats(d["wl"], d["topk_idx"])
    assert st["partition_max_over_mean"] == pytest.approx(partition, abs=0.02)
    assert st["expert_max_over_mean"] == pytest.approx(expert, abs=0.02)


def test_config_names_the_workload_and_its_layout():
    for name, wl in W.WORKLOADS.items():
        cfg = bench.workload_config(wl, 1000, 1)
        assert set(cfg) == {"workload", "description", "T", "H", "E", "top_k", "partitions", "layout",
                            "capacity", "payload", "step_bytes", "l2", "parallelism"}
        assert cfg["workload"] == name
        assert cfg["payload"] == ("fp8_e4m3" if wl.fp8 else "bf16")
        assert cfg["layout"] == ("capacity" if wl.mode == W.CAPACITY else "packed")
        assert cfg["parallelism"] == "replicas x1"


def test_traffic_is_read_only_for_the_sources_it_was_taken_on(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.txt").write_text(
        "# comment line\n"
        "grouped dispatch 1144632960 aaaaaaaaaaaaaaaa\n"
        "grouped combine 1195906048 bbbbbbbbbbbbbbbb   # trailing comment\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_digest", lambda k: {"dispatch": "aaaaaaaaaaaaaaaa",
                                                                  "combine": "cccccccccccccccc"}[k])
    assert bench.ncu_traffic("grouped", "dispatch") == 1144632960.0
    assert bench.ncu_traffic("grouped", "combine") is None        # taken on other sources
    assert bench.ncu_traffic("decode", "dispatch") is None        # no line for it


class _Proc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0

    def kill(self):
        pass


class _Thread:
    def join(self, timeout=None):
        pass


def _sampler(lines):
    cs = bench.ClockSampler(0)
    cs.proc, cs.thread, cs.lines = _Proc(), _Thread(), list(lines)
    return cs


def test_clock_samples_under_load_and_their_reasons():
    idle = "600, 2070, 100.0, 0x1, Not Active, Not Active, Not Active, Not Active"
    r = _sampler([
        idle,
        "2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "1500, 2070, 950.0, 0x8, Active, Not Active, Not Active, Not Active",
        "garbage line",
        idle,
    ]).stop()
    assert r["samples"] == 2                      # the idle samples are left out
    assert r["sm_mhz"] == pytest.approx(1785.0)   # median of the loaded ones
    assert r["sm_max_mhz"] == 2070.0
    assert r["reasons"] == ["hw_slowdown"]


def test_power_cap_is_reported_and_clean_runs_report_nothing():
    r = _sampler(["1900, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active"] * 3).stop()
    assert r["reasons"] == ["sw_power_cap"]
    r = _sampler(["2070, 2070, 800.0, 0x0, Not Active, Not Active, Not Active, Not Active"] * 3).stop()
    assert r["reasons"] == [] and r["sm_mhz"] == 2070.0
    assert bench.ClockSampler(0).stop() is None   # never started: no record


def test_per_call_percentiles():
    ms = [i / 1000 for i in range(1, 101)]        # 1 .. 100 µs
    p = bench.percentiles_us(ms)
    assert p["us_p10"] == pytest.approx(10.9) and p["us_p90"] == pytest.approx(90.1)
    assert bench.percentiles_us([0.005]) == dict(us_p10=5.0, us_p90=5.0)
    assert bench.percentiles_us([]) == {}
