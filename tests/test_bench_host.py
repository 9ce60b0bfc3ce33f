"""Host-side pieces of bench.py: per-step statistics, the clock record, and the
rule that a committed ncu traffic figure is reported only while the kernel
source it was taken on is unchanged (comments aside)."""
import json
import os

import pytest

import bench


def test_pct():
    r = bench.pct([1.0, 2.0, 3.0, 4.0, 5.0, 6.0, 7.0, 8.0, 9.0, 10.0])
    assert r["mean"] == 5.5 and r["median"] == 5.5 and r["n"] == 10
    assert r["p10"] == pytest.approx(1.9) and r["p90"] == pytest.approx(9.1)


def _sampler(lines):
    c = bench.ClockSampler(0)
    c.lines = lines
    return c.summary()


def test_clock_summary_reasons():
    s = _sampler(["2070, 2070, Not Active, Not Active, Not Active, Not Active",
                  "2055, 2070, Not Active, Not Active, Not Active, Active",
                  "1980, 2070, Not Active, Not Active, Not Active, Active"])
    assert s["sm_mhz"] == 2055 and s["sm_max_mhz"] == 2070 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"]
    s = _sampler(["1500, 2070, Active, Not Active, Active, Not Active"])
    assert s["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]


def test_clock_summary_unsampled():
    # no nvidia-smi output (or only unparsable lines) is reported as such
    assert _sampler([])["reasons"] == ["unsampled"]
    assert _sampler(["[N/A], [N/A], x, x, x, x", "short"])["sm_mhz"] is None


@pytest.fixture
def fake_root(tmp_path, monkeypatch):
    csrc = tmp_path / "quantized_kv_cache_05_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in set(sum(bench.KERNEL_SOURCES.values(), [])):
        (csrc / f).write_text(f"// {f}\nint x_{f.replace('.', '_')} = 1;  /* value */\n")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return tmp_path


def _write_traffic(root, h, nbytes=123456789):
    entry = {"gqa_fp8_L32768": {"source_hash": h, "dram_bytes_per_launch": nbytes}}
    (root / "profiles" / "traffic.json").write_text(json.dumps(entry))


def test_traffic_reported_only_for_the_captured_source(fake_root):
    h = bench.kernel_source_hash("decode")
    _write_traffic(fake_root, h)
    assert bench.ncu_traffic("gqa_fp8_L32768", "decode") == 123456789.0
    # another workload has no entry
    assert bench.ncu_traffic("nvfp4_L32768", "decode") is None
    # a comment or whitespace edit keeps the figure
    f = fake_root / "quantized_kv_cache_05_gb300" / "csrc" / "kvq_decode.cu"
    f.write_text(f.read_text().replace("/* value */", "/* another comment */") + "\n\n// more\n")
    assert bench.kernel_source_hash("decode") == h
    assert bench.ncu_traffic("gqa_fp8_L32768", "decode") == 123456789.0
    # a code edit voids it
    f.write_text(f.read_text().replace("= 1;", "= 2;"))
    assert bench.kernel_source_hash("decode") != h
    assert bench.ncu_traffic("gqa_fp8_L32768", "decode") is None


def test_traffic_missing_or_broken_file(fake_root):
    assert bench.ncu_traffic("gqa_fp8_L32768", "decode") is None
    (fake_root / "profiles" / "traffic.json").write_text("{not json")
    assert bench.ncu_traffic("gqa_fp8_L32768", "decode") is None


def test_committed_traffic_entries_name_their_capture():
    # every committed entry says what it was captured with (the figures it
    # carries are checked against the live source hash at bench time)
    with open(os.path.join(os.path.dirname(os.path.dirname(__file__)), "profiles",
                           "traffic.json")) as f:
        d = json.load(f)
    assert d, "no traffic entries"
    for name, e in d.items():
        assert e["dram_bytes_per_launch"] == e["dram_read_bytes"] + e["dram_write_bytes"], name
        assert e["command"].startswith("ncu ") and "--clock-control none" in e["command"], name
        assert len(e["source_hash"]) == 16, name
