"""Host-side logic of bench.py without a GPU: the whole-job rate, the DRAM-traffic lookup tied to
the attention kernel's source hash, and the parsing of the clock samples taken during the
timed region."""

import hashlib
import os

import pytest

import bench


def test_whole_job_rate_counts_every_replica():
    assert bench.whole_job_rate(1, 33720, 3, 2.0) == pytest.approx(33720 * 3 / 2.0)
    assert bench.whole_job_rate(4, 1000, 2, 1.0) == pytest.approx(8000.0)


def test_max_over_ranks_without_a_group_is_identity():
    assert bench.max_over_ranks(1.25) == 1.25


def _fake_tree(tmp_path, src: bytes, sha: str, bytes_, rows):
    import json

    (tmp_path / "profiles").mkdir()
    (tmp_path / "joint_video_audio_block_b300" / "csrc").mkdir(parents=True)
    (tmp_path / "joint_video_audio_block_b300" / "csrc" / "attention.cu").write_bytes(src)
    (tmp_path / "profiles" / "attention_traffic.json").write_text(json.dumps({
        "rows": rows, "traffic_bytes_per_launch": bytes_, "source_sha256": sha,
        "source": "joint_video_audio_block_b300/csrc/attention.cu"}))


def test_attention_traffic_scales_by_rows_when_the_source_matches(tmp_path, monkeypatch):
    src = b"// kernel source\n"
    _fake_tree(tmp_path, src, hashlib.sha256(src).hexdigest(), 1000, 100)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench._attention_traffic(100) == pytest.approx(1000.0)
    assert bench._attention_traffic(250) == pytest.approx(2500.0)


def test_attention_traffic_is_null_once_the_kernel_changed(tmp_path, monkeypatch):
    _fake_tree(tmp_path, b"// edited kernel\n", hashlib.sha256(b"// captured kernel\n").hexdigest(), 1000, 100)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench._attention_traffic(100) is None


def test_attention_traffic_is_null_without_a_capture(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench._attention_traffic(100) is None


def test_committed_capture_record_is_well_formed():
    import json

    with open(os.path.join(bench.ROOT, "profiles", "attention_traffic.json")) as f:
        rec = json.load(f)
    assert rec["rows"] > 0 and rec["traffic_bytes_per_launch"] > 0 and len(rec["source_sha256"]) == 64
    assert os.path.exists(os.path.join(bench.ROOT, rec["source"]))
    assert "--clock-control none" in rec["command"]


class _Done:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def test_clock_samples_median_and_throttle_reasons(tmp_path):
    path = tmp_path / "clocks.csv"
    rows = [
        "0, 1400, 2032, 1090.5, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 1420, 2032, 1095.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 1380, 2032, 1100.2, 0x4, Not Active, Not Active, Not Active, Active",
        "garbled line",
        "0, [N/A], 2032, 0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    path.write_text("\n".join(rows) + "\n")
    cs = bench.ClockSampler(None, 0, str(path))
    cs.proc = _Done()
    cs.f = open(path, "a")
    got = cs.stop()
    assert got == {"sm_mhz": 1400.0, "sm_max_mhz": 2032.0, "reasons": ["sw_power_cap"], "samples": 3}


def test_clock_samples_flag_a_thermal_slowdown(tmp_path):
    path = tmp_path / "clocks.csv"
    path.write_text("0, 1900, 2032, 900, 0x20, Not Active, Active, Not Active, Not Active\n")
    cs = bench.ClockSampler(None, 0, str(path))
    cs.proc = _Done()
    cs.f = open(path, "a")
    assert cs.stop()["reasons"] == ["hw_thermal_slowdown"]


def test_reference_arm_line(capsys):
    """The reference arm (the CPU oracle, rank 0 only) prints one line with the contract's keys;
    on the 72-row configuration it finishes in well under a second."""
    import argparse
    import json

    import synth

    args = argparse.Namespace(gpus=1, steps=2, warmup=1)
    bench.run_reference(args, synth.CONFIGS["tiny"], 0)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC and line["unit"] == bench.UNIT
    assert line["value"] > 0 and line["steps"] == 2 and line["warmup"] == 1 and line["higher_is_better"]
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": bench.UNIT, "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["config"]["workload"] == "tiny"
    # other ranks print nothing
    bench.run_reference(args, synth.CONFIGS["tiny"], 1)
    assert capsys.readouterr().out == ""


def test_page_canvas_matches_the_pages_figure():
    """The context measurement's workload and the pages' figure it sits next to come from the
    pages' 'Performance' table: 37,966 packed rows, 8.8 min per denoising step."""
    import json
    import os

    import synth

    fig = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_figures.json")))
    fig = fig["m3_ultra_step_37966_rows"]
    assert synth.CONFIGS["trunk37966"].layout.n_rows == fig["rows"]
    assert bench.PAGES_M3_ULTRA_STEP_S == fig["minutes_per_step"] * 60
    # one block timed and multiplied by 50 (the page's own extrapolation, within its rounding)
    assert abs(fig["seconds_per_block"] * 50 / 60 - fig["minutes_per_step"]) <= 0.05 + 1e-9  # 8.75 printed as 8.8
