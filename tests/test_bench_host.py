"""Host logic of bench.py that its reported numbers rest on (CPU, no GPU).

* ``cycle_states`` rebuilds every cycle's (t, fill, exited) from the ordered verdicts; the
  algorithmic bytes of the roofline are summed over those states.  It is held to the oracle's own
  cycle-by-cycle state on a run with rejects.
* ``Clocks`` parses nvidia-smi's sampled lines: median SM clock, max clock, active slowdown reasons.
* ``step_kernel_traffic_ratio`` reports the ncu traffic ratio only for the captured workload and
  while the CUDA sources hash to the captured ones; both arms share one ``config`` helper.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from oracle import spd as ospd  # noqa: E402


@pytest.mark.parametrize("alpha", [0.0, 0.6, 1.0])
def test_cycle_states_follow_the_oracle(tiny, tiny_ar, alpha):
    w, params, prompt, models = tiny
    P, G, n = len(prompt), w.gen_len, w.n_stages
    run = ospd.run_spd(w, params, prompt, G, alpha, ref=tiny_ar["tokens"], models=models, record=True)
    oracle_states = [(info["t"], info["a"], info["exited"]) for info in run.log]
    accepts = [ok for _, ok in run.trace]
    assert bench.cycle_states(P, n, accepts, run.cycles) == oracle_states


def test_cycle_states_wider_pipeline():
    # n = 4 by hand: fill 1..4, exit; a reject at the second verdict refills from fill 1
    states = bench.cycle_states(10, 4, [True, False, True], 10)
    assert states[:4] == [(11, 1, False), (12, 2, False), (13, 3, False), (14, 4, True)]
    assert states[4] == (15, 4, True)            # accepted: the pipeline stays full
    assert states[5] == (13, 1, False)           # rejected at t_e = 15-4+1 = 12: reseeded at 13
    assert [a for _, a, _ in states[5:9]] == [1, 2, 3, 4]


class _FakeProc:
    def __init__(self, out):
        self.out = out

    def terminate(self):
        pass

    def communicate(self, timeout=None):
        return self.out, ""


def test_clock_parser_median_max_and_reasons(monkeypatch):
    lines = "\n".join([
        "2070, 2070, 900.1, Not Active, Not Active, Not Active, Active",
        "2055, 2070, 950.0, Not Active, Not Active, Not Active, Active",
        "2070, 2070, 980.3, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
    ])
    c = bench.Clocks(0)
    c.proc = _FakeProc(lines)
    r = c.stop()
    assert r["sm_mhz"] == 2070.0 and r["sm_max_mhz"] == 2070.0 and r["samples"] == 3
    assert r["reasons"] == ["sw_power_cap"]
    c = bench.Clocks(0)
    c.proc = _FakeProc("1200, 2070, 500.0, Active, Not Active, Not Active, Not Active\n")
    assert c.stop()["reasons"] == ["hw_slowdown"]


def test_clock_parser_without_nvidia_smi():
    c = bench.Clocks(0)
    c.proc = None
    assert c.stop()["reasons"] == ["nvidia-smi unavailable"]


def test_traffic_ratio_only_for_the_captured_sources(tmp_path, monkeypatch):
    import hashlib
    import json
    src = tmp_path / "speculative_pipeline_decoding_gb300" / "csrc"
    src.mkdir(parents=True)
    (src / "a.cu").write_text("kernel one")
    (src / "b.cuh").write_text("header")
    (src / "notes.txt").write_text("not hashed")
    h = hashlib.sha1()
    for f in ("a.cu", "b.cuh"):
        h.update((src / f).read_bytes())
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "step_kernel_traffic.json").write_text(json.dumps(
        {"workload": "gqa9b_bf16_n8", "sources_sha1": h.hexdigest(), "dram_bytes": 9.871e9,
         "algorithmic_bytes": 1.0e10}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.step_kernel_traffic_ratio("gqa9b_bf16_n8") == pytest.approx(0.9871)
    assert bench.step_kernel_traffic_ratio("dense1.5b_bf16_n8") is None  # another workload's capture
    (src / "notes.txt").write_text("still not hashed")
    assert bench.step_kernel_traffic_ratio("gqa9b_bf16_n8") == pytest.approx(0.9871)
    (src / "a.cu").write_text("kernel two")
    assert bench.step_kernel_traffic_ratio("gqa9b_bf16_n8") is None


def test_both_arms_report_the_same_config_keys():
    import spd_inputs as si
    w = si.WORKLOADS["gqa9b_bf16_n8"]
    c = bench.bench_config(w, 0.9, 1)
    assert c["workload"] == "gqa9b_bf16_n8" and c["alpha"] == 0.9 and c["prompt"] == 2048
    assert set(c) >= {"workload", "prompt", "gen", "alpha", "n_stages", "pdm_layers", "anchors", "l2",
                      "parallelism"}


def test_measured_peaks_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_peaks() == (6800.0, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text('{"hbm_gbs": 6778.3}')
    assert bench.measured_peaks() == (6778.3, "measured")
