"""The bench's JSON line (composed on the host; no GPU): the keys the bench
contract asks for are present, the decode headline is at top level, and the
line with every optional measurement filled stays under 1500 characters, so a
log tail of that length holds all of it."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads as W  # noqa: E402


def full_line():
    tf = {"value": 1523.4567, "roofline": {"frac": 0.7831234}}
    return bench.bench_line(
        world=1, steps=200, warmup=5, value=1523.4567, dec_value=6575.123, dec_frac=0.98456,
        step_ms=0.82061, S=3, pre_achieved=1523.4567, tc_peak=1945.4, traffic=133140000.0,
        e2e={"value": 732.61234, "unit": "TFLOP/s", "h2d_bytes_per_step": 100663296,
             "d2h_bytes_per_step": 68157440, "ms": 0.75},
        cpu={"value": 0.0030631, "unit": "TFLOP/s", "cores": 16}, cpu_rows_n=93, launches=800,
        clk={"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 78},
        dec_avg=0.32781, dec_e2e={"value": 5788.123}, det={"value": 6308.1}, adaptive={"value": 5990.9},
        prefill_2048=tf, prefill_paged=tf, merge_pair={"value": 6291.2},
        mixed={"prefill_tflops": 1270.1, "decode_rows_gbs": 5786.4, "decode_alone_gbs": 6410.2},
        decode_b1={W.DECODE_S32K.name: {"us_per_call": 22.9012, "frac_of_hbm": 0.87751},
                   W.DECODE_70B_TP8.name: {"us_per_call": 9.4241, "frac_of_hbm": 0.26671}})


def test_contract_keys_and_decode_headline():
    line = full_line()
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "roofline",
                "e2e", "cpu_baseline", "gpu_launches", "clocks", "decode_gbs", "decode_frac"):
        assert key in line, key
    assert list(line)[:5] == ["metric", "value", "unit", "decode_gbs", "decode_frac"]
    assert set(line["roofline"]) >= {"bound", "achieved", "peak", "unit", "frac", "traffic"}
    assert set(line["e2e"]) == {"value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"}
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert "workload" in line["config"]


def test_line_fits_a_1500_character_tail():
    text = json.dumps(full_line())
    assert len(text) < 1500, len(text)
    assert json.loads(text)["x"]["b1_70b_tp8_us"] == 9.424
