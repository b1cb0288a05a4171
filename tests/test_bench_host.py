"""The benchmark's reference arm and command line, on the host.

``bench.py --impl reference`` times the float64 oracle on the host cores: it
needs no GPU, so its JSON line is checked here key by key.  Under several
ranks only rank 0 works and prints; fewer than three warm-up steps are
refused.
"""
from __future__ import annotations

import json
import os
import subprocess
import sys
from pathlib import Path

import bench

_ROOT = Path(__file__).resolve().parents[1]


def _bench(*args, env=None, timeout=300):
    e = dict(os.environ)
    e.update(env or {})
    return subprocess.run([sys.executable, str(_ROOT / "bench.py"), *args], capture_output=True, text=True,
                          timeout=timeout, env=e, cwd=str(_ROOT))


def test_reference_arm_line():
    r = _bench("--impl", "reference", "--steps", "2", "--warmup", "3")
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT == "TFLOP/s"
    assert d["value"] > 0 and d["higher_is_better"] is True
    assert (d["n_gpus"], d["steps"], d["warmup"]) == (1, 2, 3)
    assert d["ms_per_step"] > 0 and d["data"] == "synthetic" and d["vs_baseline"] is None
    assert d["config"]["workload"] == bench.WORKLOAD
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    # the value is the causal-adjusted FLOPs of one 511-token layer per step over the step time
    p = bench.workloads.CONFIGS[bench.WORKLOAD].problem
    assert abs(d["value"] - p.flops() / (d["ms_per_step"] / 1e3) / 1e12) <= 1e-9 * d["value"] + 1e-12


def test_reference_arm_other_ranks_are_silent():
    r = _bench("--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3",
               env={"WORLD_SIZE": "2", "RANK": "1", "LOCAL_RANK": "1"})
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_too_few_warmup_steps_are_refused():
    r = _bench("--impl", "reference", "--steps", "1", "--warmup", "2")
    assert r.returncode != 0
    assert "warmup" in r.stderr


# --- the parity field of the bench line -----------------------------------------

def test_parity_summary_reads_distances_and_empty_rows():
    import numpy as np
    eo = np.zeros((1, 2, 3, 4))
    el = np.array([[[0.5, -np.inf, 1.0], [0.2, 0.3, 0.4]]])
    s = bench.parity_summary(eo.copy(), el.copy(), eo, el)
    assert s["within_tolerance"] and s["empty_rows_match"] and s["max_abs_o"] == 0.0 and s["max_abs_lse"] == 0.0
    o = eo.copy()
    o[0, 1, 2, 3] = 0.03  # above the 2e-2 bound
    s = bench.parity_summary(o, el.copy(), eo, el)
    assert not s["within_tolerance"] and abs(s["max_abs_o"] - 0.03) < 1e-12
    lse = el.copy()
    lse[0, 0, 1] = 0.0  # a row the oracle calls empty must stay empty
    s = bench.parity_summary(eo.copy(), lse, eo, el)
    assert not s["empty_rows_match"] and not s["within_tolerance"]


def test_parity_of_the_benchmark_layer_shapes():
    """The bench's expression on stand-ins for its output buffers: the
    oracle's own layer 0, stored as bf16 O and fp32 lse, is within the bf16
    tolerance of itself, with the shapes the timed graph writes."""
    import torch
    flops, secs, layers, threads, first = bench.time_oracle_layers(0.0, max_layers=1)
    assert layers == 1 and flops > 0 and secs > 0
    eo, el = first
    p = bench.workloads.CONFIGS[bench.WORKLOAD].problem
    assert eo.shape == (p.B, p.Hq, p.Tq, p.d) and el.shape == (p.B, p.Hq, p.Tq)
    outs = [(torch.from_numpy(eo).to(torch.bfloat16), torch.from_numpy(el).float())]
    s = {"layer": 0, **bench.parity_summary(outs[0][0].float().cpu().numpy(), outs[0][1].cpu().numpy(), *first)}
    assert s["within_tolerance"], s
    assert 0 < s["max_abs_o"] <= 2 ** -8 * float(abs(eo).max())  # bf16 rounding of O only


# --- the roofline's traffic figure ------------------------------------------------

def test_recorded_traffic_follows_the_kernel_sources(tmp_path):
    """A capture is read while the kernel sources match its digest; a record
    with another digest (the kernel changed since) reads as None."""
    rec = {bench.WORKLOAD: {"dram_bytes_per_launch": 123, "kernel_sources_sha256": bench.kernel_sources_digest()}}
    f = tmp_path / "t.json"
    f.write_text(json.dumps(rec))
    assert bench.recorded_traffic(bench.WORKLOAD, str(f)) == 123
    rec[bench.WORKLOAD]["kernel_sources_sha256"] = "0" * 64
    f.write_text(json.dumps(rec))
    assert bench.recorded_traffic(bench.WORKLOAD, str(f)) is None
    assert bench.recorded_traffic("no_such_workload", str(f)) is None
    assert bench.recorded_traffic(bench.WORKLOAD, str(tmp_path / "missing.json")) is None
    f.write_text("{not json")
    assert bench.recorded_traffic(bench.WORKLOAD, str(f)) is None


def _lc(name, ms, tf, frac, ms_seq, tf_seq, frac_seq):
    return {"workload": name, "ms": ms, "tflops": tf, "frac_of_measured_peak": frac, "ms_per_call_in_sequence": ms_seq,
            "tflops_in_sequence": tf_seq, "frac_in_sequence": frac_seq,
            "clocks": {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"] if "32768" in name else []}}


def test_compact_summary_fits_the_stored_tail():
    """The compact summary carries every configuration's figures in a few
    hundred bytes, so a record that keeps only the last 1,500 characters of
    the line still holds them all."""
    lc = [_lc(n, 0.02, 700.0, 0.36, 0.02, 850.0, 0.437) for n in bench.LONG_CONTEXT]
    others = []
    for name in bench._SHORT:
        for dt in ("f32", "f32tc", "bf16", "e4m3"):
            e = {"workload": name, "dtype": dt, "ms": 0.123456, "tflops": 123.456}
            if dt == "f32":
                e["frac_of_fp32_simt_peak"] = 0.17
            if dt == "f32tc":
                e.update(frac_of_tensor_ceiling=0.15, frac_of_fp32_simt_peak=0.8)
            if dt == "e4m3":
                e["frac_of_fp8_peak"] = 0.2
            if name.startswith("window"):
                e["frac_of_hbm_peak"] = 0.11
            others.append(e)
    others = others[:17]  # the bench times 17 such entries
    decode = [{"workload": f"decode_gqa16x8_d128_k{k}", "us_per_call": 12.34, "frac_of_hbm_peak": 0.4,
               "clocks": {"sm_mhz": 2070.0, "reasons": []}} for k in (2044, 8192, 32768, 1, 2, 3, 4)]
    for e in decode[:4]:  # the contiguous decode steps are also timed through fa_fwd_splitkv
        e["splitkv_workspace"] = {"us_per_call": 10.5, "frac_of_hbm_peak": 0.612}
    parity = {"layer": 0, "max_abs_o": 0.0077, "mean_abs_o": 0.00021, "max_abs_lse": 1e-6, "within_tolerance": True,
              "tolerance": {"o_max": 0.02}}
    summ = bench.compact_summary(lc, others, decode, parity, {"reasons": []})
    text = json.dumps({"summary": summ})
    assert len(text) < 1400, len(text)
    assert set(summ["long_context"]) == {"t2044", "t8192", "t32768"}
    assert summ["long_context"]["t2044"][5] == 0.437
    assert len(summ["other_paths"]) == 17 and len(summ["decode"]) == 7
    assert summ["decode"]["k2044"] == [12.3, 0.4, 10.5, 0.612]
    assert summ["clocks_all"] == {"sm_mhz_min": 2070.0, "reasons": ["sw_power_cap"]}


def test_summary_is_the_last_key_of_the_line():
    """run_fa builds the line with the verbose records first and the summary
    last (json.dumps keeps insertion order)."""
    import inspect
    src = inspect.getsource(bench.run_fa)
    body = src[src.index("line = {"):src.index("print(json.dumps(line)")]
    keys = [k for k in ("\"detail\"", "\"metric\"", "\"cpu_baseline\"", "\"parity\"", "\"summary\"") if k in body]
    assert keys == ["\"detail\"", "\"metric\"", "\"cpu_baseline\"", "\"parity\"", "\"summary\""]
    assert body.index("\"summary\"") > body.index("\"parity\"") > body.index("\"cpu_baseline\"")
