"""Host logic of the benchmark (no GPU): the algorithmic FLOP counts behind
``tflops`` and the roofline, the clock-record summary that decides whether a
timed run is kept, the rule that a profiled DRAM traffic figure is reported
only while the kernel sources are the ones it was measured on, the workload
``config`` both arms share, and the reference arm's JSON line (the fp64
oracle on the host cores) run end to end on the smallest workload."""
import hashlib
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402


# ---------------------------------------------------------------------------
# FLOPs: per layer and direction, the forward's contractions are the input
# projection 2*G*H*I_l*B*T and the recurrent product 2*G*H*H*B*T; the
# backward repeats both (dx and the recurrent dh), and the weight update has
# one of each again (dW_ih, dW_hh) - three times the forward in all.
# ---------------------------------------------------------------------------
def test_headline_flops_by_hand():
    wl = synth.WORKLOADS["gru_ra_bf16_T128_B64_H512"]
    # 2 * 3 gates * 512 * (512 + 512) * 64 * 128 = 25,769,803,776 per pass
    assert wl.flops() == 3 * 25_769_803_776
    fl = bench.class_flops(wl)
    assert fl["persist_fwd"] == fl["persist_bwd"] == 2 * 3 * 512 * 512 * 64 * 128
    assert fl["gemm_proj"] == fl["gemm_dx"] == 2 * 3 * 512 * 512 * 64 * 128
    assert fl["gemm_dw"] == 2 * fl["gemm_proj"]
    assert fl["layout_seq"] == fl["layout_pack"] == fl["recompute_cells"] == 0.0


@pytest.mark.parametrize("name", sorted(synth.WORKLOADS))
def test_class_flops_sum_to_the_step(name):
    wl = synth.WORKLOADS[name]
    fl = bench.class_flops(wl)
    G, H, B, T, D = wl.gates, wl.hidden_size, wl.batch, wl.seq_len, wl.dirs
    inputs = [wl.input_size] + [D * H] * (wl.num_layers - 1)      # layer l > 0 reads [y_fwd | y_bwd]
    fwd = sum(D * 2 * G * H * (I + H) * B * T for I in inputs)
    assert fl["persist_fwd"] + fl["gemm_proj"] == fwd
    if wl.forward_only:
        assert wl.flops() == fwd
    else:
        assert sum(fl.values()) == wl.flops() == 3 * fwd


# ---------------------------------------------------------------------------
# clock records (nvidia-smi csv, no header, no units)
# ---------------------------------------------------------------------------
def _row(sm, smax, hw="Not Active", hwt="Not Active", swt="Not Active", cap="Not Active"):
    return f"0, {sm}, {smax}, 950.00, 0x0000000000000000, {hw}, {hwt}, {swt}, {cap}\n"


def test_clock_summary_median_and_reasons():
    lines = [_row(1965, 2070), _row(1980, 2070, cap="Active"), _row(2010, 2070), "garbage\n",
             "0, [N/A], 2070, 1, 0x0, Not Active, Not Active, Not Active, Not Active\n"]
    c = bench.parse_clock_lines(lines)
    assert c["sm_mhz"] == 1980 and c["sm_max_mhz"] == 2070 and c["samples"] == 3
    assert c["reasons"] == ["sw_power_cap"]


def test_clock_summary_flags_every_slowdown():
    c = bench.parse_clock_lines([_row(1200, 2070, hw="Active"), _row(1100, 2070, hwt="Active", swt="Active")])
    assert c["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]


def test_clock_summary_without_samples():
    assert bench.parse_clock_lines([]) == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}


# ---------------------------------------------------------------------------
# profiled traffic: taken only while the kernel sources match the profile
# ---------------------------------------------------------------------------
def _sources_sha():
    h = hashlib.sha256()
    for f in bench.KERNEL_SOURCES:
        h.update(bench.code_only(open(os.path.join(ROOT, f)).read()).encode())
    return h.hexdigest()[:16]


def test_code_only_ignores_comments_and_whitespace():
    a = "int f(int x) {  // the sum\n  return x + 1; /* one\n more */ }\n"
    b = "int f(int x){return x+1;}"
    assert bench.code_only(a) == bench.code_only(b)
    assert bench.code_only(a) != bench.code_only(b.replace("+ 1", "+ 2").replace("+1", "+2"))


@pytest.mark.parametrize("sha_ok", [True, False])
def test_profiled_traffic_follows_the_sources(tmp_path, monkeypatch, sha_ok):
    prof = tmp_path / "persist_bwd_tc_{workload}.md"
    (tmp_path / "persist_bwd_tc_w.md").write_text(
        "# summary\n\ntraffic-bytes-per-launch: 1234567\n"
        f"kernel-source-sha256: {_sources_sha() if sha_ok else '0' * 16}\n")
    monkeypatch.setitem(bench.PROFILE_FOR_CLASS, "persist_bwd", str(prof))
    assert bench.profiled_traffic("persist_bwd", "w") == (1234567 if sha_ok else None)
    assert bench.profiled_traffic("persist_bwd", "other_workload") is None      # no summary
    assert bench.profiled_traffic("gemm_dw", "w") is None                      # class never profiled


def test_committed_profiles_name_a_traffic_and_a_sha():
    import glob
    found = 0
    for cls, path in bench.PROFILE_FOR_CLASS.items():
        for p in glob.glob(os.path.join(ROOT, path.format(workload="*"))):
            keys = {ln.split(":", 1)[0].strip() for ln in open(p) if ":" in ln}
            assert {"traffic-bytes-per-launch", "kernel-source-sha256"} <= keys, p
            found += 1
    assert found >= 1


# ---------------------------------------------------------------------------
# the config both arms report
# ---------------------------------------------------------------------------
def test_workload_config():
    wl = synth.WORKLOADS["gru_ra_bf16_T128_B64_H512_varlen"]
    lengths = synth.make_lengths(wl)
    assert lengths is not None and len(lengths) == wl.batch
    assert (lengths == synth.make_inputs(wl, batch_subset=range(wl.batch)).lengths).all()
    c = bench.workload_config(wl, lengths, 1)
    assert c["workload"] == wl.name and c["parallelism"] == "replicas1"
    assert c["seq_lengths"]["valid_frac"] == pytest.approx(lengths.sum() / (wl.seq_len * wl.batch))
    assert 0.5 <= c["seq_lengths"]["valid_frac"] <= 1.0
    assert "seq_lengths" not in bench.workload_config(synth.WORKLOADS[bench.DEFAULT_WORKLOAD], None, 2)


def _run_reference(extra_env=None):
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", **(extra_env or {}))
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                           "--warmup", "1", "--workload", "lstm_f32_T16_B4_I32_H32"],
                          capture_output=True, text=True, env=env, cwd=ROOT, timeout=600)


def test_reference_arm_json_line():
    r = _run_reference()
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["value"] > 0 and d["higher_is_better"] is True and d["vs_baseline"] is None
    assert (d["n_gpus"], d["steps"], d["warmup"]) == (1, 2, 1)
    assert d["ms_per_step"] > 0 and d["scaling"] == "weak" and d["data"] == "synthetic"
    assert d["config"] == bench.workload_config(synth.WORKLOADS["lstm_f32_T16_B4_I32_H32"], None, 1)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and "fwd+bwd" in cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_print_nothing():
    r = _run_reference({"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


@pytest.mark.parametrize("threads", [1, 0])
def test_oracle_timing_subprocess(threads):
    wl = synth.WORKLOADS["lstm_f32_T16_B4_I32_H32"]
    out, cores = bench.run_oracle_subprocess(wl, 0.0, 3, reps=2, threads=threads)
    assert cores == (1 if threads == 1 else (os.cpu_count() or 1))
    assert len(out["times"]) == 2 and all(t > 0 for t in out["times"])
    assert out["units_per_rep"] == wl.seq_len * 3


def test_fp32_peak_derivation():
    # 152 SMs x 128 FP32 lanes x 2 flops per FMA x 2070 MHz
    assert bench.fp32_fma_tflops(152, 2070.0) == pytest.approx(80.54784)
    assert bench.load_peaks()["sm_max_mhz"] > 0


# ---------------------------------------------------------------------------
# layout kernels: achieved bandwidth = algorithmic bytes / event time, against
# the HBM copy rate; classes with no launch are left out
# ---------------------------------------------------------------------------
def test_layout_report_bandwidth():
    names = ("persist_fwd", "persist_bwd", "gemm_proj", "gemm_dx", "gemm_dw", "layout_seq", "layout_pack",
             "recompute_cells")
    ms = [5.0, 6.0, 1.0, 1.0, 1.0, 0.5, 0.1, 0.0]
    n = [2, 2, 2, 2, 4, 2, 6, 0]
    by = [0, 0, 0, 0, 0, 3.0e9, 2.0e8, 0]
    rep = bench.layout_report(names, ms, n, by, 2, 6000.0)
    assert set(rep) == {"layout_seq", "layout_pack"}
    assert rep["layout_seq"]["achieved_gbs"] == pytest.approx(3.0e9 / 0.5e-3 / 1e9)
    assert rep["layout_seq"]["frac_of_hbm"] == pytest.approx(6000.0 / 6000.0)
    assert rep["layout_pack"]["bytes_per_step"] == pytest.approx(1.0e8)
    assert rep["layout_pack"]["launches_per_step"] == 3


def test_both_arms_share_the_config():
    wl = synth.WORKLOADS[bench.DEFAULT_WORKLOAD]
    a = bench.workload_config(wl, None, 1)
    b = bench.workload_config(wl, synth.make_lengths(wl), 1)
    assert a == b
    assert a["workload"] == "lstm2bi_bf16_T512_B128_H1024"
    assert "reserve_bytes" not in a


def test_gpus_flag_starts_its_own_ranks():
    # no WORLD_SIZE in the environment: bench.py starts 2 ranks itself
    # (torch.distributed.run, gloo without a GPU) and rank 0 reports both
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    env["CUDA_VISIBLE_DEVICES"] = ""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--probe-ranks"],
                       capture_output=True, text=True, env=env, cwd=ROOT, timeout=300)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    assert lines[0]["n_gpus"] == 2 and lines[0]["rank_sum"] == 3.0 and lines[0]["max_rank"] == 1.0
