"""bench.py's host logic on the CPU: the mode it labels and counts launches for,
the algorithmic byte and FLOP accounting behind the roofline, the L2 policy, and
the lookup of the committed DRAM-traffic record."""
import importlib.util
import json
import os
import types

import numpy as np
import pytest

import gen

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("k3moe_bench", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_expert_bytes_is_the_mxfp4_footprint(bench):
    s = gen.CONFIGS["decode"]
    # codes (half a byte) + e8m0 scales (one byte per 32) of W_gate, W_up and W_down
    assert bench.expert_bytes(s) == 3 * 7168 * 2048 // 2 + 3 * 7168 * 2048 // 32 == 23_396_352


def test_kernel_counts_and_labels_per_mode(bench):
    s = gen.CONFIGS["decode"]
    assert bench.resolved_mode(s, 0) == 1
    assert bench.resolved_mode(gen.CONFIGS["prefill"], 0) == 3
    assert [bench.ffn_kernel_count(s, m) for m in (1, 2, 3, 4)] == [4, 4, 6, 6]  # 2 runs the GEMV kernels
    assert "mxf4" in bench.ffn_kernel_label(s, 4) and "GEMV" in bench.ffn_kernel_label(s, 0)


def test_tensor_figures_use_the_mode_peaks(bench, monkeypatch):
    monkeypatch.setattr(bench, "measured_peaks", lambda: {"bf16_tflops": 2000.0})
    s = gen.CONFIGS["prefill"]
    flops = 2.0 * s.T * s.k * 3 * s.H * s.I
    assert bench.tensor_figures(gen.CONFIGS["decode"], 0, 1e-4) is None  # GEMV: no tensor core
    f16 = bench.tensor_figures(s, 3, 1e-2)
    fp4 = bench.tensor_figures(s, 4, 1e-2)
    assert f16["tflops"] == pytest.approx(flops / 1e-2 / 1e12)
    assert f16["peak_tflops"] == 2000.0 and fp4["peak_tflops"] == 12000.0
    assert fp4["fp4_dense_frac"] == pytest.approx(fp4["tflops"] / 12000.0)


def test_l2_policy(bench):
    s = gen.CONFIGS["decode"]
    sets = [bench.input_set("decode", s, i) for i in range(2)]
    a = types.SimpleNamespace(l2_flush=False)
    flush, text = bench.l2_policy(a, s, sets)
    assert not flush and "no flush" in text  # 16 experts x 23.4 MB >> 2 x L2
    a.l2_flush = True
    assert bench.l2_policy(a, s, sets)[0]
    tiny = gen.CONFIGS["tiny"]
    a.l2_flush = False
    assert bench.l2_policy(a, tiny, [bench.input_set("tiny", tiny, 0)])[0]


def test_routed_experts_matches_the_oracle_rule(bench):
    s = gen.CONFIGS["decode"]
    logits = gen.make_logits("decode", s)
    picks = bench.routed_experts(s, logits)[0]
    order = sorted(range(s.E), key=lambda e: (-float(logits[0, e]), e))[: s.k]
    assert list(picks) == order


def test_traffic_record_follows_the_sources(bench, tmp_path, monkeypatch):
    rec = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    # the committed record is reported only while it is keyed by the current sources
    if rec["decode"]["source_hash"] == bench.kernel_source_hash(rec["decode"].get("source_files")):
        assert bench.recorded_traffic("decode") == rec["decode"]["dram_bytes_per_call"]
    else:
        assert bench.recorded_traffic("decode") is None
    # a record taken on other sources is not reported
    (tmp_path / "profiles").mkdir()
    rec["decode"]["source_hash"] = "0" * 16
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("decode") is None
    assert bench.recorded_traffic("prefill") is None


def test_host_cpu_is_described(bench):
    h = bench.host_cpu()
    assert h["nproc"] >= 1 and h["oracle_threads"] == 1 and isinstance(h["model"], str) and h["model"]


def test_ffn_bytes_and_per_expert_roofline(bench, monkeypatch):
    monkeypatch.setattr(bench, "measured_peaks", lambda: {"hbm_gbs": 8000.0, "bf16_tflops": 2000.0})
    s = gen.CONFIGS["decode"]
    A = s.T * s.k
    assert bench.ffn_bytes_per_call(s, 16) == 16 * 23_396_352 + 7168 * 2 + A * 2048 * 4 + A * 7168 * 4
    counts = np.zeros(s.E, np.int64)
    counts[:16] = 1
    # CUDA-core GEMV: the HBM term alone, expert by expert, plus x, h and Y
    t = bench.per_expert_roofline_s(s, counts, 1)
    assert t == pytest.approx(bench.ffn_bytes_per_call(s, 16) / 8e12)
    # a compute-bound expert on the FP4 tensor core: n * 6 H I / (6 x bf16 peak)
    p = gen.CONFIGS["probe"]
    cp = np.zeros(p.E, np.int64)
    cp[:] = 2048
    t4 = bench.per_expert_roofline_s(p, cp, 4)
    extra = (p.T * p.H * 2 + p.T * p.I * 4 + p.T * p.H * 4) / 8e12
    assert t4 == pytest.approx(16 * max(23_396_352 / 8e12, 2048 * 6.0 * 7168 * 2048 / 12e15) + extra)
    t3 = bench.per_expert_roofline_s(p, cp, 3)
    assert t3 == pytest.approx(16 * 2048 * 6.0 * 7168 * 2048 / 2e15 + extra)


def test_extra_workloads_cover_the_configs_and_modes(bench):
    names = {n for n, _ in bench.LEGS}
    assert {"batch8", "prefill", "skewed", "probe", "spec2", "spec4", "spec12", "spec16"} <= names
    for n in ("prefill", "skewed"):
        modes = {bench.mode_name(gen.CONFIGS[n], m) for nn, m in bench.LEGS if nn == n}
        assert modes == {"gemm_w4a16", "w4a4"}
    for n in ("batch8", "spec2", "spec4", "spec12", "spec16"):
        modes = {bench.mode_name(gen.CONFIGS[n], m) for nn, m in bench.LEGS if nn == n}
        assert modes == {"gemv", "gemm_w4a16"}


def test_layer_kernel_count(bench):
    assert bench.layer_kernel_count(gen.CONFIGS["decode"], 0) == 5     # single-block front + 3 FFN + combine
    assert bench.layer_kernel_count(gen.CONFIGS["spec4"], 0) == 5
    assert bench.layer_kernel_count(gen.CONFIGS["spec12"], 0) == 1 + 1 + 4 + 1
    assert bench.layer_kernel_count(gen.CONFIGS["prefill"], 0) == 1 + 3 + 6 + 1
    assert bench.layer_kernel_count(gen.CONFIGS["batch8"], 3) == 1 + 1 + 6 + 1


def test_legs_option(bench, monkeypatch):
    """--legs router times the router entry point alone (its own router matrix, so it
    runs beside a small expert set); the default times every workload."""
    monkeypatch.setattr("sys.argv", ["bench.py", "--legs", "router", "--experts", "64"])
    a = bench.parse()
    assert a.legs == "router" and a.experts == 64
    monkeypatch.setattr("sys.argv", ["bench.py"])
    assert bench.parse().legs == "all"
    monkeypatch.setattr("sys.argv", ["bench.py", "--legs", "some"])
    with pytest.raises(SystemExit):
        bench.parse()
