"""Host-side logic of bench.py (CPU): the algorithmic work counted for the
roofline, the launches per forward, and the kernel-code hash that decides
whether a recorded ncu traffic figure still describes the GEMM."""
import json
import os
import subprocess
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from moe_expert_layer_grouped_gb300 import synth  # noqa: E402


def test_strip_comments_keeps_code_and_string_literals():
    src = ('int a; // line comment\n'
           '/* block\n   comment */ int b = 1;\n'
           '\n'
           'asm("tcgen05.ld // not a comment /* either */");\n'
           'x /* inline */ y;\n')
    out = bench._strip_comments(src)
    assert "comment" not in out.replace("not a comment", "")
    assert 'asm("tcgen05.ld // not a comment /* either */");' in out
    assert out.splitlines() == ['int a;', ' int b = 1;',
                                'asm("tcgen05.ld // not a comment /* either */");', 'x  y;']


def test_code_hash_ignores_comments_but_not_code():
    base = "int f(int x) {\n  return x + 1;  // add one\n}\n"
    same = "// header\nint f(int x) {\n\n  return x + 1;  /* plus one */\n}\n"
    other = "int f(int x) {\n  return x + 2;\n}\n"
    s = bench._strip_comments
    assert s(base) == s(same)
    assert s(base) != s(other)


def test_recorded_traffic_needs_the_current_code(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    # the kernel sources the hash reads
    src = tmp_path / "moe_expert_layer_grouped_gb300" / "csrc"
    src.mkdir(parents=True)
    for f in ("gemm.cu", "gemm_common.cuh", "ptx.cuh", "common.cuh"):
        (src / f).write_text(f"// {f}\nint {f.split('.')[0]};\n")
    h = bench.kernel_source_hash()
    (prof / "grouped_gemm_w13_wl.md").write_text(
        f"- dram_bytes_per_launch: 123456\n- kernel_source_sha256_16: {h}\n")
    assert bench.recorded_traffic("wl") == 123456.0
    (src / "gemm.cu").write_text("// gemm.cu, comment edited\nint gemm;\n")
    assert bench.recorded_traffic("wl") == 123456.0  # comments only
    (src / "gemm.cu").write_text("int gemm2;\n")
    assert bench.recorded_traffic("wl") is None      # the code changed
    assert bench.recorded_traffic("missing") is None


def test_step_work_counts_active_experts_only():
    wl = synth.Workload("w", 4, 128, 64, 4, 1, 1, 2, synth.SOFTMAX, True, 1.0, "none")
    off = np.array([0, 3, 3, 8, 8], dtype=np.int64)  # experts 0 and 2 active
    w = bench.step_work(wl, [off])
    T, H, I, K, E = 4, 128, 64, 2, 4
    M = T * K
    w13 = 2 * (2 * I * H + 2 * I * 4)
    assert w["active"] == 2
    assert w["gemm13_bytes"] == w13 + M * H + M * 4 + M * I * 2 + (E + 1) * 4
    assert w["flops13"] == 2.0 * M * 2 * I * H
    assert w["flops2"] == 2.0 * M * H * I


def test_launches_per_forward():
    dec = synth.WORKLOADS["dsv3_decode_t128"]   # T*K = 1024 slots: one pre-reorder launch
    pre = synth.WORKLOADS["dsv3_prefill_t8192"]  # three
    assert bench.launches_per_forward(dec) == 6
    assert bench.launches_per_forward(pre) == 8


def test_reference_arm_prints_the_contract_line():
    # the reference arm times the oracle on the host cores: no GPU needed
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny", "--steps", "2", "--warmup", "1"],
                       env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 1
    assert d["n_gpus"] == 1 and d["higher_is_better"] is True and d["value"] > 0
    assert d["config"] == bench.workload_config(synth.WORKLOADS["tiny"], 1)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert cb["unit"] == d["unit"] and "tiny" in cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_peaks_come_from_the_measured_file_else_the_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    pk = bench.peaks()                      # no file: the earlier measurements
    assert pk["source"] == "fallback"
    assert (pk["hbm"], pk["bf16"], pk["bf16_sustained"]) == (6800.0, 1900.0, 1700.0)
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps(
        {"hbm_gbs": 6681.8, "bf16_tflops": 1850.0, "bf16_tflops_sustained": 1765.2,
         "sm_max_mhz": 2070}))
    pk = bench.peaks()
    assert pk["source"] == "measured"
    assert (pk["hbm"], pk["bf16"], pk["bf16_sustained"]) == (6681.8, 1850.0, 1765.2)


def test_timed_regions_are_bracketed_by_sync_and_barrier():
    calls = []

    class _Cuda:
        @staticmethod
        def synchronize():
            calls.append("sync")

    class _Torch:
        cuda = _Cuda

    bench.align(_Torch, None)                     # one rank: the device only
    assert calls == ["sync"]
    calls.clear()
    bench.align(_Torch, lambda: calls.append("barrier"))
    assert calls == ["sync", "barrier", "sync"]   # own work done, ranks met, then time


def test_step_work_block_scales_shared_experts_and_batch_average():
    # block FP8: one scale per 128 x 128 weight block and per 128 activation channels
    wl = synth.Workload("b", 2, 256, 128, 4, 1, 1, 2, synth.SOFTMAX, True, 1.0, "none",
                        quant="block")
    off = np.array([0, 4, 4, 4, 4], dtype=np.int64)            # one active expert
    w = bench.step_work(wl, [off])
    T, H, I, M = 2, 256, 128, 4
    w13 = 2 * I * H + (2 * I // 128) * (H // 128) * 4
    assert w["gemm13_bytes"] == w13 + M * H + M * (H // 128) * 4 + M * I * 2 + 5 * 4
    w2 = H * I + (H // 128) * (I // 128) * 4
    assert w["gemm2_bytes"] == w2 + M * I + M * (I // 128) * 4 + M * H * 2 + 5 * 4
    # a shared expert: E + 1 experts, K + 1 slots, always active; logits stay [T, E]
    wl = synth.Workload("s", 3, 128, 64, 4, 1, 1, 2, synth.SOFTMAX, True, 1.0, "none",
                        n_shared=1)
    T, H, I, M = 3, 128, 64, 9
    a = np.array([0, 3, 3, 6, 6, 9], dtype=np.int64)           # experts 0, 2 and the shared one
    b = np.array([0, 0, 0, 0, 6, 9], dtype=np.int64)           # expert 3 and the shared one
    wa, wb, avg = bench.step_work(wl, [a]), bench.step_work(wl, [b]), bench.step_work(wl, [a, b])
    assert (wa["active"], wb["active"], avg["active"]) == (3, 2, 2.5)
    assert wa["flops13"] == 2.0 * M * 2 * I * H
    per_expert = (2 * I * H + 2 * I * 4) + (H * I + H * 4)
    assert wa["layer_bytes"] == 3 * per_expert + T * H * 2 + T * 4 * 4 + T * H * 2
    assert avg["layer_bytes"] == (wa["layer_bytes"] + wb["layer_bytes"]) / 2


def test_roofline_objects(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))      # no recorded traffic here
    pk = dict(hbm=7000.0, bf16=1900.0, bf16_sustained=850.0, sm_max=2070.0, source="measured")
    r = {"kern": {"grouped_gemm_w13": 0.5}, "work": {"gemm13_bytes": 3.5e9, "flops13": 0.85e12}}
    d = bench.roofline_decode(r, pk, "some_workload")
    assert (d["bound"], d["unit"], d["achieved"], d["peak"], d["frac"]) == \
        ("hbm", "GB/s", 7000.0, 7000.0, 1.0)
    assert d["traffic"] is None and d["algorithmic_bytes_per_launch"] == 3500000000
    pk = dict(hbm=7000.0, bf16=850.0, bf16_sustained=425.0, sm_max=2070.0, source="measured")
    p = bench.roofline_prefill(r, pk)
    # the GEMM is timed in a short loop at full clock (a burst): FP8 peak =
    # the burst bf16 figure x 2 = 1700 TFLOP/s; 0.85 TFLOP in 0.5 ms
    assert (p["bound"], p["unit"], p["achieved"], p["peak"], p["frac"]) == \
        ("tensor", "TFLOP/s", 1700.0, 1700.0, 1.0)
    assert "burst" in p["peak_source"] and p["traffic"] is None
    # the sustained-derived fraction stands beside it
    assert (p["sustained_peak"], p["frac_of_sustained_peak"]) == (850.0, 2.0)
    assert "clock_normalised" not in p                       # no clock record given
    # at a median 1035 MHz of 2070 the same launch would run twice as fast
    p = bench.roofline_prefill(r, pk, {"sm_mhz": 1035.0, "sm_max_mhz": 2070.0})
    assert p["clock_normalised"] == {"achieved": 3400.0, "frac": 2.0, "sm_mhz": 1035.0,
                                     "to_mhz": 2070.0}
    # the layer's fractions: 1.7 TFLOP per 1 ms step
    lf = bench.layer_fracs({"work": {"layer_flops": 1.7e12}, "ms": 1.0}, pk,
                           {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0})
    assert lf == {"layer_fp8_tensor_frac": 1.0, "layer_fp8_tensor_frac_of_sustained": 2.0,
                  "layer_fp8_tensor_frac_clock_normalised": 1.0}


def test_both_arms_print_the_same_config():
    """The reference arm's config is the same object as ours (nothing
    measured in it), so the driver can match the two lines."""
    wl = synth.WORKLOADS["dsv3_prefill_t8192"]
    a, b = bench.workload_config(wl, 1), bench.workload_config(wl, 1)
    assert a == b and a["workload"] == wl.name
    for k in ("T", "H", "I", "E", "num_groups", "topk_group", "top_k", "scoring", "rsf",
              "n_shared", "quant", "batches_cycled", "l2", "parallelism"):
        assert k in a, k
    assert a["num_groups"] == 8 and a["topk_group"] == 4 and a["scoring"] == "sigmoid"


def test_clock_summary_reads_the_timed_window():
    cs = bench.ClockSampler(0)
    row = "0, {sm}, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, {cap}"
    cs.lines = [(0.5, row.format(sm=1000, cap="Active")),          # before the window
                (1.0, row.format(sm=2070, cap="Not Active")),
                (1.5, row.format(sm=1900, cap="Active")),
                (2.0, row.format(sm=2000, cap="Not Active")),
                (2.2, "garbled line"),
                (3.5, row.format(sm=1200, cap="Not Active"))]      # after it
    s = cs.summary(1.0, 2.5)
    assert s["sm_mhz"] == 2000.0 and s["sm_max_mhz"] == 2070.0     # median of 1900, 2000, 2070
    assert s["reasons"] == ["sw_power_cap"]
    # no sample inside the window: the last few samples stand in
    s = cs.summary(10.0, 11.0)
    assert s["sm_mhz"] == 2000.0 and s["samples"] == 3


def test_layer_bound_takes_the_larger_of_tensor_and_hbm_time():
    pk = {"bf16": 2000.0, "hbm": 8000.0}
    # 4 TFLOP at 4000 TFLOP/s (FP8 = 2 x bf16) = 1 ms; 16 GB at 8 TB/s = 2 ms
    r = {"work": {"layer_flops": 4e12, "layer_bytes": 16e9}, "ms": 4.0}
    b = bench.layer_bound(r, pk)
    assert b["bound"] == "hbm" and b["tensor_ms"] == 1.0 and b["hbm_ms"] == 2.0
    assert b["frac"] == 0.5
    r = {"work": {"layer_flops": 12e12, "layer_bytes": 8e9}, "ms": 6.0}
    b = bench.layer_bound(r, pk)
    assert b["bound"] == "tensor" and b["tensor_ms"] == 3.0 and b["frac"] == 0.5
    # FP4 operands: the tensor time at 6 x bf16
    r = {"work": {"layer_flops": 12e12, "layer_bytes": 10e9}, "ms": 2.5}
    b = bench.layer_bound(r, pk, bench.FP4_PER_BF16)
    assert b["tensor_ms"] == 1.0 and b["hbm_ms"] == 1.25 and b["bound"] == "hbm"
    assert b["frac"] == 0.5
