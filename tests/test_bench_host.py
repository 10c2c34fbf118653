"""Host logic of bench.py (no GPU): the reference arm's JSON line, workload naming after a
size override, the ncu-traffic record (ingest, lookup gated by workload sizes and kernel
sources), GEMM record names, clock parsing and the whole-job throughput."""
import json
import os
import subprocess
import sys

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _args(*argv):
    old = sys.argv
    sys.argv = ["bench.py", *argv]
    try:
        return bench.parse()
    finally:
        sys.argv = old


def _run_bench(*argv, env=None):
    e = dict(os.environ)
    e.update(env or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *argv], cwd=ROOT,
                          env=e, capture_output=True, text=True, timeout=300)


def test_reference_arm_prints_one_contract_line():
    r = _run_bench("--impl", "reference", "--workload", "1", "--steps", "1", "--warmup", "0")
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s"
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert d["steps"] == 1 and d["warmup"] == 0 and d["n_gpus"] == 1
    assert d["vs_baseline"] is None and d["dtype"] == "f64"
    assert d["config"]["workload"] == "tiny-gelu T128 H256 F1024 t2"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_is_silent_on_other_ranks():
    r = _run_bench("--impl", "reference", "--workload", "1", "--steps", "1", "--warmup", "0",
                   "--gpus", "2", env={"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_size_override_renames_the_workload():
    assert bench.bench_shape(_args()).name == "gelu T8192 H5120 F20480 t8"
    s = bench.bench_shape(_args("--tokens", "2048"))
    assert (s.tokens, s.name) == (2048, "gelu T2048 H5120 F20480 t8")
    s = bench.bench_shape(_args("--workload", "5", "--tp", "4"))
    assert (s.tp, s.name) == (4, "sp-preln-swiglu T8192 H8192 F28672 t4")
    with pytest.raises(SystemExit):
        bench.bench_shape(_args("--workload", "3", "--branch"))  # no LayerNorm to branch from


def test_record_names_of_gemm_kernels():
    assert bench.record_name("void gemm_pair_kernel<8, 0>(CUtensorMap_st, GemmParams)") == \
        "wgrad_w2"
    assert bench.record_name("void gemm_pair_kernel<3, 1>(CUtensorMap_st)") == "dgrad_gelu_f8"
    assert bench.record_name("void gemm_pair_kernel<0, 0>(x)") == "fc1_gelu"
    assert bench.record_name("colsum_bf16_kernel(const __nv_bfloat16 *, long)") is None


def _fake_root(tmp_path):
    """A root holding the real kernel sources (for the hash) and an empty profiles/."""
    os.symlink(os.path.join(ROOT, "megatron_tensor_transformer_tma_gb300"),
               tmp_path / "megatron_tensor_transformer_tma_gb300")
    (tmp_path / "profiles").mkdir()
    return tmp_path


def _ncu_csv(path, launches):
    head = ["ID", "Process ID", "Process Name", "Host Name", "Kernel Name", "Context", "Stream",
            "Block Size", "Grid Size", "Device", "CC", "Section Name", "Metric Name",
            "Metric Unit", "Metric Value"]
    rows = ['==PROF== Connected to process 1', ",".join(f'"{h}"' for h in head)]
    for i, (kernel, rd, wr) in enumerate(launches):
        for metric, unit, v in (("dram__bytes_read.sum", "byte", rd),
                                ("dram__bytes_write.sum", "byte", wr),
                                ("gpu__time_duration.sum", "ns", 1000)):
            r = [str(i), "1", "python3", "127.0.0.1", kernel, "1", "7", "(192, 1, 1)",
                 "(152, 1, 1)", "0", "10.3", "Command line profiler metrics", metric, unit,
                 f"{v:,}"]
            rows.append(",".join(f'"{x}"' for x in r))
    path.write_text("\n".join(rows) + "\n")


def test_ingest_averages_launches_and_lookup_is_gated(tmp_path, monkeypatch):
    root = _fake_root(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(root))
    csv_path = tmp_path / "traffic.csv"
    _ncu_csv(csv_path, [
        ("void gemm_pair_kernel<3, 0>(CUtensorMap_st, CUtensorMap_st, GemmParams)", 1000, 300),
        ("void gemm_pair_kernel<3, 0>(CUtensorMap_st, CUtensorMap_st, GemmParams)", 1200, 500),
        ("void gemm_pair_kernel<8, 1>(CUtensorMap_st, CUtensorMap_st, GemmParams)", 10, 20),
        ("colsum_bf16_kernel(const __nv_bfloat16 *, long, long, long, float *)", 7, 7),
    ])
    per = bench.ingest_ncu_traffic(str(csv_path), 3)
    assert sorted(per) == ["dgrad_gelu", "wgrad_w2_f8"] and len(per["dgrad_gelu"]) == 2
    recs = json.loads((root / "profiles" / "traffic.json").read_text())
    dg = [r for r in recs if r["kernel"] == "dgrad_gelu"][0]
    assert (dg["dram_read"], dg["dram_write"], dg["dram_bytes_per_launch"]) == (1100, 400, 1500)
    assert dg["source_hash"] == bench.kernel_source_hash() and dg["launches"] == 2

    from inputs import workload
    w3 = workload(3)
    assert bench.recorded_traffic("dgrad_gelu", 3, w3) == 1500
    assert bench.recorded_traffic("dgrad_gelu", 4, workload(4)) is None  # other workload
    assert bench.recorded_traffic("dgrad_gelu", 3, w3.with_tokens(2048)) is None  # resized
    assert bench.recorded_traffic("dgrad_gelu", 3, w3.with_tp(4)) is None
    # a re-ingest replaces the workload's records of the kernels it saw, keeps the rest
    _ncu_csv(csv_path, [("void gemm_pair_kernel<3, 0>(a)", 5, 5)])
    bench.ingest_ncu_traffic(str(csv_path), 3)
    recs = json.loads((root / "profiles" / "traffic.json").read_text())
    assert sorted(r["kernel"] for r in recs) == ["dgrad_gelu", "wgrad_w2_f8"]
    assert bench.recorded_traffic("dgrad_gelu", 3, w3) == 10
    # records taken on other kernel sources are not reported
    for r in recs:
        r["source_hash"] = "0" * 16
    (root / "profiles" / "traffic.json").write_text(json.dumps(recs))
    assert bench.recorded_traffic("dgrad_gelu", 3, w3) is None


def test_clock_parsing():
    lines = [
        "1965, 2070, 1310.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "1830, 2070, 1398.2, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "2070, 2070, 900.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "[N/A], 2070, 0, 0, Not Active, Not Active, Not Active, Not Active",
        "garbage",
    ]
    c = bench.parse_clocks(lines)
    assert c == {"sm_mhz": 1965.0, "sm_max_mhz": 2070.0, "samples": 3,
                 "reasons": ["sw_power_cap"]}
    hot = bench.parse_clocks(["1500, 2070, 1400, 0x68, Active, Active, Not Active, Active"])
    assert hot["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_power_cap"]
    assert bench.parse_clocks([]) is None


def test_job_throughput_counts_every_replica():
    assert bench.job_tflops(1e12, 1, 1000.0) == pytest.approx(1.0)
    assert bench.job_tflops(1e12, 4, 1000.0) == pytest.approx(4.0)
    assert bench.reduce_max(3.5, None, 1) == 3.5


def test_peak_regime_follows_the_sampled_clock():
    peaks = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
    assert bench.peak_regime({"sm_mhz": 2070.0, "sm_max_mhz": 2070.0}, peaks) == ("burst", 1900.0)
    assert bench.peak_regime({"sm_mhz": 1967.0, "sm_max_mhz": 2070.0}, peaks) == ("burst", 1900.0)
    assert bench.peak_regime({"sm_mhz": 1960.0, "sm_max_mhz": 2070.0}, peaks) == \
        ("sustained", 1700.0)
    assert bench.peak_regime(None, peaks) == ("sustained", 1700.0)
