"""bench.py without a GPU: its helpers exist and the reference arm (the fp64
CPU oracle on a bounded sample) prints one well-formed JSON line."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_bench_helpers_exist():
    for name in ("time_prefill", "decode_line", "verify_line", "time_graph", "time_hybrid",
                 "hybrid_line", "bf16_out_line", "time_e2e", "prefill_roofline",
                 "cpu_oracle_sample", "cpu_oracle_call", "cpu_global_layer", "with_clocks",
                 "run_reference", "run_ours", "recorded_traffic", "high_sparse_line",
                 "long_context_line", "job_rate", "_event_ms"):
        assert callable(getattr(bench, name)), name


def test_reduce_without_process_group():
    assert bench.reduce_value(None, 2.5, "max") == 2.5


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True,
                       timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "TFLOP/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_source_hash_ignores_comments_and_whitespace():
    import bench
    a = 'int f(int x) {\n  return x + 1;  // one\n}\n/* block */ const char* s = "a // b /* c */";\n'
    b = 'int f(int x){return x+1;}\nconst char* s = "a // b /* c */";'
    c = 'int f(int x) { return x + 2; }\nconst char* s = "a // b /* c */";'
    assert bench.source_code_only(a) == bench.source_code_only(b)
    assert bench.source_code_only(a) != bench.source_code_only(c)
    assert '"a // b /* c */"' in bench.source_code_only(a)


def test_clock_sampler_with_a_fake_nvml():
    """The sampler's host logic: samples and clock-event reasons gathered in
    a thread while the region runs (NVML replaced by a fake that reads
    nothing from a GPU)."""
    import time

    class Fake:
        n = 0

        def sm_mhz(self):
            Fake.n += 1
            return 1900 + (Fake.n % 3)

        def sm_max_mhz(self):
            return 2032

        def reasons(self):
            return 0x4          # sw_power_cap

    bench.ClockSampler._nvml_cache[97] = Fake()
    try:
        with bench.ClockSampler(97) as clk:
            time.sleep(0.05)
        d = clk.summary()
    finally:
        del bench.ClockSampler._nvml_cache[97]
    assert d["source"] == "nvml" and d["samples"] >= 5
    assert 1900 <= d["sm_mhz"] <= 1902 and d["sm_max_mhz"] == 2032
    assert d["reasons"] == ["sw_power_cap"]


def test_traffic_record_applies_to_its_own_workload_only(tmp_path):
    # a record is per kernel, workload shape and source hash: another shape of
    # the same kernel, or changed sources, get no traffic figure
    shape = bench.traffic_shape(B=256, Hq=64, Hkv=8, D=128, W=128)
    assert shape == "B256 Hq64 Hkv8 D128 W128"
    rec = tmp_path / "traffic.txt"
    rec.write_text("# comment\n"
                   "decode_tc_kernel.bytes_per_launch: 123456\n"
                   f"decode_tc_kernel.source_hash: {bench.kernel_source_hash('decode_tc_kernel')}\n"
                   f"decode_tc_kernel.shape: {shape}\n")
    assert bench.recorded_traffic("decode_tc_kernel", shape, str(rec)) == 123456
    other = bench.traffic_shape(B=256, Hq=32, Hkv=8, D=128, W=128)
    assert bench.recorded_traffic("decode_tc_kernel", other, str(rec)) is None
    rec.write_text(rec.read_text().replace("source_hash: ", "source_hash: 0"))
    assert bench.recorded_traffic("decode_tc_kernel", shape, str(rec)) is None
    assert bench.recorded_traffic("verify_tc_kernel", shape, str(rec)) is None


def test_traffic_record_of_a_kernel_mode(tmp_path):
    # a second record of one kernel (its sparse mode) is keyed by its own name
    # but checked against the kernel's source hash
    k = "swa_fwd_tc_global_kernel"
    shape = bench.traffic_shape(B=1, T=32768, Hq=64, Hkv=8, D=128, QB=64, topk=16)
    rec = tmp_path / "traffic.txt"
    rec.write_text(f"{k}.bytes_per_launch: 111\n"
                   f"{k}.source_hash: {bench.kernel_source_hash(k)}\n"
                   f"{k}.shape: B1 T32768 Hq64 Hkv8 D128 W32768\n"
                   f"{k}.sparse.bytes_per_launch: 222\n"
                   f"{k}.sparse.source_hash: {bench.kernel_source_hash(k)}\n"
                   f"{k}.sparse.shape: {shape}\n")
    assert bench.recorded_traffic(k, shape, str(rec), record=f"{k}.sparse") == 222
    assert bench.recorded_traffic(k, shape, str(rec)) is None
    assert bench.recorded_traffic(k, "B1 T32768 Hq64 Hkv8 D128 W32768", str(rec)) == 111
