"""The benchmark's host logic on CPU: the reference arm's JSON line, the byte arithmetic of the
roofline, the gate on committed ncu counters and the clock record's parsing."""
import hashlib
import json
import os
import subprocess
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from routed_moe_fp4_gb300 import synthetic as S  # noqa: E402


def _run_bench(*args, env_extra=None):
    env = dict(os.environ, **(env_extra or {}))
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, env=env,
                          capture_output=True, text=True, timeout=600)


def test_reference_arm_prints_one_contract_line():
    p = _run_bench("--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "1")
    assert p.returncode == 0, p.stderr
    lines = [ln for ln in p.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "tokens/s"
    assert d["steps"] == 2 and d["warmup"] == 3          # warm-up is raised to at least 3
    assert d["value"] > 0 and d["higher_is_better"] is True and d["n_gpus"] == 1
    assert abs(d["value"] - 4 / (d["ms_per_step"] * 1e-3)) < 1e-6 * d["value"]
    assert d["config"]["workload"].startswith("tiny:")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_exit_quietly():
    p = _run_bench("--impl", "reference", "--workload", "tiny", "--steps", "1",
                   env_extra={"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert p.returncode == 0, p.stderr
    assert p.stdout.strip() == ""


def _routing(wl, touched):
    cnt = np.zeros(wl.E + 1, np.int32)
    cnt[:touched] = 1
    return {"cnt": cnt}


def test_layer_bytes_match_the_expert_sizes():
    # one expert's three MXFP4 matrices, H*I*(1/2 + 1/32) bytes each, worked out by hand:
    # 3 x 4096 x 2048 x 17/32 = 13,369,344 B and 3 x 7168 x 2048 x 17/32 = 23,396,352 B
    for name, per_expert in (("decode", 13_369_344), ("skewed", 23_396_352)):
        wl = S.WORKLOADS[name]
        for touched in (1, 62, wl.E):
            b = bench.algorithmic_bytes(wl, _routing(wl, touched))
            assert b["touched_experts"] == touched
            extra = wl.E * wl.H * 4 + 2 * wl.T * wl.H * 2          # router weights, x in, out
            assert b["layer"] == (touched + 1) * per_expert + extra


def test_gate_up_and_down_bytes_split_the_weights():
    wl = S.WORKLOADS["decode"]
    b = bench.algorithmic_bytes(wl, _routing(wl, 62))
    rows = wl.T * wl.top_k + wl.T
    # four E2M1 terms of x and of h, each with a UE8M0 byte per 32
    x_terms = 4 * rows * (wl.H // 2 + wl.H // 32)
    h_terms = 4 * rows * (wl.I // 2 + wl.I // 32)
    gu_w = 63 * 2 * wl.I * (wl.H // 2 + wl.H // 32)
    dn_w = 63 * wl.H * (wl.I // 2 + wl.I // 32)
    assert b["ffn_gate_up"] == gu_w + x_terms + h_terms
    assert b["ffn_down"] == dn_w + h_terms + rows * wl.H * 4
    assert gu_w + dn_w == 63 * 13_369_344
    # NVFP4: scale bytes per 16 elements
    b3 = bench.algorithmic_bytes(wl, _routing(wl, 62), path="nvf4", group=16)
    assert b3["layer"] - b["layer"] == 63 * 3 * wl.H * wl.I // 32


def test_committed_counters_are_used_only_for_the_source_they_were_taken_on(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    src_dir = tmp_path / "routed_moe_fp4_gb300" / "csrc"
    src_dir.mkdir(parents=True)
    src = src_dir / "kern.cu"
    src.write_bytes(b"__global__ void k() {}\n")
    prof = {"source_sha256": hashlib.sha256(src.read_bytes()).hexdigest(),
            "gate_up": {"dram_read_bytes": 1000, "dram_write_bytes": 24}}
    (tmp_path / "profiles" / "kern_decode.json").write_text(json.dumps(prof))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("kern", "decode") == 1024
    assert bench.profiled_traffic("kern", "prefill") is None          # no counters for it
    src.write_bytes(b"__global__ void k() { }\n")                       # the kernel changed
    assert bench.profiled_traffic("kern", "decode") is None


def test_committed_decode_counters_name_an_existing_source():
    with open(os.path.join(ROOT, "profiles", "gemm_mx4_decode.json")) as f:
        prof = json.load(f)
    assert len(prof["source_sha256"]) == 64
    assert prof["gate_up"]["dram_read_bytes"] > 0


class _FakeProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def test_clock_record_parsing():
    cs = bench.ClockSampler(0)
    cs.proc = _FakeProc()
    cs.lines = [
        "0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 2055, 2070, 1350.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 1980, 2070, 1399.0, 0x4, Not Active, Not Active, Not Active, Active",
        "garbled line",
        "0, [N/A], 2070, 0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    r = cs.stop()
    assert r["sm_mhz"] == 2055 and r["sm_max_mhz"] == 2070 and r["samples"] == 3
    assert r["reasons"] == ["sw_power_cap"]
    cs2 = bench.ClockSampler(0)
    cs2.proc = _FakeProc()
    cs2.lines = ["0, 1500, 2070, 800, 0x8, Active, Not Active, Active, Not Active"]
    assert cs2.stop()["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]


def test_clock_record_without_nvidia_smi():
    assert bench.ClockSampler(0).stop()["reasons"] == ["nvidia-smi unavailable"]


def test_ffn_path_names_are_unique_per_abi_value():
    abi = [v[0] for v in bench.FFN_PATHS.values() if v[0] is not None]
    assert len(abi) == len(set(abi))
    assert bench.PATH_BY_ABI[2] == "mxf4" and "nvf4" not in bench.PATH_BY_ABI.values()



class _FakeNvml:
    """Stands in for libnvidia-ml: a GPU found by UUID, an SM clock sequence and reason bits."""

    def __init__(self, clocks, reasons, uuid="GPU-abc"):
        self.clocks, self.reasons, self.uuid = list(clocks), list(reasons), uuid
        self.i = 0
        self.shutdown = False

    def nvmlInit_v2(self):
        return 0

    def nvmlDeviceGetHandleByUUID(self, u, h):
        if u.decode() != self.uuid:
            return 13
        h._obj.value = 1234
        return 0

    def nvmlDeviceGetHandleByPciBusId_v2(self, bus, h):
        return 13

    def nvmlDeviceGetHandleByIndex_v2(self, i, h):
        return 13

    def nvmlDeviceGetMaxClockInfo(self, h, kind, out):
        out._obj.value = 2070
        return 0

    def nvmlDeviceGetClockInfo(self, h, kind, out):
        out._obj.value = self.clocks[min(self.i, len(self.clocks) - 1)]
        return 0

    def nvmlDeviceGetCurrentClocksEventReasons(self, h, out):
        out._obj.value = self.reasons[min(self.i, len(self.reasons) - 1)]
        self.i += 1
        return 0

    def nvmlShutdown(self):
        self.shutdown = True
        return 0


def _poll(fake, ids, n):
    import time
    p = bench.NvmlPoller(ids, lib=fake, period_s=0.0005)
    assert p.start()
    t0 = time.perf_counter()
    while len(p.samples) < n and time.perf_counter() - t0 < 5:
        time.sleep(0.001)
    return p.stop()


def test_nvml_poller_reads_clocks_and_reasons():
    fake = _FakeNvml([2070, 2055, 1980, 2070], [0x1, 0x4, 0x4 | 0x40, 0x0])
    r = _poll(fake, [("pci", "0:1:0.0"), ("uuid", "GPU-abc")], 4)
    assert fake.shutdown and r["samples"] >= 4 and r["sm_max_mhz"] == 2070
    assert r["sm_min_mhz"] == 1980 and 1980 <= r["sm_mhz"] <= 2070
    # the idle bit (0x1) is not a slowdown; power cap and hardware thermal are
    assert r["reasons"] == ["sw_power_cap", "hw_thermal_slowdown"]


def test_nvml_poller_without_a_matching_device():
    p = bench.NvmlPoller([("uuid", "GPU-other"), ("index", 3)], lib=_FakeNvml([2070], [0]))
    assert not p.start() and p.error and p.stop() is None


def test_clock_record_prefers_the_in_region_nvml_samples():
    c = bench.Clocks(0, nvml_lib=_FakeNvml([1900], [0x8]), smi=False, ids=[("uuid", "GPU-abc")])
    c.start()
    import time
    time.sleep(0.02)
    r = c.stop()
    assert r["source"].startswith("NVML") and r["sm_mhz"] == 1900 and r["reasons"] == ["hw_slowdown"]
    # no NVML: the record says where its numbers come from
    c2 = bench.Clocks(0, nvml_lib=_FakeNvml([1900], [0], uuid="GPU-x"), smi=False, ids=[("uuid", "GPU-y")])
    c2.start()
    r2 = c2.stop()
    assert r2["sm_mhz"] is None and "no NVML handle" in r2["source"]


def test_layer_flops_match_the_closed_form():
    # algorithmic flops = T (k + 1) 6 H I + 2 T E H, worked out by hand per workload: decode
    # 8 x 9 x 6 x 4096 x 2048 + 2 x 8 x 256 x 4096 = 3.64 GFLOP, skewed 3.262 TFLOP, ...
    for name, gflop, rel in (("decode", 3.6, 0.02), ("prefill", 233.0, 0.005), ("skewed", 3262.0, 0.001),
                             ("sweep_T1", 0.79, 0.02), ("sweep_T128", 101.5, 0.005)):
        got = bench.algorithmic_flops(S.WORKLOADS[name]) / 1e9
        assert abs(got - gflop) <= rel * gflop, (name, got)


def test_layer_roofline_takes_the_binding_bound():
    # decode-like: bytes bind; 847 MB in 0.18 ms against 6782 GB/s
    r = bench.layer_roofline(846_594_048, 3.64e9, 0.18, 6782.1, 1879.7, "measured")
    assert r["binding"] == "hbm" and abs(r["frac"] - 846_594_048 / 0.18e-3 / 6782.1e9) < 1e-12
    assert r["frac_combined"] == r["frac"] and r["fp4_peak_tflops"] == 1879.7 * 6
    # compute-heavy: 3.26 TFLOP and 1 GB in 1 ms; the FP4 bound (0.289 ms) exceeds the HBM one
    r = bench.layer_roofline(1_000_000_000, 3.26e12, 1.0, 6782.1, 1879.7, "measured")
    assert r["binding"] == "tensor"
    assert abs(r["frac_combined"] - 3.26e12 / (1879.7 * 6e12) / 1e-3) < 1e-12
    assert abs(r["tensor_frac"] - r["frac_combined"]) < 1e-12


def test_cpu_model_on_an_arm_host_without_a_model_name(tmp_path, monkeypatch):
    """Grace's /proc/cpuinfo has no "model name": the model comes from lscpu, else from the Arm part."""
    import subprocess
    info = tmp_path / "cpuinfo"
    info.write_text("processor\t: 0\nBogoMIPS\t: 2000.00\nCPU implementer\t: 0x41\nCPU architecture: 8\n"
                    "CPU part\t: 0xd4f\n")

    def no_lscpu(*a, **k):
        raise OSError("no lscpu")
    monkeypatch.setattr(subprocess, "run", no_lscpu)
    assert bench.cpu_model(str(info)) == "Arm Neoverse-V2"

    class Out:
        stdout = "Architecture: aarch64\nModel name:   Neoverse-V2\n"
    monkeypatch.setattr(subprocess, "run", lambda *a, **k: Out())
    assert bench.cpu_model(str(info)) == "Neoverse-V2"
    x86 = tmp_path / "cpuinfo_x86"
    x86.write_text("processor\t: 0\nmodel name\t: Example CPU @ 3.0GHz\n")
    assert bench.cpu_model(str(x86)) == "Example CPU @ 3.0GHz"


def test_config_targets_follow_the_scope_table():
    """Decode shapes are judged against HBM at 0.70, the prefill shapes against the combined
    roofline at 0.50; the pass covers every configuration beside the headline decode."""
    assert bench.config_target("prefill") == ("frac_combined", 0.50)
    assert bench.config_target("skewed") == ("frac_combined", 0.50)
    for t in S.SWEEP_T:
        assert bench.config_target(f"sweep_T{t}") == ("frac", 0.70)
    assert bench.config_target("v4pro_decode") == ("frac", 0.70)
    assert set(bench.CONFIG_PASS) == {"prefill", "skewed", "v4pro_decode"} | {f"sweep_T{t}" for t in S.SWEEP_T}
