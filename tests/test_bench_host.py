"""bench.py's host-side logic on the CPU: arguments, the whole-job
aggregate, the traffic record gated on the kernel sources, and the clock
record that decides whether a timed run is rejected."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_arguments():
    a = bench.parse_args([])
    assert (a.gpus, a.workload, a.impl, a.scan_mode) == (1, "l1b5", "ours", "auto")
    assert a.warmup >= 3
    with pytest.raises(SystemExit):
        bench.parse_args(["--warmup", "2"])
    with pytest.raises(SystemExit):
        bench.parse_args(["--workload", "nope"])
    for w in ("tiny", "l169m", "l1b5", "long", "l169m_bf16", "l169m_gated", "decode", "decode_bf16", "shift", "cmix"):
        assert bench.parse_args(["--workload", w]).workload == w
        assert w in bench.DEFAULT_STEPS


def test_aggregate_one_rank():
    value, t = bench.aggregate(2.0, 100.0, 1)
    assert (value, t) == (50.0, 2.0)


def test_traffic_record_follows_the_sources(tmp_path, monkeypatch):
    rec = {"seq_bwd_kernel@l169m": {"source_hash": "abc", "dram_bytes_per_launch": 123}}
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "ncu_traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", tmp_path)
    monkeypatch.setattr(bench, "kernel_source_hash", lambda kernel=None: "abc")
    assert bench.ncu_traffic("seq_bwd_kernel", "l169m") == 123
    assert bench.ncu_traffic("seq_fwd_kernel", "l169m") is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda kernel=None: "changed")
    assert bench.ncu_traffic("seq_bwd_kernel", "l169m") is None
    (tmp_path / "profiles" / "ncu_traffic.json").unlink()
    assert bench.ncu_traffic("seq_bwd_kernel", "l169m") is None


def test_source_hash_covers_the_kernel_sources():
    h = bench.kernel_source_hash()
    assert len(h) == 16 and h == bench.kernel_source_hash()
    # a kernel's hash covers its own files only: every listed file exists,
    # and the sequential and decode kernels hash differently
    csrc = bench.ROOT / "rwkv_linear_attention_backward_b300" / "csrc"
    for files in bench.KERNEL_FILES.values():
        assert all((csrc / f).exists() for f in files)
    assert bench.kernel_source_hash("seq_bwd_kernel") == bench.kernel_source_hash("seq_fwd_kernel")
    assert bench.kernel_source_hash("seq_bwd_kernel") != bench.kernel_source_hash("decode_kernel_vec4<float>")


def _sampler(samples, reasons, max_mhz=2032.0):
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.samples, s.reasons, s.max_mhz, s.source, s.error = list(samples), set(reasons), max_mhz, "test", None
    return s


def test_clock_rejection():
    assert not _sampler([2032] * 5, []).rejected()
    assert not _sampler([1900] * 5, ["sw_power_cap"]).rejected()  # kept and noted
    for r in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"):
        assert _sampler([2032] * 5, [r]).rejected()
    assert _sampler([1000] * 5, []).rejected()  # stuck well below max with no reason: a clock lock
    assert not _sampler([1000] * 5, ["sw_power_cap"]).rejected()
    s = _sampler([2032, 2032, 1500], ["gpu_idle"]).summary()
    assert s["sm_mhz"] == 2032 and s["reasons"] == []  # idle is not a reason


def test_smi_lines_are_read():
    class Proc:
        stdout = ["2032, 2032, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n",
                  "garbage\n",
                  "1800, 2032, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n",
                  "1700, 2032, 0x0000000000000008, Active, Not Active, Not Active, Not Active\n"]

    s = _sampler([], [])
    s._proc = Proc()
    s._run_smi()
    assert s.samples == [2032.0, 1800.0, 1700.0]
    assert {"sw_power_cap", "hw_slowdown"} <= s.reasons
    assert s.rejected()


def test_ctypes_nvml_reads_through_the_library_calls():
    """The ctypes NVML binding (hosts without pynvml) passes the SM clock
    domain, returns what the library writes, takes the older name of the
    clock-event call when the newer one is missing, and raises on a
    non-zero status."""
    calls = []

    class FakeLib:
        def nvmlInit_v2(self):
            calls.append("init")
            return 0

        def nvmlDeviceGetHandleByIndex_v2(self, index, ref):
            ref._obj.value = 0x1234 + index.value
            return 0

        def nvmlDeviceGetClockInfo(self, h, domain, ref):
            assert h.value == 0x1234 and domain.value == 1
            ref._obj.value = 1965
            return 0

        def nvmlDeviceGetMaxClockInfo(self, h, domain, ref):
            ref._obj.value = 2032
            return 0

        def nvmlDeviceGetCurrentClocksThrottleReasons(self, h, ref):
            ref._obj.value = 0x4 | 0x8
            return 0

    nv = bench.CtypesNvml(FakeLib())
    assert calls == ["init"]
    h = nv.nvmlDeviceGetHandleByIndex(0)
    assert nv.nvmlDeviceGetClockInfo(h, nv.NVML_CLOCK_SM) == 1965
    assert nv.nvmlDeviceGetMaxClockInfo(h, nv.NVML_CLOCK_SM) == 2032
    assert nv.nvmlDeviceGetCurrentClocksEventReasons(h) == 0xC

    class Failing(FakeLib):
        def nvmlDeviceGetClockInfo(self, h, domain, ref):
            return 3

    nv = bench.CtypesNvml(Failing())
    with pytest.raises(RuntimeError, match="status 3"):
        nv.nvmlDeviceGetClockInfo(nv.nvmlDeviceGetHandleByIndex(0), nv.NVML_CLOCK_SM)
