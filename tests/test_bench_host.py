"""Host-side arithmetic of bench.py, on CPU: the roofline fraction and the
peak it is taken against, the throttle reasons read from nvidia-smi clock
samples, and the DRAM traffic that is reported only while the CUDA sources
are the ones it was measured on.  No GPU."""
import bench

PEAKS = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1500.0, "source": "measured"}


def test_hbm_roofline_is_algorithmic_bytes_over_event_time():
    # two launches per step of 1e9 and 5e8 elements at 4 and 2 bytes each,
    # CUDA-event times (ms) of two steps, interleaved launch by launch
    units = [(4.0, 1e9), (2.0, 5e8)]
    times = [1.0, 0.25, 1.2, 0.35]
    r = bench.roofline_of("nvfp4_quantize_requant", times, units, 2, PEAKS)
    byts = 4.0 * 1e9 + 2.0 * 5e8
    ms = (1.0 + 1.2) / 2 + (0.25 + 0.35) / 2
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert abs(r["achieved"] - byts / (ms / 1e3) / 1e9) < 1e-6
    assert r["peak"] == 6000.0 and abs(r["frac"] - r["achieved"] / 6000.0) < 1e-12
    assert r["algorithmic_bytes_per_step"] == byts


def test_tensor_roofline_takes_the_dtype_peak():
    fl = [2e12, 1e12]
    times = [1.0, 0.5]
    fp8 = bench.roofline_of("grouped_gemm_mxfp8_dw", times, fl, 1, PEAKS)
    fp4 = bench.roofline_of("grouped_gemm_nvfp4_fwd", times, fl, 1, PEAKS)
    assert fp8["bound"] == fp4["bound"] == "tensor"
    assert abs(fp8["achieved"] - 3e12 / 1.5e-3 / 1e12) < 1e-9
    # the sustained bf16 figure times the nominal dense ratios 4.5/2.25 and 13.5/2.25
    assert abs(fp8["peak"] - 1500.0 * 2.0) < 1e-9
    assert abs(fp4["peak"] - 1500.0 * 6.0) < 1e-9
    assert abs(fp4["frac"] - fp4["achieved"] / 9000.0) < 1e-12


class _Proc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0

    def kill(self):
        pass


class _Thread:
    def join(self, timeout=None):
        pass


def _stopped(lines):
    cs = bench.ClockSampler()
    cs.proc, cs.t, cs.lines = _Proc(), _Thread(), lines
    return cs.stop()


def test_clock_samples_give_median_max_and_reasons():
    idle = "Not Active"
    lines = [
        f"0, 2070, 2070, 900.5, 0x0, {idle}, {idle}, {idle}, {idle}",
        f"0, 1950, 2070, 1390.0, 0x4, {idle}, {idle}, {idle}, Active",
        f"0, 2040, 2070, 1200.0, 0x0, {idle}, {idle}, {idle}, {idle}",
        "garbled line",
    ]
    c = _stopped(lines)
    assert c["sm_mhz"] == 2040.0 and c["sm_max_mhz"] == 2070.0 and c["samples"] == 3
    assert c["reasons"] == ["sw_power_cap"]
    hot = _stopped([f"0, 1500, 2070, 1400.0, 0x40, {idle}, Active, Active, {idle}"])
    assert hot["reasons"] == ["hw_thermal_slowdown", "sw_thermal_slowdown"]


def test_clocks_without_nvidia_smi_say_so():
    assert bench.ClockSampler().stop()["reasons"] == ["nvidia-smi unavailable"]


def _traffic_file(tmp_path, digest):
    p = tmp_path / "traffic.txt"
    p.write_text("# header\n# source-sha256: " + digest + "\n"
                 "nvfp4_quantize_requant 0 300 100\n"
                 "grouped_gemm_mxfp8_dw 0 7 8\n"
                 "nvfp4_quantize_requant 1 100 100\n")
    return str(p)


def test_traffic_is_the_mean_per_call_while_the_sources_match(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "TRAFFIC_FILE", _traffic_file(tmp_path, bench.source_digest()))
    assert bench.measured_traffic("nvfp4_quantize_requant") == 300.0
    assert bench.measured_traffic("grouped_gemm_mxfp8_dw") == 15.0
    assert bench.measured_traffic("grouped_gemm_mxfp8_dx") is None


def test_traffic_of_other_sources_is_not_reported(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "TRAFFIC_FILE", _traffic_file(tmp_path, "0" * 64))
    assert bench.measured_traffic("nvfp4_quantize_requant") is None
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tmp_path / "missing.txt"))
    assert bench.measured_traffic("nvfp4_quantize_requant") is None

