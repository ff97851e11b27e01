"""Host-side arithmetic of bench.py, on CPU: the roofline fraction and the
peak it is taken against, the throttle reasons read from nvidia-smi clock
samples, the DRAM traffic that is reported only while the CUDA sources are
the ones it was measured on, and the MoE step's per-call bytes, FLOPs and
launch count.  No GPU."""
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



# --- the MoE step's accounting: per-call units and the launch count ----------
from types import SimpleNamespace

from precision_moe_numerics_nvfp4_gb300 import pipeline as PL


def _layer(**kw):
    """The attributes MoELayer's accounting reads, without allocating (the
    MoE step's shape and default choices)."""
    base = dict(M=131072, d=4096, I=1536, E=64, fuse_swiglu=True, fuse_requant=True, fuse_swiglu_bwd=True,
                per_token=False, four_six=False, side=None, gathers_rows=True)
    base.update(kw)
    lay = SimpleNamespace(**base)
    lay.flops = lambda: PL.MoELayer.flops(lay)
    return lay


def test_gather_bytes_count_every_tensor_of_the_call():
    """The gathered quantization's algorithmic bytes, summed tensor by tensor:
    the tokens read by the amax pass and by their quantization, their NVFP4
    codes and scales written once, then per routed row the token's codes and
    scales read, copied to the routed layout and re-quantized to MXFP8 (one
    byte per value plus one E8M0 scale per 32)."""
    T, M, d = 16384, 131072, 4096
    nv = d / 2 + d / 16           # NVFP4 bytes of one row: codes and E4M3 scales
    mx = d + d / 32               # MXFP8 bytes of one row
    total = T * (2 * d) + T * (2 * d + nv) + M * (nv + nv + mx)
    assert abs(bench.gather_bytes_per_routed_elem(T, M) * M * d - total) < 1e-6 * total
    # more tokens than rows: the routed rows themselves read twice (amax, quantize)
    total_rows = M * (2 * d + 2 * d + nv + mx)
    assert abs(bench.gather_bytes_per_routed_elem(4 * M, M) * M * d - total_rows) < 1e-6 * total_rows


def test_gemm_units_add_up_to_the_step_flops_once_each():
    m = SimpleNamespace(x=SimpleNamespace(shape=(16384, 4096)))
    lay = _layer()
    units = bench.kernel_units(lay, m)
    gemm = [f for k, v in units.items() if k.startswith("grouped_gemm") for f in v]
    assert abs(sum(gemm) - sum(lay.flops())) < 1e-6 * sum(lay.flops())
    # the fused w2 dgrad carries the SwiGLU backward: no separate call is counted
    assert "nvfp4moe_swiglu_bwd" not in units and len(units["grouped_gemm_mxfp8_dx_swiglu_bwd"]) == 1
    # three quantize + requant calls (w13, w2, h) and one gathered x
    assert len(units["nvfp4_quantize_requant"]) == 3 and len(units["nvfp4_quantize_requant_gather"]) == 1


def test_launches_of_the_default_step():
    """21 kernels: w13 and w2 (amax, finalize, quantize + requant: 3 each); x
    from its tokens (token maxima, their maximum over the row map, finalize,
    the tokens' NVFP4 pass, the routed rows' copy + requant: 5); the w13 GEMM
    with SwiGLU and its outer-scale kernel (2); h's quantize + requant (1);
    the w2 GEMM (1); two gradient quantizations (2); four backward GEMMs, the
    w2 dgrad carrying the SwiGLU backward (4)."""
    lay = _layer()
    assert PL.MoELayer.launches_per_step(lay, gathered=True, tokens=16384) == 3 + 3 + 5 + 2 + 1 + 1 + 2 + 4
    # the unfused SwiGLU backward adds its own kernel
    assert PL.MoELayer.launches_per_step(_layer(fuse_swiglu_bwd=False), gathered=True, tokens=16384) == 22
