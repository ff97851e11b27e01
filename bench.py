"""Benchmark of the NVFP4-forward / MXFP8-backward expert hot path on GB300.

One step = one pass of the whole path over one batch: the routed experts of a
MoE layer with 16384 tokens, d_model 4096, 64 experts, top-8 routing and
SwiGLU experts (gate/up 4096 -> 1536 x 2, down 1536 -> 4096), forward and
backward:
  forward   NVFP4 quantization of x, w13, w2 (amax -> FP32 outer scale ->
            1x16 E4M3 block scales -> E2M1), grouped NVFP4 GEMM w13, SwiGLU,
            NVFP4 quantization of h, grouped NVFP4 GEMM w2
  backward  dequant -> transpose -> SR requant to MXFP8 of w13, w2, x_q, h_q;
            SR MXFP8 quantization (row-wise + transposed per expert) of the
            down-output gradient g2 and of dy13; grouped MXFP8 dgrad and wgrad
            GEMMs for the down and gate/up projections; SwiGLU backward.
Inputs are seeded synthetic tensors of that shape (the pages measure on no
public dataset): x ~ N(0,1), weights ~ N(0,0.02), router logits and bias
~ N(0,1), g2 ~ N(0,1e-3).

value  = GEMM FLOPs of the step (forward + backward, unpadded groups) / step
         time, with inputs resident in HBM, in TFLOP/s.
e2e    = the same, with every step's activations and upstream gradient copied
         from pinned host memory and its dx read back inside the timed region;
         the copies of neighbouring steps overlap the compute
         (pipeline.HostStaged: one copy stream per direction, two slots).
roofline: the kernel with the largest share of the step, achieved against
         MEASURED_PEAKS.json (HBM GB/s, bf16 TFLOP/s x the nominal fp8/fp4
         ratio) or the documented fallback.

--impl reference times the CPU oracle (oracle/, numpy) on a bounded sample of
the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "NVFP4/MXFP8 expert GEMM TFLOPS + quant/requant GB/s, % of GB300 roofline"
WORKLOAD = "moe_expert_layer_fwd_bwd: 16384 tokens x top-8 (131072 rows), d_model 4096, d_ff 1536, 64 experts"
SHAPE = dict(tokens=16384, topk=8, d_model=4096, d_ff=1536, experts=64)

# fallbacks when MEASURED_PEAKS.json is absent (one earlier GB300 measurement)
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
NOMINAL_RATIO = {"bf16": 1.0, "fp8": 4.5 / 2.25, "fp4": 13.5 / 2.25}


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic_moe_layer_fwd_bwd.txt")


def source_digest():
    """sha256 over the library's CUDA sources and its header: DRAM counters
    taken from an older build no longer describe the kernels."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "precision_moe_numerics_nvfp4_gb300", "csrc")
    files = sorted(os.path.join(csrc, f) for f in os.listdir(csrc) if f.endswith((".cu", ".cuh", ".h")))
    for f in files + [os.path.join(ROOT, "include", "nvfp4moe.h")]:
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def measured_traffic(entry_point):
    """DRAM bytes (read + write) per launch of `entry_point` in the MoE step,
    averaged over its calls, from the committed one-pass ncu capture; None
    when the capture is missing or was taken from different sources."""
    try:
        with open(TRAFFIC_FILE) as fh:
            lines = fh.read().splitlines()
    except OSError:
        return None
    digest = next((l.split(":", 1)[1].strip() for l in lines if l.startswith("# source-sha256:")), None)
    if digest != source_digest():
        return None
    vals = []
    for l in lines:
        f = l.split()
        if len(f) == 4 and not l.startswith("#") and f[0] == entry_point:
            vals.append(int(f[2]) + int(f[3]))
    return sum(vals) / len(vals) if vals else None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            return {
                "hbm_gbs": float(d.get("hbm_gbs", FALLBACK["hbm_gbs"])),
                "bf16_tflops": float(d.get("bf16_tflops", FALLBACK["bf16_tflops"])),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d.get("bf16_tflops", 1700.0))),
                "source": "measured",
            }
        except Exception:
            pass
    return dict(FALLBACK, source="fallback")


# ---------------------------------------------------------------------------
# distributed plumbing (replicas: one process per GPU, no data-path collective)
# ---------------------------------------------------------------------------
def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def init_dist(backend):
    import torch.distributed as dist
    rank, world, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return rank, world


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(x: float, device=None) -> float:
    """Largest value of x over all ranks (the slowest replica sets the time)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(units_per_rank: float, seconds_max: float, world: int) -> float:
    """Whole-job throughput: units all ranks processed / the slowest rank's time."""
    return units_per_rank * world / seconds_max


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index=0, out_path=None):
        self.gpu, self.out_path, self.proc, self.lines = gpu_index, out_path, None, []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        if self.out_path:
            with open(self.out_path, "w") as f:
                f.write(self.FIELDS + "\n" + "\n".join(self.lines) + "\n")
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
class EventLog:
    """CUDA events around each library call on the launching stream."""

    def __init__(self):
        self.rec = []

    def call(self, name, fn, *a, **k):
        import torch
        s = k.get("stream")  # the call's own stream when it names one, else the current one
        if s is None:
            s = next((v for v in a if isinstance(v, torch.cuda.Stream)), None)
        if s is None:
            s = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        r = fn(*a, **k)
        e1.record(s)
        self.rec.append((name, e0, e1))
        return r

    def per_name_ms(self):
        out = {}
        for name, e0, e1 in self.rec:
            out.setdefault(name, []).append(e0.elapsed_time(e1))
        return out


def build_step(layer, m, log: EventLog | None, only: str | None = None):
    """Returns step() running the whole path; with `log`, each call (or each
    call of the entry point `only`) is bracketed by events."""
    from precision_moe_numerics_nvfp4_gb300 import nvfp4moe as N
    from precision_moe_numerics_nvfp4_gb300 import pipeline as PL

    def wrap(name, fn):
        if log is None or (only is not None and name != only):
            return fn
        return lambda *a, **k: log.call(name, fn, *a, **k)

    class Proxy:  # the layer's launching calls go through the event log (size queries do not)
        def __getattr__(self, n):
            f = getattr(N, n)
            return wrap(n, f) if callable(f) and not n.startswith("_") and not n.endswith("_bytes") else f

    rows = m.rows if layer.gathers_rows else None

    def step(x, g2):  # x: the tokens (the x quantization gathers the routed rows), else the routed rows
        saved = PL.N
        PL.N = Proxy()
        try:
            layer.step(x, m.w13, m.w2, g2, m.group_offsets, seed=3, x_rows=rows)
        finally:
            PL.N = saved

    return step


def gather_bytes_per_routed_elem(T, M):
    """Algorithmic bytes per routed-row element of nvfp4_quantize_requant_gather
    with T tokens and M routed rows."""
    if T <= M:  # tokens quantized once, routed rows copied + re-quantized from their codes
        return 0.5625 + 0.5625 + 1.03125 + (2.0 + 2.5625) * T / M
    return 3.59375 + 2.0  # routed rows read by the amax pass and by the quantize pass


def kernel_units(layer, m):
    """Algorithmic bytes (quantizers) and FLOPs (GEMMs) per call, by call name
    and argument pattern, in the order MoELayer.step issues them."""
    units = _kernel_units(layer, m)
    if getattr(layer, "fuse_swiglu_bwd", False):
        # the w2 dgrad carries the SwiGLU backward in its epilogue: its own
        # entry point (counted by its FLOPs), no separate SwiGLU backward call
        fl2, fl13 = units["grouped_gemm_mxfp8_dx"]
        units["grouped_gemm_mxfp8_dx_swiglu_bwd"] = [fl2]
        units["grouped_gemm_mxfp8_dx"] = [fl13]
        del units["nvfp4moe_swiglu_bwd"]
    return units


def _kernel_units(layer, m):
    M, d, I, E = layer.M, layer.d, layer.I, layer.E
    T = m.x.shape[0]  # tokens
    fl13 = 2.0 * M * 2 * I * d
    fl2 = 2.0 * M * d * I
    # quantize (+ requant) of h: no amax pass when the w13 epilogue produced its outer scale
    h_amax = 0.0 if layer.fuse_swiglu else 2.0
    side = getattr(layer, "side", None) is not None
    if side or getattr(layer, "four_six", False):
        # side stream: the amax passes of w13, w2 and x are nvfp4_outer_scale
        # calls and the quantize calls take the scales as given; Four Over Six:
        # the activation calls have their own names
        a = 0.0 if side else 2.0
        act = "_four_over_six" if getattr(layer, "four_six", False) else ""
        q, qr = (2.5625, 3.59375)
        w_q = [(E * 2 * I * d, q + a), (E * d * I, q + a)]
        w_qr = [(E * 2 * I * d, qr + a), (E * d * I, qr + a)]
        x_q = [(M * d, q + a), (M * I, q + h_amax)]
        x_qr = [(M * d, qr + a), (M * I, qr + h_amax)]
        units = {
            "grouped_gemm_nvfp4_fwd": [fl2] if layer.fuse_swiglu else [fl13, fl2],
            "grouped_gemm_nvfp4_fwd_swiglu": [fl13],
            "dequant_transpose_requant_sr": [(E * 2 * I * d, 1.59375), (E * d * I, 1.59375), (M * d, 1.59375),
                                             (M * I, 1.59375)],
            "mxfp8_quantize": [(M * d, 4.0625), (M * 2 * I, 4.0625)],
            "grouped_gemm_mxfp8_dx": [fl2, fl13],
            "grouped_gemm_mxfp8_dw": [fl2, fl13],
            "nvfp4moe_swiglu_fwd": [(M * I, 3 * 2.0)],
            "nvfp4moe_swiglu_bwd": [(M * I, 5 * 2.0)],
        }
        if side:
            units["nvfp4_outer_scale"] = [(E * 2 * I * d, 2.0), (E * d * I, 2.0), (M * d, 2.0)]
        if act:
            units.update({"nvfp4_quantize": w_q, "nvfp4_quantize_requant": w_qr,
                          "nvfp4_quantize" + act: x_q, "nvfp4_quantize_requant" + act: x_qr})
        else:
            units.update({"nvfp4_quantize": w_q + x_q, "nvfp4_quantize_requant": w_qr + x_qr})
        return units
    if getattr(layer, "per_token", False):  # activations: the row amax pass (2 B/elem) runs inside the call
        return {
            "nvfp4_quantize_rows": [(M * d, 4.5625), (M * I, 2.5625 + h_amax)],
            "nvfp4_quantize_requant_rows": [(M * d, 5.59375), (M * I, 3.59375 + h_amax)],
            "nvfp4_quantize": [(E * 2 * I * d, 4.5625), (E * d * I, 4.5625)],
            "nvfp4_quantize_requant": [(E * 2 * I * d, 5.59375), (E * d * I, 5.59375)],
            "grouped_gemm_nvfp4_fwd_rows": [fl2] if layer.fuse_swiglu else [fl13, fl2],
            "grouped_gemm_nvfp4_fwd_swiglu_rows": [fl13],
            "dequant_transpose_requant_sr": [(E * 2 * I * d, 1.59375), (E * d * I, 1.59375)],
            "dequant_transpose_requant_sr_rows": [(M * d, 1.59375), (M * I, 1.59375)],
            "mxfp8_quantize": [(M * d, 4.0625), (M * 2 * I, 4.0625)],
            "grouped_gemm_mxfp8_dx": [fl2, fl13],
            "grouped_gemm_mxfp8_dw": [fl2, fl13],
            "nvfp4moe_swiglu_fwd": [(M * I, 3 * 2.0)],
            "nvfp4moe_swiglu_bwd": [(M * I, 5 * 2.0)],
        }
    return {
        # a call = the amax pass (2 B/elem) + the quantize pass (2 + 0.5 + 1/16 B/elem)
        "nvfp4_quantize": [(E * 2 * I * d, 4.5625), (E * d * I, 4.5625), (M * d, 4.5625), (M * I, 2.5625 + h_amax)],
        # amax pass (2) + one pass reading bf16 (2) and writing NVFP4 (0.5 + 1/16) and MXFP8 (1 + 1/32);
        # x: the tokens read by the amax pass (2 B per token element) and quantized once (2 + 0.5625),
        # then per routed-row element the token's NVFP4 codes and scales read (0.5625), copied to the
        # routed layout (0.5625) and re-quantized to MXFP8 (1 + 1/32)
        "nvfp4_quantize_requant": [(E * 2 * I * d, 5.59375), (E * d * I, 5.59375), (M * I, 3.59375 + h_amax)],
        "nvfp4_quantize_requant_gather": [(M * d, gather_bytes_per_routed_elem(T, M))],
        "grouped_gemm_nvfp4_fwd": [fl2] if layer.fuse_swiglu else [fl13, fl2],
        "grouped_gemm_nvfp4_fwd_swiglu": [fl13],
        "dequant_transpose_requant_sr": [(E * 2 * I * d, 1.59375), (E * d * I, 1.59375), (M * d, 1.59375),
                                         (M * I, 1.59375)],
        "mxfp8_quantize": [(M * d, 4.0625), (M * 2 * I, 4.0625)],
        "grouped_gemm_mxfp8_dx": [fl2, fl13],
        "grouped_gemm_mxfp8_dw": [fl2, fl13],
        "nvfp4moe_swiglu_fwd": [(M * I, 3 * 2.0)],
        "nvfp4moe_swiglu_bwd": [(M * I, 5 * 2.0)],
    }


def run_ours(args):
    import torch
    from precision_moe_numerics_nvfp4_gb300 import nvfp4moe as N
    from precision_moe_numerics_nvfp4_gb300 import workloads as W
    from precision_moe_numerics_nvfp4_gb300.pipeline import MoELayer

    rank, world = init_dist("nccl")
    _, _, local = dist_env()
    torch.cuda.set_device(local)
    N.lib()
    peaks = load_peaks()
    m = W.moe("cuda", seed=2, with_grad=True, grad_seed=3)
    M = m.x_perm.shape[0]
    layer = MoELayer(M, SHAPE["d_model"], SHAPE["d_ff"], SHAPE["experts"], per_token=args.per_token,
                     four_over_six=args.four_over_six)
    workload = WORKLOAD + (", per-token activation outer scales" if args.per_token else "") + (
        ", Four Over Six activation blocks" if args.four_over_six else "")
    fwd_fl, bwd_fl = layer.flops()
    step_flops = fwd_fl + bwd_fl
    x_in = m.x if layer.gathers_rows else m.x_perm  # the step's activation input

    # warm-up
    plain = build_step(layer, m, None)
    for _ in range(args.warmup):
        plain(x_in, m.g2)
    torch.cuda.synchronize()
    st = N.nvfp4moe_get_device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} after warm-up")

    # per-entry-point breakdown: untimed steps with an event pair around
    # every call (those events would add about 1% to a timed step)
    blog = EventLog()
    logged = build_step(layer, m, blog)
    n_logged = max(1, min(args.steps, 5))
    for _ in range(n_logged):
        logged(x_in, m.g2)
    torch.cuda.synchronize()
    per_all = blog.per_name_ms()
    dom = max(per_all, key=lambda k: sum(per_all[k]))

    # timed region: device-resident inputs; events only around the dominant
    # entry point's calls, for its roofline
    log = EventLog()
    step = build_step(layer, m, log, only=dom)
    sampler = ClockSampler(local, args.clocks_csv)
    sampler.start()
    barrier()
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(s)
    for _ in range(args.steps):
        step(x_in, m.g2)
    t1.record(s)
    torch.cuda.synchronize()
    barrier()
    clocks = sampler.stop()
    ms = t0.elapsed_time(t1) / args.steps
    ms_max = max_over_ranks(ms, torch.device("cuda"))
    value = aggregate(step_flops / 1e12, ms_max / 1e3, world)
    st = N.nvfp4moe_get_device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} after the timed region")

    # per-kernel breakdown (the logged steps; shares of the timed step)
    per = log.per_name_ms()
    units = kernel_units(layer, m)
    kernels = {}
    for name, times in per_all.items():
        n_per_step = len(units.get(name, [])) or 1
        tot = sum(times) / n_logged
        u = units.get(name, [])
        entry = {"ms_per_step": tot, "share": tot / ms, "calls_per_step": n_per_step}
        if u and isinstance(u[0], tuple):
            by = [sum(times[i::n_per_step]) / n_logged for i in range(n_per_step)]
            gbs = [uu[0] * uu[1] / (b / 1e3) / 1e9 for uu, b in zip(u, by)]
            entry.update({"GB_s": gbs, "frac_hbm": [g / peaks["hbm_gbs"] for g in gbs]})
        elif u:
            by = [sum(times[i::n_per_step]) / n_logged for i in range(n_per_step)]
            entry.update({"TFLOP_s": [f / (b / 1e3) / 1e12 for f, b in zip(u, by)]})
        kernels[name] = entry
    roof = roofline_of(dom, per[dom], units[dom], args.steps, peaks)
    roof["traffic"] = measured_traffic(dom)
    roof["traffic_unit"] = "bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum), null if stale"

    # e2e through host buffers: the tokens, their routed rows' source map and
    # g2 in, dx out, every step; the copies of neighbouring steps overlap the
    # compute (pipeline.HostStaged)
    from precision_moe_numerics_nvfp4_gb300.pipeline import HostStaged
    x_h = x_in.cpu().pin_memory()
    rows_h = m.rows.cpu().pin_memory() if layer.gathers_rows else None
    g_h = m.g2.cpu().pin_memory()
    dx_h = torch.empty(layer.dx.shape, dtype=layer.dx.dtype).pin_memory()
    staged = HostStaged(layer, tokens=m.x.shape[0] if layer.gathers_rows else None)
    staged.step(x_h, g_h, dx_h, m.w13, m.w2, m.group_offsets, seed=3, rows_h=rows_h)  # untimed: first use
    staged.synchronize()
    e2e_steps = max(2, min(args.steps, 20))  # the copy pipeline's fill and drain amortized as over the timed steps
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    staged.s_in.wait_event(e0)
    for _ in range(e2e_steps):
        last = staged.step(x_h, g_h, dx_h, m.w13, m.w2, m.group_offsets, seed=3, rows_h=rows_h)
    s.wait_event(last)
    e1.record(s)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, torch.device("cuda"))
    h2d, d2h = staged.bytes_per_step()
    st = N.nvfp4moe_get_device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} after the end-to-end steps")

    cpu = None
    if rank == 0 and not args.no_cpu_baseline and not args.per_token and not args.four_over_six:
        # the oracle step is the per-tensor, plain-rule one
        cpu = cpu_baseline(args.cpu_tokens)
    configs = None
    if not args.no_configs and not args.per_token and not args.four_over_six:
        del staged, x_h, rows_h, g_h, dx_h
        configs = other_configs(peaks, rank == 0 and not args.no_cpu_baseline)

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "nvfp4 fwd / mxfp8 bwd (fp32 accumulate)", "data": "synthetic",
        "config": {"workload": workload, "global_batch": SHAPE["tokens"] * world, "rows": M,
                   "group_sizes": "top-8 of logits~N(0,1)+bias~N(0,1), uneven", "seed": 2,
                   "parallelism": f"replicas x{world}", "l2": "inputs > L2 (GB-sized tensors), no flush",
                   "activations": ("per token [16384 x 4096]; the quantization of x gathers the routed rows"
                                   if layer.gathers_rows else "routed rows [T*k x 4096], already dispatched")},
        "gemm_flops_per_step": step_flops,
        "roofline": roof, "kernels": kernels, "clocks": clocks,
        "kernels_note": (f"per entry point: {n_logged} untimed steps with an event pair around every call; "
                         "shares of the timed step; the roofline's kernel timed live in the timed region"),
        "e2e": {"value": aggregate(step_flops / 1e12, e2e_ms / 1e3, world), "unit": "TFLOP/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "overlap": "copies in (step i+1) and out (step i-1) on their own streams during step i",
                "inputs": ("tokens x [16384 x 4096] bf16, the routed rows' source tokens (int32), g2 per routed row"
                           if layer.gathers_rows else "routed rows x [T*k x 4096] bf16, g2 per routed row")},
        "gpu_launches": layer.launches_per_step(gathered=layer.gathers_rows, tokens=m.x.shape[0]) * args.steps,
        "peaks": peaks,
        "cpu_baseline": cpu,
        "configs": configs,
    }
    if rank == 0:
        print(json.dumps(line))


def roofline_of(name, times, units, steps, peaks):
    n = len(units)
    per_launch = [sum(times[i::n]) / steps for i in range(n)]
    if isinstance(units[0], tuple):
        byts = sum(u[0] * u[1] for u in units)
        dur = sum(per_launch)
        ach = byts / (dur / 1e3) / 1e9
        return {"kernel": name, "bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": ach / peaks["hbm_gbs"], "traffic": None,
                "peak_source": peaks["source"] + " (HBM copy)", "algorithmic_bytes_per_step": byts}
    fl = sum(units)
    dur = sum(per_launch)
    ach = fl / (dur / 1e3) / 1e12
    ratio = NOMINAL_RATIO["fp4"] if "nvfp4" in name else NOMINAL_RATIO["fp8"]
    peak = peaks["bf16_tflops_sustained"] * ratio
    return {"kernel": name, "bound": "tensor", "achieved": ach, "peak": peak, "unit": "TFLOP/s",
            "frac": ach / peak, "traffic": None,
            "peak_source": f"{peaks['source']} sustained bf16 x {ratio:g} (nominal {'fp4' if ratio > 3 else 'fp8'}/bf16)",
            "algorithmic_flops_per_step": fl}


# ---------------------------------------------------------------------------
# the oracle: cpu_baseline and the reference arm
# ---------------------------------------------------------------------------
def oracle_sample_step(tokens: int, seed: int = 2, d_ff: int | None = None):
    """One expert (of the workload's 64) with `tokens` routed rows, full
    d_model and the first `d_ff` hidden features (all of them by default),
    through every step of the path in the oracle.  Returns the sample's GEMM
    FLOPs."""
    import torch
    from oracle import gemm as G
    from oracle import layout as L
    from oracle import mxfp8 as MX
    from oracle import nvfp4 as NV
    from oracle import requant as RQ
    from oracle import swiglu as SW
    d, I = SHAPE["d_model"], d_ff or SHAPE["d_ff"]
    gen = torch.Generator().manual_seed(seed)
    x = (torch.randn((tokens, d), generator=gen)).to(torch.bfloat16).float().numpy()
    w13 = (torch.randn((2 * I, d), generator=gen) * 0.02).to(torch.bfloat16).float().numpy()
    w2 = (torch.randn((d, I), generator=gen) * 0.02).to(torch.bfloat16).float().numpy()
    g2 = (torch.randn((tokens, d), generator=gen) * 1e-3).to(torch.bfloat16).float().numpy()
    o = np.array([0, tokens])
    P = L.padded_cap(tokens, 1)
    xc, xs, xsg = NV.quantize(x)
    w13c, w13s, w13sg = NV.quantize(w13)
    w2c, w2s, w2sg = NV.quantize(w2)
    y13, _ = G.grouped_rows(NV.dequantize_f64(xc, xs, xsg), NV.dequantize_f64(w13c, w13s, w13sg)[None], o)
    h = SW.forward(y13.astype(np.float32))
    hc, hs, hsg = NV.quantize(h.astype(np.float32))
    G.grouped_rows(NV.dequantize_f64(hc, hs, hsg), NV.dequantize_f64(w2c, w2s, w2sg)[None], o)
    w13t = RQ.requant_weights(w13c[None], w13s[None], np.array([w13sg]), 3, 0)
    w2t = RQ.requant_weights(w2c[None], w2s[None], np.array([w2sg]), 3, 1)
    xt = RQ.requant_grouped(xc, xs, xsg, o, 3, 2, P)
    ht = RQ.requant_grouped(hc, hs, hsg, o, 3, 3, P)
    gr = RQ.quantize_grad_rowwise(g2, 3, 4)
    gt = RQ.transposed_grouped_sr(g2, o, 3, 5, P)
    dh, _ = G.grouped_rows(MX.dequantize_f64(*gr), MX.dequantize_f64(w2t[0][0], w2t[1][0])[None], o)
    G.grouped_contraction(MX.dequantize_f64(*gt), MX.dequantize_f64(*ht), np.array([0, P]))
    dy13 = SW.backward(dh, y13).astype(np.float32)
    dr = RQ.quantize_grad_rowwise(dy13, 3, 6)
    dt = RQ.transposed_grouped_sr(dy13, o, 3, 7, P)
    G.grouped_rows(MX.dequantize_f64(*dr), MX.dequantize_f64(w13t[0][0], w13t[1][0])[None], o)
    G.grouped_contraction(MX.dequantize_f64(*dt), MX.dequantize_f64(*xt), np.array([0, P]))
    return 3 * (2.0 * tokens * 2 * I * d + 2.0 * tokens * d * I)


def cpu_baseline(tokens: int):
    t0 = time.perf_counter()
    flops = oracle_sample_step(tokens)
    dt = time.perf_counter() - t0
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"one expert of the workload with {tokens} routed rows, full d_model/d_ff, every step "
                      f"(quantize, GEMM references in float64, requant, SR) in numpy; {dt:.1f} s"}


# ---------------------------------------------------------------------------
# the oracle on the other workloads: bounded samples, timed on one host core
# and on all of them (spawned worker processes, one BLAS thread each)
# ---------------------------------------------------------------------------
def _oracle_single_linear(payload):
    """The single linear layer, forward and backward, through the oracle: NVFP4
    x and w, the FP64 forward GEMM, the SR re-quantization of both, the SR
    MXFP8 quantization of g (row-wise and transposed) and the two backward
    GEMMs.  Returns the GEMM FLOPs."""
    from oracle import gemm as G
    from oracle import layout as L
    from oracle import mxfp8 as MX
    from oracle import nvfp4 as NV
    from oracle import requant as RQ
    x, w, g = payload
    T, din = x.shape
    dout = w.shape[0]
    o = np.array([0, T])
    P = L.padded_cap(T, 1)
    xc, xs, xsg = NV.quantize(x)
    wc, ws, wsg = NV.quantize(w)
    G.grouped_rows(NV.dequantize_f64(xc, xs, xsg), NV.dequantize_f64(wc, ws, wsg)[None], o)
    wt = RQ.requant_weights(wc[None], ws[None], np.array([wsg]), 0, 0)
    xt = RQ.requant_grouped(xc, xs, xsg, o, 0, 1, P)
    gr = RQ.quantize_grad_rowwise(g, 0, 2)
    gt = RQ.transposed_grouped_sr(g, o, 0, 3, P)
    G.grouped_rows(MX.dequantize_f64(*gr), MX.dequantize_f64(wt[0][0], wt[1][0])[None], o)
    G.grouped_contraction(MX.dequantize_f64(*gt), MX.dequantize_f64(*xt), np.array([0, P]))
    return 3 * 2.0 * T * din * dout


def _oracle_quant_op(payload):
    """One op of the quantization sweep on a slice of rows; returns its
    algorithmic bytes (the GPU kernel's per-element figure x elements)."""
    from oracle import nvfp4 as NV
    from oracle import requant as RQ
    op, x, extra = payload
    n = x.size
    if op == "nvfp4_amax":  # far faster than the others: repeated so that the task outlasts its dispatch
        for _ in range(100):
            NV.outer_scale(x)
        return 100 * 2.0 * n
    if op == "nvfp4_quantize":
        NV.quantize(x, extra)
        return 2.5625 * n
    if op == "mxfp8_quantize_rn":
        RQ.quantize_rowwise_rn(x)
        return 3.03125 * n
    codes, scales, sg = extra  # dequant_transpose_requant_sr of the slice's NVFP4 form
    RQ.requant_weights(codes[None], scales[None], np.array([sg]), 1, 0)
    return 1.59375 * n


def _oracle_decode_expert(payload):
    """One expert of the decode forward through the oracle: its rows
    quantized to NVFP4, the FP64 w13 GEMM over the dequantized (pre-quantized)
    weights, SwiGLU, NVFP4 of h, the w2 GEMM.  Returns the NVFP4 weight +
    scale bytes it consumed (0.5625 per parameter; the weight matrices here
    are [2 I' x d] and [d x I'] for a slice of I' hidden features)."""
    from oracle import gemm as G
    from oracle import nvfp4 as NV
    from oracle import swiglu as SW
    x, w13q, w2q = payload
    o = np.array([0, x.shape[0]])
    xc, xs, xsg = NV.quantize(x)
    y13, _ = G.grouped_rows(NV.dequantize_f64(xc, xs, xsg), NV.dequantize_f64(*w13q)[None], o)
    h = SW.forward(y13.astype(np.float32))
    hc, hs, hsg = NV.quantize(h.astype(np.float32))
    G.grouped_rows(NV.dequantize_f64(hc, hs, hsg), NV.dequantize_f64(*w2q)[None], o)
    return 0.5625 * (w13q[0].size + w2q[0].size)


_ORACLE_TASKS = {"single_linear": _oracle_single_linear, "quant_op": _oracle_quant_op,
                 "decode_expert": _oracle_decode_expert}


def _oracle_worker(task):
    """Runs one oracle task in a worker process and times it there."""
    kind, payload = task
    t0 = time.perf_counter()
    units = _ORACLE_TASKS[kind](payload)
    return units, time.perf_counter() - t0


class OraclePools:
    """Two pools of spawned worker processes (never forked from a process
    that has used the GPU), one BLAS thread each: one worker for the
    single-thread timings and one per host core for the all-core ones."""

    KEYS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS")

    def __init__(self, cores):
        import multiprocessing as mp
        self.cores = cores
        saved = {k: os.environ.get(k) for k in self.KEYS}
        for k in self.KEYS:
            os.environ[k] = "1"
        try:
            ctx = mp.get_context("spawn")
            self.one = ctx.Pool(1)
            self.all = ctx.Pool(cores)
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        warm = [("quant_op", ("nvfp4_amax", np.zeros((1, 16), np.float32), None))]
        self.one.map(_oracle_worker, warm)
        self.all.map(_oracle_worker, warm * cores, chunksize=1)

    def time(self, tasks_single, tasks_all):
        """Units per second: the single-thread tasks one after another in one
        worker (their own run time), and the all-core tasks at once (wall)."""
        res = self.one.map(_oracle_worker, tasks_single, chunksize=1)
        single = sum(u for u, _ in res) / sum(t for _, t in res)
        t0 = time.perf_counter()
        res = self.all.map(_oracle_worker, tasks_all, chunksize=1)
        allc = sum(u for u, _ in res) / (time.perf_counter() - t0)
        return single, allc

    def close(self):
        for p in (self.one, self.all):
            p.close()
            p.join()


def _bf16_numpy(t):
    import torch
    return t.detach().to("cpu", torch.float32).numpy()


def oracle_single_linear(pools):
    from precision_moe_numerics_nvfp4_gb300 import workloads as W
    s = W.single_linear("cpu")
    payload = (_bf16_numpy(s.x), _bf16_numpy(s.w), _bf16_numpy(s.g))
    single, allc = pools.time([("single_linear", payload)] * 2, [("single_linear", payload)] * pools.cores)
    fl = 3 * 2.0 * 256 * 512 * 1024
    return {"kind": "oracle", "cores": pools.cores, "unit": "us per fwd+bwd",
            "sample": "the whole layer (seed 0), every step; all cores: one layer per core at once",
            "single_thread": {"value": fl / single * 1e6, "threads": 1},
            "all_cores": {"value": fl / allc * 1e6, "threads": pools.cores}}


def oracle_quant_sweep(shapes, pools, rows_per_task=32):
    """Per (shape, op): GB/s of algorithmic bytes on `rows_per_task` rows per
    task (one task single-threaded, one per core at once)."""
    from oracle import nvfp4 as NV
    from precision_moe_numerics_nvfp4_gb300 import workloads as W
    cores = pools.cores
    out = []
    for shape in shapes:
        x = W.quant_sweep(shape, "cpu")
        R, C = shape
        slices = [_bf16_numpy(x[(i * rows_per_task) % R:(i * rows_per_task) % R + rows_per_task])
                  for i in range(cores)]
        del x
        sg = [NV.outer_scale(v) for v in slices]
        nvf = []
        for v, g in zip(slices, sg):
            c, sc, _ = NV.quantize(v, g)
            nvf.append((c, sc, g))
        for op in ("nvfp4_amax", "nvfp4_quantize", "mxfp8_quantize_rn", "dequant_transpose_requant_sr"):
            extra = {"nvfp4_amax": [None] * cores, "nvfp4_quantize": sg,
                     "mxfp8_quantize_rn": [None] * cores, "dequant_transpose_requant_sr": nvf}[op]
            tasks = [("quant_op", (op, v, e)) for v, e in zip(slices, extra)]
            single, allc = pools.time(tasks[:1], tasks)
            out.append({"shape": [R, C], "op": op, "single_thread_GB_s": single / 1e9,
                        "all_cores_GB_s": allc / 1e9})
    return {"kind": "oracle", "cores": cores, "unit": "GB/s (algorithmic bytes)",
            "sample": f"{rows_per_task} rows of each tensor per task (full width); all cores: one task per core, "
                      f"different rows", "ops": out}


def oracle_decode(sample, pools):
    """`sample`: expert 0's weights restricted to the first 256 hidden
    features (bf16, from the GPU run) and the routed rows of the first
    experts; the weights are quantized once here (untimed, as on the GPU)."""
    from oracle import nvfp4 as NV
    w13, w2, rows = sample
    w13q, w2q = NV.quantize(w13), NV.quantize(w2)
    tasks = [("decode_expert", (r, w13q, w2q)) for r in rows[:pools.cores]]
    single, allc = pools.time(tasks[:1], tasks)
    return {"kind": "oracle", "cores": pools.cores, "unit": "GB/s of NVFP4 weight + scale bytes",
            "sample": "expert 0's gate/up/down restricted to 256 of the 2048 hidden features, pre-quantized; one "
                      "task per expert's routed rows; all cores: one task per core at once",
            "single_thread": {"value": single / 1e9, "threads": 1},
            "all_cores": {"value": allc / 1e9, "threads": pools.cores}}


# ---------------------------------------------------------------------------
# the other workloads on the GPU, measured in the default run beside the
# MoE step: the single linear layer, the quantization sweep, the decode
# ---------------------------------------------------------------------------
class L2Flush:
    """Writes a buffer larger than the L2 cache (512 MiB) so that the next
    call reads its inputs from HBM."""

    def __init__(self):
        import torch
        self.buf = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")

    def __call__(self):
        self.buf.zero_()


def time_calls(fn, iters, flush=None):
    """Mean device ms of fn() over `iters` calls, CUDA events on the current
    stream around each call (the flush, when given, runs between calls,
    outside the events)."""
    import torch
    s = torch.cuda.current_stream()
    evs = []
    for _ in range(iters):
        if flush is not None:
            flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        fn()
        e1.record(s)
        evs.append((e0, e1))
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in evs) / iters


def gpu_single_linear(iters=50):
    """Config: one expert linear layer x [256 x 512], w [1024 x 512], g [256 x
    1024] (seed 0), forward and backward through the library; microseconds
    per fwd+bwd, eager and replayed as one CUDA graph."""
    import torch
    from precision_moe_numerics_nvfp4_gb300 import workloads as W
    from precision_moe_numerics_nvfp4_gb300.pipeline import MoELayer, SingleLinear
    s = W.single_linear("cuda")
    layer = SingleLinear(256, 512, 1024)
    fn = lambda: layer.enqueue(s.x, s.w, s.g, seed=0)
    for _ in range(3):
        fn()
    eager = time_calls(fn, iters)
    graph = MoELayer.capture(fn)
    for _ in range(3):
        graph.replay()
    replay = time_calls(graph.replay, iters)
    return {"workload": "single expert linear, x [256 x 512] (4 rows x64), w [1024 x 512] (8 elements x100), "
                        "g [256 x 1024], seed 0: NVFP4 quantization of x and w with their SR requant in the same "
                        "pass, NVFP4 fwd GEMM, SR MXFP8 of g (row-wise + transposed), dgrad + wgrad",
            "us_per_fwd_bwd": eager * 1e3, "us_per_fwd_bwd_graph": replay * 1e3, "calls": 6, "launches": 10,
            "gemm_flops": 3 * 2.0 * 256 * 512 * 1024, "roofline": "latency-bound (no roofline bar)"}


def gpu_quant_sweep(peaks, iters=20):
    """Config: the quantization-only sweep, bf16 [8192 x 8192] and [16384 x
    7168], Student-t(3) x 0.05 with 0.01% x1000 (seed 1).  Per op: the amax
    pass alone (nvfp4_outer_scale, 2 B/elem), the NVFP4 quantization with the
    outer scale given (2.5625 B/elem), both in one call (4.5625), MXFP8 RN
    row-wise (3.03125) and dequant -> transpose -> SR requant of the NVFP4
    result (1.59375).  L2 is flushed before every timed call."""
    import torch
    from precision_moe_numerics_nvfp4_gb300 import nvfp4moe as N
    from precision_moe_numerics_nvfp4_gb300 import workloads as W
    from precision_moe_numerics_nvfp4_gb300.pipeline import MxRows, MxTransposed, NvTensor
    flush = L2Flush()
    out = []
    for R, C in W.QUANT_SWEEP_SHAPES:
        x = W.quant_sweep((R, C), "cuda")
        nv = NvTensor(1, R, C, torch.device("cuda"))
        mr = MxRows(R, C, torch.device("cuda"))
        mt = MxTransposed(R, C, torch.device("cuda"), batch=1)
        sg = torch.empty(1, dtype=torch.float32, device="cuda")
        nv.quantize(x)
        torch.cuda.synchronize()
        ops = {
            "nvfp4_amax": (lambda: N.nvfp4_outer_scale(x, 1, R * C, sg, nv.ws), 2.0),
            "nvfp4_quantize_given_scale": (lambda: nv.quantize(x, sg_in=nv.sg), 2.5625),
            "nvfp4_quantize": (lambda: nv.quantize(x), 4.5625),
            "mxfp8_quantize_rn": (lambda: N.mxfp8_quantize(x, R, C, None, N.NV_RN, 0, 0, 0, mr.codes, mr.scales,
                                                           None, None), 3.03125),
            "dequant_transpose_requant_sr": (lambda: N.dequant_transpose_requant_sr(
                nv.codes, nv.scales, nv.sg, 1, R, C, None, 1, 0, mt.codes, mt.scales), 1.59375),
        }
        for name, (fn, bpe) in ops.items():
            for _ in range(3):
                fn()
            ms = time_calls(fn, iters, flush)
            gbs = R * C * bpe / (ms / 1e3) / 1e9
            out.append({"shape": [R, C], "op": name, "ms": ms, "GB_s": gbs, "frac_hbm": gbs / peaks["hbm_gbs"],
                        "bytes_per_elem": bpe})
        assert N.nvfp4moe_get_device_status() == 0
        del x, nv, mr, mt
    del flush
    torch.cuda.empty_cache()
    return {"workload": "quantization sweep: bf16 [8192 x 8192] and [16384 x 7168], Student-t(3) x 0.05 with 0.01% "
                        "of elements x1000, seed 1", "l2": "flushed (512 MiB write) before every timed call",
            "peak": peaks["hbm_gbs"], "ops": out}


def gpu_decode(peaks, iters=50):
    """Config: the sampler-style decode forward (128 experts [7168 x 2048]
    gate/up/down pre-quantized, 256 tokens top-8), replayed as one CUDA
    graph; GB/s of the NVFP4 weight + scale bytes (0.5625 B per parameter)."""
    import torch
    from precision_moe_numerics_nvfp4_gb300 import nvfp4moe as N
    from precision_moe_numerics_nvfp4_gb300 import workloads as W
    from precision_moe_numerics_nvfp4_gb300.pipeline import MoELayer
    m = W.decode("cuda")
    M, D, I, E = m.x_perm.shape[0], 7168, 2048, 128
    layer = MoELayer(M, D, I, E, backward=False)
    layer.quantize_weights(m.w13, m.w2)
    wbytes = E * (2 * I * D + D * I) * 0.5625
    graph = MoELayer.capture(lambda: layer.forward_activations(m.x_perm, m.group_offsets))
    for _ in range(3):
        graph.replay()
    ms = time_calls(graph.replay, iters)
    assert N.nvfp4moe_get_device_status() == 0
    sizes = torch.diff(m.group_offsets.to(torch.int64))
    gbs = wbytes / (ms / 1e3) / 1e9
    go = m.group_offsets.to("cpu", torch.int64)
    # the oracle's sample: expert 0 restricted to 256 hidden features, and
    # the routed rows of the first experts
    sample = (_bf16_numpy(torch.cat([m.w13[0, :256], m.w13[0, I:I + 256]])), _bf16_numpy(m.w2[0][:, :256]),
              [_bf16_numpy(m.x_perm[int(go[e]):int(go[e + 1])]) for e in range(min(E, 64))])
    del layer, m, graph
    torch.cuda.empty_cache()
    return sample, {"workload": "decode: 128 experts, gate/up/down [7168 x 2048] NVFP4 (pre-quantized), 256 tokens top-8, "
                        f"{int(sizes.min())}..{int(sizes.max())} rows per expert, seed 4",
            "ms": ms, "GB_s": gbs, "frac_hbm": gbs / peaks["hbm_gbs"], "weight_bytes": wbytes, "graph": True,
            "l2": "weights (3.2 GB) exceed L2"}


def other_configs(peaks, with_oracle):
    """The single linear layer, the quantization sweep and the decode, each
    with the oracle beside it (rank 0 only)."""
    sample, dec = gpu_decode(peaks)
    cfg = {"single_linear": gpu_single_linear(), "quant_sweep": gpu_quant_sweep(peaks), "decode": dec}
    if with_oracle:
        from precision_moe_numerics_nvfp4_gb300 import workloads as W
        pools = OraclePools(os.cpu_count() or 1)
        try:
            cfg["single_linear"]["oracle"] = oracle_single_linear(pools)
            cfg["quant_sweep"]["oracle"] = oracle_quant_sweep(W.QUANT_SWEEP_SHAPES, pools)
            cfg["decode"]["oracle"] = oracle_decode(sample, pools)
        finally:
            pools.close()
    return cfg


def run_reference(args):
    rank, world = init_dist("gloo")
    if rank != 0:
        return
    for _ in range(args.warmup):
        oracle_sample_step(args.ref_tokens, d_ff=args.ref_dff)
    t0 = time.perf_counter()
    flops = 0.0
    for _ in range(args.steps):
        flops += oracle_sample_step(args.ref_tokens, d_ff=args.ref_dff)
    dt = time.perf_counter() - t0
    v = flops / dt / 1e12
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 oracle",
        "data": "synthetic", "config": {"workload": WORKLOAD, "sample_rows_per_step": args.ref_tokens,
                                        "sample_d_ff": args.ref_dff},
        "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": f"one expert, {args.ref_tokens} rows and a {args.ref_dff}-wide slice of "
                                   f"d_ff per step, full d_model, every step of the path"},
        "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def run_quant_sweep(args):
    """The quantization-only workload: bf16 [8192 x 8192] and [16384 x 7168],
    Student-t(3) x 0.05 with 0.01% of elements x1000.  Ops: NVFP4 1x16 RN
    quantize (with its amax pass), MXFP8 1x32 RN quantize along rows, and
    dequant -> transpose -> SR requant of the NVFP4 result.  One JSON line per
    (shape, op) with achieved GB/s of algorithmic bytes."""
    import torch
    from precision_moe_numerics_nvfp4_gb300 import nvfp4moe as N
    from precision_moe_numerics_nvfp4_gb300 import workloads as W
    from precision_moe_numerics_nvfp4_gb300.pipeline import MxRows, MxTransposed, NvTensor

    N.lib()
    peaks = load_peaks()
    shapes = W.QUANT_SWEEP_SHAPES if args.sweep_shape is None else [tuple(int(v) for v in args.sweep_shape.split("x"))]
    for shape in shapes:
        R, C = shape
        x = W.quant_sweep(shape, "cuda")
        nv = NvTensor(1, R, C, torch.device("cuda"))
        mr = MxRows(R, C, torch.device("cuda"))
        mt = MxTransposed(R, C, torch.device("cuda"), batch=1)
        mt2 = MxTransposed(R, C, torch.device("cuda"), E=1)
        ops = {
            "nvfp4_quantize": (lambda: nv.quantize(x), 4.5625),
            "mxfp8_quantize_rn": (lambda: N.mxfp8_quantize(x, R, C, None, N.NV_RN, 0, 0, 0, mr.codes, mr.scales,
                                                           None, None), 3.03125),
            "dequant_transpose_requant_sr": (lambda: N.dequant_transpose_requant_sr(
                nv.codes, nv.scales, nv.sg, 1, R, C, None, 1, 0, mt.codes, mt.scales), 1.59375),
            # not ops of the sweep: NVFP4 quantize + requant in one pass, and the gradient's SR
            # quantization (row-wise + transposed), on the same tensor
            "nvfp4_quantize_requant": (lambda: N.nvfp4_quantize_requant(
                x, 1, R, C, None, None, nv.sg, nv.codes, nv.scales, nv.ws, 1, 0, mt.codes, mt.scales), 5.59375),
            "mxfp8_quantize_sr_dual": (lambda: N.mxfp8_quantize(x, R, C, None, N.NV_SR, 0, 0, 1, mr.codes, mr.scales,
                                                                mt2.codes, mt2.scales), 4.0625),
        }
        nv.quantize(x)
        torch.cuda.synchronize()
        for name, (fn, bpe) in ops.items():
            if args.sweep_op and args.sweep_op != name:
                continue
            for _ in range(args.warmup):
                fn()
            torch.cuda.synchronize()
            s = torch.cuda.current_stream()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            for _ in range(args.steps):
                fn()
            e1.record(s)
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / args.steps
            gbs = R * C * bpe / (ms / 1e3) / 1e9
            print(json.dumps({"workload": "quant_sweep", "shape": [R, C], "op": name, "ms": ms, "GB_s": gbs,
                              "frac_hbm": gbs / peaks["hbm_gbs"], "bytes_per_elem": bpe,
                              "peak_source": peaks["source"]}))
        assert N.nvfp4moe_get_device_status() == 0
        del x, nv, mr, mt, mt2
        torch.cuda.empty_cache()


def run_gemm(args):
    """One grouped GEMM of the MoE layer at a reduced token count, optionally
    over fewer experts (same depth per expert, smaller footprint; for
    profiling): fwd = x_q w13^T (N 3072, K 4096), swiglu = the same GEMM with
    SwiGLU and max |h| in its epilogue (y13 and h written), dx = dy13 w13
    (N 3072, K 4096), dx_swiglu = the w2 dgrad g2 w2 (N 4096, K 1536) with
    the SwiGLU backward in its epilogue (y13 read, dy13 written), dw = dy13^T
    x_q.  Prints achieved TFLOP/s (of the GEMM's FLOPs)."""
    import torch
    from precision_moe_numerics_nvfp4_gb300 import nvfp4moe as N
    from precision_moe_numerics_nvfp4_gb300 import workloads as W
    from precision_moe_numerics_nvfp4_gb300.pipeline import MxRows, MxTransposed, NvTensor

    N.lib()
    dev = torch.device("cuda")
    m = W.moe("cuda", seed=2, tokens=args.gemm_tokens, experts=args.gemm_experts, bias_std=args.gemm_bias_std)
    M, d, I2, E = m.x_perm.shape[0], SHAPE["d_model"], 2 * SHAPE["d_ff"], args.gemm_experts
    go = m.group_offsets
    sizes = torch.diff(go.to(torch.int64))
    flops = float(2 * M * I2 * d)
    xq, wq = NvTensor(1, M, d, dev, E=E), NvTensor(E, I2, d, dev)
    xq.quantize(m.x_perm, go)
    wq.quantize(m.w13)
    if args.gemm_kind == "fwd":
        y = torch.empty((M, I2), dtype=torch.bfloat16, device=dev)
        fn = lambda: N.grouped_gemm_nvfp4_fwd(None, xq.sg, xq.codes, xq.scales, wq.codes, wq.scales, wq.sg, go, E, M,
                                              I2, d, y, N.NV_OUT_BF16)
    elif args.gemm_kind == "swiglu":
        y13 = torch.empty((M, I2), dtype=torch.bfloat16, device=dev)
        h = torch.empty((M, I2 // 2), dtype=torch.bfloat16, device=dev)
        h_sg = torch.empty(1, dtype=torch.float32, device=dev)
        fn = lambda: N.grouped_gemm_nvfp4_fwd_swiglu(xq.sg, xq.codes, xq.scales, wq.codes, wq.scales, wq.sg, go, E, M,
                                                     I2 // 2, d, y13, h, h_sg)
    elif args.gemm_kind == "dx_swiglu":
        I = I2 // 2
        flops = float(2 * M * d * I)
        g2 = (torch.randn((M, d), device=dev) * 1e-3).to(torch.bfloat16)
        gr2, gt2 = MxRows(M, d, dev, E=E), MxTransposed(M, d, dev, E=E)
        N.mxfp8_quantize(g2, M, d, go, N.NV_SR, 3, 6, 7, gr2.codes, gr2.scales, gt2.codes, gt2.scales)
        w2 = (torch.randn((E, d, I), device=dev) * 0.02).to(torch.bfloat16)
        w2q = NvTensor(E, d, I, dev)
        w2q.quantize(w2)
        w2t = MxTransposed(d, I, dev, batch=E)
        N.dequant_transpose_requant_sr(w2q.codes, w2q.scales, w2q.sg, E, d, I, None, 3, 1, w2t.codes, w2t.scales)
        y13 = torch.randn((M, I2), device=dev).to(torch.bfloat16)
        dy13 = torch.empty((M, I2), dtype=torch.bfloat16, device=dev)
        fn = lambda: N.grouped_gemm_mxfp8_dx_swiglu_bwd(gr2.codes, gr2.scales, w2t.codes, w2t.scales, go, E, M, d, I,
                                                        y13, dy13)
    else:
        g = (torch.randn((M, I2), device=dev) * 1e-3).to(torch.bfloat16)
        gr, gt = MxRows(M, I2, dev, E=E), MxTransposed(M, I2, dev, E=E)
        N.mxfp8_quantize(g, M, I2, go, N.NV_SR, 3, 6, 7, gr.codes, gr.scales, gt.codes, gt.scales)
        if args.gemm_kind == "dx":
            wt = MxTransposed(I2, d, dev, batch=E)
            N.dequant_transpose_requant_sr(wq.codes, wq.scales, wq.sg, E, I2, d, None, 3, 0, wt.codes, wt.scales)
            dx = torch.empty((M, d), dtype=torch.bfloat16, device=dev)
            fn = lambda: N.grouped_gemm_mxfp8_dx(gr.codes, gr.scales, wt.codes, wt.scales, go, E, M, I2, d, dx,
                                                 N.NV_OUT_BF16)
        else:
            xt = MxTransposed(M, d, dev, E=E)
            N.dequant_transpose_requant_sr(xq.codes, xq.scales, xq.sg, 1, M, d, go, 3, 2, xt.codes, xt.scales)
            dw = torch.empty((E, I2, d), dtype=torch.float32, device=dev)
            fn = lambda: N.grouped_gemm_mxfp8_dw(gt.codes, gt.scales, xt.codes, xt.scales, go, E, M, I2, d, dw)
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(args.steps):
        fn()
    e1.record(s)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    assert N.nvfp4moe_get_device_status() == 0
    print(json.dumps({"workload": "gemm", "kind": args.gemm_kind, "rows": M, "experts": E,
                      "min_group": int(sizes.min()), "max_group": int(sizes.max()), "ms": ms,
                      "TFLOP_s": flops / (ms / 1e3) / 1e12}))


def run_gather(args):
    """The quantization of the MoE layer's activations from its tokens
    (nvfp4_quantize_requant_gather) alone: the tokens [T x d_model] bf16 and
    the routed rows' source tokens in; the routed rows' NVFP4 codes, scales and
    outer scale and their transposed MXFP8 SR re-quantization out.  T =
    --gemm-tokens, top-8 over --gemm-experts experts (the MoE step's routing
    recipe; fewer experts give a smaller case for profiling).  Prints achieved
    GB/s of algorithmic bytes (the amax pass included)."""
    import torch
    from precision_moe_numerics_nvfp4_gb300 import nvfp4moe as N
    from precision_moe_numerics_nvfp4_gb300 import workloads as W
    from precision_moe_numerics_nvfp4_gb300.pipeline import MxTransposed, NvTensor

    N.lib()
    peaks = load_peaks()
    dev = torch.device("cuda")
    E = args.gemm_experts
    m = W.moe("cuda", seed=2, tokens=args.gemm_tokens, experts=E, bias_std=args.gemm_bias_std, weights=False)
    T, d = m.x.shape
    M = m.rows.shape[0]
    q, mx = NvTensor(1, M, d, dev, E=E), MxTransposed(M, d, dev, E=E)
    ws = q.gather_workspace(T)
    fn = lambda: N.nvfp4_quantize_requant_gather(m.x, m.rows, T, M, d, m.group_offsets, None, q.sg, q.codes,
                                                 q.scales, ws, 3, 1, mx.codes, mx.scales)
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    ms = time_calls(fn, args.steps)
    assert N.nvfp4moe_get_device_status() == 0
    bpe = gather_bytes_per_routed_elem(T, M)
    gbs = M * d * bpe / (ms / 1e3) / 1e9
    print(json.dumps({"workload": "gather", "tokens": T, "rows": M, "experts": E, "ms": ms, "GB_s": gbs,
                      "frac_hbm": gbs / peaks["hbm_gbs"], "bytes_per_routed_elem": bpe}))


def run_rht_s2f6(args):
    """RHT-32 + block-scaled S2F6 of the MoE layer's output (the combine
    direction): 131072 routed rows x d_model 4096, bf16, values Student-t(3)
    x 0.05 with 0.01% outliers x1000 (the quantization sweep's recipe at this
    shape), a fixed random sign mask.  Quantize reads 2 and writes 1 + 1/32
    bytes per value; the inverse reads 1 + 1/32 and writes 2 (bf16)."""
    import torch
    from precision_moe_numerics_nvfp4_gb300 import nvfp4moe as N
    from precision_moe_numerics_nvfp4_gb300 import workloads as W

    N.lib()
    peaks = load_peaks()
    rows, cols, mask = 131072, SHAPE["d_model"], 0x9E3779B9
    x = W.quant_sweep((rows, cols), "cuda", seed=6)
    codes = torch.empty((rows, cols), dtype=torch.int8, device="cuda")
    scales = torch.empty((rows, cols // 32), dtype=torch.uint8, device="cuda")
    y = torch.empty((rows, cols), dtype=torch.bfloat16, device="cuda")
    ops = {
        "rht32_s2f6_quantize": lambda: N.rht32_s2f6_quantize(x, rows, cols, mask, codes, scales),
        "s2f6_dequantize_rht32_inverse": lambda: N.s2f6_dequantize_rht32_inverse(codes, scales, rows, cols, mask, y,
                                                                                 N.NV_OUT_BF16),
    }
    for name, fn in ops.items():
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        s = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(args.steps):
            fn()
        e1.record(s)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / args.steps
        gbs = rows * cols * 3.03125 / (ms / 1e3) / 1e9
        print(json.dumps({"workload": "rht_s2f6", "op": name, "shape": [rows, cols], "ms": ms, "GB_s": gbs,
                          "frac_hbm": gbs / peaks["hbm_gbs"], "bytes_per_value": 3.03125,
                          "peak_source": peaks["source"]}))
    assert N.nvfp4moe_get_device_status() == 0

    # the w2 (down-projection) GEMM with the quantizer in its epilogue, against
    # the GEMM followed by the standalone quantizer: h [131072 x 1536] NVFP4,
    # w2 [64 x 4096 x 1536] NVFP4, the benchmark's routing
    from precision_moe_numerics_nvfp4_gb300.pipeline import NvTensor
    m = W.moe("cuda", seed=2, tokens=SHAPE["tokens"], weights=False)
    go = m.group_offsets
    E, Kh = go.numel() - 1, SHAPE["d_ff"]
    del m
    g = torch.Generator(device="cuda").manual_seed(7)
    h = torch.randn((rows, Kh), generator=g, device="cuda").to(torch.bfloat16)
    w2 = (torch.randn((E, cols, Kh), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    hq, wq = NvTensor(1, rows, Kh, torch.device("cuda"), E=E), NvTensor(E, cols, Kh, torch.device("cuda"))
    hq.quantize(h, go)
    wq.quantize(w2)
    del h, w2
    gemm = lambda: N.grouped_gemm_nvfp4_fwd(None, hq.sg, hq.codes, hq.scales, wq.codes, wq.scales, wq.sg, go, E, rows,
                                            cols, Kh, y, N.NV_OUT_BF16)
    fused = lambda yy: N.grouped_gemm_nvfp4_fwd_rht_s2f6(hq.sg, hq.codes, hq.scales, wq.codes, wq.scales, wq.sg, go,
                                                         E, rows, cols, Kh, mask, yy, codes, scales)
    ops2 = {
        "w2_gemm_bf16": gemm,
        "w2_gemm_bf16_then_rht32_s2f6_quantize": lambda: (gemm(), ops["rht32_s2f6_quantize"]()),
        "w2_gemm_rht_s2f6_epilogue": lambda: fused(None),
        "w2_gemm_rht_s2f6_epilogue_and_bf16": lambda: fused(y),
    }
    fl = 2.0 * rows * cols * Kh
    for name, fn in ops2.items():
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        s = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(args.steps):
            fn()
        e1.record(s)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / args.steps
        print(json.dumps({"workload": "rht_s2f6", "op": name, "shape": [rows, cols, Kh], "experts": E, "ms": ms,
                          "gemm_TFLOP_s": fl / (ms / 1e3) / 1e12}))
    assert N.nvfp4moe_get_device_status() == 0


def run_decode(args):
    """Sampler-style decode forward: 128 experts, SwiGLU gate/up [7168 -> 2048
    x2] and down [2048 -> 7168] quantized to NVFP4 beforehand (untimed), 256
    tokens routed top-8 (~16 rows per expert).  Timed: NVFP4 quantization of
    the activations, both grouped NVFP4 GEMMs and SwiGLU.  Reported as HBM
    GB/s of the NVFP4 weight + scale bytes (0.5625 B per parameter)."""
    import torch
    from precision_moe_numerics_nvfp4_gb300 import nvfp4moe as N
    from precision_moe_numerics_nvfp4_gb300 import workloads as W
    from precision_moe_numerics_nvfp4_gb300.pipeline import MoELayer

    N.lib()
    peaks = load_peaks()
    E = args.decode_experts  # fewer experts (same per-expert shapes, ~16 rows each) for profiling
    m = W.decode("cuda", tokens=256 * E // 128, experts=E)
    M, D, I = m.x_perm.shape[0], 7168, 2048
    layer = MoELayer(M, D, I, E, backward=False)
    layer.quantize_weights(m.w13, m.w2)
    params = E * (2 * I * D + D * I)
    wbytes = params * 0.5625
    fwd = lambda: layer.forward_activations(m.x_perm, m.group_offsets)
    if args.graph:  # the whole forward as one CUDA graph: no launch gaps between its kernels
        graph = MoELayer.capture(fwd)
        fwd = graph.replay
    for _ in range(args.warmup):
        fwd()
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(args.steps):
        fwd()
    e1.record(s)
    torch.cuda.synchronize()
    assert N.nvfp4moe_get_device_status() == 0
    ms = e0.elapsed_time(e1) / args.steps
    gbs = wbytes / (ms / 1e3) / 1e9
    sizes = torch.diff(m.group_offsets.to(torch.int64))
    print(json.dumps({"workload": "decode", "graph": bool(args.graph), "experts": E, "rows": M,
                      "min_group": int(sizes.min()),
                      "max_group": int(sizes.max()), "weight_bytes": wbytes, "ms": ms, "GB_s": gbs,
                      "frac_hbm": gbs / peaks["hbm_gbs"], "peak_source": peaks["source"]}))


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-tokens", type=int, default=256)
    ap.add_argument("--ref-tokens", type=int, default=64)
    ap.add_argument("--ref-dff", type=int, default=256)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="moe workload: skip the single-layer, quantization-sweep and decode records")
    ap.add_argument("--clocks-csv", default=None, help="also write the nvidia-smi clock samples of the timed region here")
    ap.add_argument("--workload", choices=["moe", "quant_sweep", "gemm", "gather", "decode", "rht_s2f6"],
                    default="moe")
    ap.add_argument("--gemm-kind", choices=["fwd", "swiglu", "dx", "dx_swiglu", "dw"], default="fwd")
    ap.add_argument("--graph", action="store_true", help="decode workload: replay the forward as a CUDA graph")
    ap.add_argument("--decode-experts", type=int, default=128,
                    help="decode workload: experts (tokens scale with them, ~16 rows per expert); for profiling")
    ap.add_argument("--four-over-six", action="store_true",
                    help="moe workload: the Four Over Six block rule for the activations x and h")
    ap.add_argument("--per-token", action="store_true",
                    help="moe workload: one outer scale per token for the activations x and h")
    ap.add_argument("--gemm-tokens", type=int, default=16384)
    ap.add_argument("--gemm-experts", type=int, default=SHAPE["experts"])
    ap.add_argument("--gemm-bias-std", type=float, default=1.0)
    ap.add_argument("--sweep-op", default=None)
    ap.add_argument("--sweep-shape", default=None, help="RxC, e.g. 8192x8192")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "quant_sweep":
        run_quant_sweep(args)
    elif args.workload == "gemm":
        run_gemm(args)
    elif args.workload == "gather":
        run_gather(args)
    elif args.workload == "rht_s2f6":
        run_rht_s2f6(args)
    elif args.workload == "decode":
        run_decode(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
