"""Benchmark: one DiT block forward at 1024x1024 picture scale per step, on N GPUs.

Workload: the single block at 1024x1024 (34 text rows + 64x64 image tokens, hidden 3072, 24 heads
x 128, gated-SiLU MLP 8192, batch 1), synthetic seeded inputs.  A step is one mi_block_forward
(every kernel of the block) over that batch.  Each rank runs its own independent block (weak
scaling, no data-path collective); value = image tokens of all ranks / max-over-ranks time.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the float64 CPU oracle (rank 0 only) on a bounded sample of the same
workload and prints the same JSON line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import mi_synth  # noqa: E402

METRIC = "image tokens/s per DiT block fwd (1 GB300); attn+GEMM TFLOP/s as % bf16 peak"
UNIT = "image tokens/s"
WORKLOAD = "block_1024"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# nominal GB300 figures, reported beside the measured ones (which stay the primary denominators)
NOMINAL_PEAKS = {"hbm_gbs": 7900.0, "bf16_tflops": 2250.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def flops_of(g: mi_synth.Geometry):
    """Algorithmic FLOPs of one block forward: GEMMs 2 R (3H^2 + H^2 + 2HI + IH) and attention
    4 S_q S_k,valid d heads per batch element (valid keys only)."""
    H, I, S = g.hidden, g.mlp_inter, g.seq
    gemm = 0
    attn = 0
    for b in range(g.batch):
        gemm += 2 * S * (3 * H * H + H * H + 2 * H * I + I * H)
        sk = g.n_img + g.n_text[b]
        attn += 4 * S * sk * 128 * g.n_heads
    return gemm, attn


def kernel_bytes(g: mi_synth.Geometry):
    """Algorithmic HBM bytes per launch of the element-wise kernels."""
    R, H, I = g.rows, g.hidden, g.mlp_inter
    return {"mod_rmsnorm": 4 * R * H, "qk_norm_rope": 8 * R * H + 512 * R}


# ------------------------------------------------------------------------------ clocks
# Clock-event reason bits of NVML (nvmlClocksEventReason*): the ones a measurement must report.
NVML_REASONS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
                "hw_thermal_slowdown": 0x40, "hw_power_brake_slowdown": 0x80}


def _nvml_index(torch_index: int) -> int:
    """NVML index of the torch device (CUDA_VISIBLE_DEVICES renumbers the devices torch sees)."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    ids = [v.strip() for v in vis.split(",") if v.strip()]
    if ids and torch_index < len(ids) and ids[torch_index].isdigit():
        return int(ids[torch_index])
    return torch_index


class ClockSampler:
    """SM clock, power and clock-event reasons sampled every ~2 ms through NVML (read-only queries)
    on a background thread, so that even a timed region of a few milliseconds holds samples; falls
    back to nvidia-smi at 200 ms when NVML cannot be loaded."""

    SMI_FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                  "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                  "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_s: float = 0.002):
        self.gpu = _nvml_index(gpu_index)
        self.period = period_s
        self.samples = []  # (wall time, sm MHz, max MHz, reason bits, power W)
        self.source = None
        self._stop = None
        self._thread = None
        self._smi = None

    def _nvml(self):
        import ctypes

        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.gpu), ctypes.byref(h)) != 0:
            raise OSError("no NVML handle")
        reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        return lib, h, reasons_fn

    def start(self):
        import ctypes
        import threading

        try:
            lib, h, reasons_fn = self._nvml()
        except (OSError, AttributeError):
            self._start_smi()
            return
        self.source = "nvml"
        self._stop = threading.Event()
        mx = ctypes.c_uint(0)
        lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))  # NVML_CLOCK_SM

        def run():
            clk, rs, pw = ctypes.c_uint(), ctypes.c_ulonglong(), ctypes.c_uint()
            while not self._stop.is_set():
                ok = lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0
                ok = ok and reasons_fn(h, ctypes.byref(rs)) == 0
                lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw))
                if ok:
                    self.samples.append((time.time(), float(clk.value), float(mx.value), int(rs.value),
                                         pw.value * 1e-3))
                time.sleep(self.period)

        self._thread = threading.Thread(target=run, daemon=True)
        self._thread.start()

    def _start_smi(self):
        try:
            fd, self._path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self._fh = open(self._path, "w")
            self._smi = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.SMI_FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "200"], stdout=self._fh,
                                         stderr=subprocess.DEVNULL)
            self.source = "nvidia-smi"
        except (OSError, FileNotFoundError):
            self._smi = None

    def _read_smi(self):
        from datetime import datetime

        self._smi.terminate()
        try:
            self._smi.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self._smi.kill()
        self._fh.close()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self._path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    clk, mxv = float(parts[2]), float(parts[3])
                    pw = float(parts[4])
                except ValueError:
                    continue
                bits = 0
                for n, v in zip(names, parts[6:10]):
                    if v.lower() == "active":
                        bits |= NVML_REASONS[n]
                self.samples.append((ts, clk, mxv, bits, pw))
        os.unlink(self._path)

    def stop(self):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=5)
        elif self._smi is not None:
            self._read_smi()

    def summary(self, t_begin, t_end):
        """Median SM clock, max clock, active reasons over the samples taken in [t_begin, t_end]."""
        sel = [smp for smp in self.samples if t_begin <= smp[0] <= t_end]
        if not sel:
            return None
        bits = 0
        for smp in sel:
            bits |= smp[3]
        return {"sm_mhz": statistics.median(smp[1] for smp in sel), "sm_max_mhz": sel[0][2],
                "reasons": sorted(n for n, b in NVML_REASONS.items() if bits & b), "samples": len(sel),
                "power_w_median": statistics.median(smp[4] for smp in sel), "source": self.source,
                "window_ms": 1e3 * (t_end - t_begin)}


# ------------------------------------------------------------------------------ host logic
def aggregate(ms_per_step_ranks, tokens_per_step_per_rank):
    """Whole-job throughput: every rank's image tokens over the slowest rank's step time."""
    worst = max(ms_per_step_ranks)
    total_tokens = tokens_per_step_per_rank * len(ms_per_step_ranks)
    return total_tokens / (worst * 1e-3), worst


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ------------------------------------------------------------------------------ CPU oracle legs
def oracle_sample_rate(g, inp, n_rows, repeats=1):
    """Image tokens/s of the float64 oracle on `n_rows` query rows of the block (keys and values
    still projected from every row)."""
    from oracle import mi_oracle as O

    w = inp.weights
    args = (O.widen(inp.x[:1]), O.widen(inp.mod[:1]), O.widen(w.w_qkv), O.widen(w.w_o), O.widen(w.w_gu),
            O.widen(w.w_d), O.widen(w.q_norm_w), O.widen(w.k_norm_w), inp.rope_cos.astype(np.float64),
            inp.rope_sin.astype(np.float64))
    rows = np.linspace(g.text_pad, g.seq - 1, n_rows).astype(np.int64)
    times = []
    for _ in range(repeats):
        t0 = time.perf_counter()
        O.block_forward_rows(*args, rows, inp.key_mask[:1], g.n_heads, g.eps)
        times.append(time.perf_counter() - t0)
    return n_rows, times


def cpu_baseline(g, inp):
    """The oracle as it stands on one block forward of every image-token row, on the host cores."""
    n, times = oracle_sample_rate(g, inp, g.n_img, 1)
    return {"value": n / times[0], "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"one {g.name} block forward for all {n} image-token rows (keys/values from all "
                      f"{g.seq} rows), float64 NumPy, {times[0]:.1f} s"}


def oracle_baselines():
    """The oracle on the host cores at the other configurations (bounded samples, ~30 s in all):
    the tiny block and the 1200x880 block whole (every image-token row), the long-sequence block on
    512 sampled image-token query rows (keys and values from all 16418 rows), and one of the 24
    blocks of the guided step at 1024x1024 (batch 2, both branches, with the embedding and the
    velocity head), whose time times 24 is reported as the step's, labelled extrapolated."""
    from oracle import mi_oracle as O

    out = {"cores": os.cpu_count(), "kind": "oracle"}
    for name in ("tiny_8x8", "block_1200x880"):
        g = mi_synth.GEOMETRIES[name]
        inp = mi_synth.block_inputs(g, 0)
        n, times = oracle_sample_rate(g, inp, g.n_img, 1)
        out[name] = {"value": n / times[0], "unit": UNIT, "seconds": times[0],
                     "sample": f"one block forward, all {n} image-token rows"}
    g = mi_synth.GEOMETRIES["block_2048"]
    inp = mi_synth.block_inputs(g, 0)
    n, times = oracle_sample_rate(g, inp, 512, 1)
    out["block_2048"] = {"value": n / times[0], "unit": UNIT, "seconds": times[0],
                         "sample": f"{n} of {g.n_img} image-token query rows (keys/values from all {g.seq} rows)"}
    del inp
    base = mi_synth.GEOMETRIES["step_1024_cfg"]
    g1 = mi_synth.Geometry("step_1024_cfg_1block", base.batch, base.text_pad, base.n_text, base.grid_h,
                           base.grid_w, base.hidden, base.n_heads, base.mlp_inter, n_blocks=1)
    si = mi_synth.step_inputs(g1, 0)
    a = O.step_inputs_widened(si)
    t0 = time.perf_counter()
    O.denoise_step(**a, dt=-0.02, guidance=3.0)
    t1 = time.perf_counter() - t0
    out["step_1024_cfg"] = {"seconds_one_block": t1, "seconds_step_extrapolated": base.n_blocks * t1,
                            "unit": "s per guided step",
                            "sample": f"one of {base.n_blocks} blocks of the guided step (batch 2, both branches, "
                                      "embedding and velocity head), times the block count (extrapolated)"}
    return out


def run_reference(args):
    """The float64 oracle on the host cores, on the same workload, metric and unit.

    Each step is one block forward: the block output of every image-token query row (keys and
    values projected from every row, as attention needs them), about 6 s at 1024x1024 on 16 host
    cores; above 8192 image tokens, a sample of 512 query rows.  The number of timed steps is
    capped so the whole run stays within about two minutes."""
    world, rank, _ = dist_setup()
    if rank != 0:
        return 0
    g = mi_synth.GEOMETRIES[args.workload]
    inp = mi_synth.block_inputs(g, 0)
    rows = g.n_img if g.n_img <= 8192 else 512
    _, t_cal = oracle_sample_rate(g, inp, rows, 1)  # first warm-up step, also the calibration
    for _ in range(min(args.warmup, 2) - 1):
        oracle_sample_rate(g, inp, rows, 1)
    steps = max(1, min(args.steps, int(120.0 / max(t_cal[0], 1e-3))))
    _, times = oracle_sample_rate(g, inp, rows, steps)
    total = sum(times)
    value = rows * steps / total
    sample = (f"{rows} of {g.n_img} image-token query rows per step of {g.name} (keys/values projected "
              f"from all {g.seq} rows), float64 NumPy; {steps} of {args.steps} requested steps timed")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": steps, "steps_requested": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_of(g),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def config_of(g):
    return {"workload": g.name, "batch": g.batch, "seq": g.seq, "text_rows": g.text_pad,
            "grid": f"{g.grid_h}x{g.grid_w}", "hidden": g.hidden, "heads": g.n_heads, "head_dim": 128,
            "mlp_inter": g.mlp_inter, "parallelism": "independent block per GPU (replicas)",
            "l2": "no flush: weights 226.5 MB + activations > 129 MB L2 per step"}


# ------------------------------------------------------------------------------ GPU leg
def _traffic_for(kernel: str):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, if the kernel source is
    unchanged since the counters were taken; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    ent = d.get(kernel)
    if not ent or "sources" not in ent:
        return None
    for rel, sha in ent["sources"].items():
        src = os.path.join(ROOT, rel)
        if not os.path.exists(src) or hashlib.sha256(open(src, "rb").read()).hexdigest() != sha:
            return None
    return ent["dram_bytes_per_launch"]


def run_ours(args):
    import torch

    import diffusion_transformer_denoiser_gb300 as mi

    world, rank, local = dist_setup()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    devc = torch.device("cuda", torch.cuda.current_device())
    mi.lib()
    if not mi.device_supported():
        raise SystemExit("mi_block: " + mi.lib().mi_last_error().decode())

    g = mi_synth.GEOMETRIES[args.workload]
    inp = mi_synth.block_inputs(g, seed=rank)

    def t(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(devc)

    w = inp.weights
    blk = mi.Block(t(w.w_qkv), t(w.w_o), t(w.w_gu), t(w.w_d), t(w.q_norm_w), t(w.k_norm_w), g.n_heads, g.eps,
                   fuse_epilogues=True)
    layout = mi.SeqLayout(g.batch, g.text_pad, g.grid_h, g.grid_w)
    x = t(inp.x)
    mod = t(inp.mod)
    cos = torch.from_numpy(inp.rope_cos).to(devc)
    sin = torch.from_numpy(inp.rope_sin).to(devc)
    mask = torch.from_numpy(inp.key_mask).to(devc)
    ws = torch.empty(blk.workspace_size(g.batch, g.seq), dtype=torch.uint8, device=devc)
    stream = torch.cuda.current_stream()

    def step():
        blk.forward(layout, x, x, mod, cos, sin, mask, ws)

    def barrier():
        if world > 1:
            import torch.distributed as dist

            dist.barrier()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if mi.device_error() != 0:
        raise SystemExit("a kernel reported a pipeline timeout during warm-up")

    # ---- timed region: K block forwards back to back.  The clock sampler polls NVML every ~2 ms
    # from before the region to the end of the per-kernel timings; each figure keeps the samples
    # taken inside its own window.
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    time.sleep(0.05)
    barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t_begin = time.time()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    t_end = time.time()
    barrier()
    clocks = sampler.summary(t_begin, t_end)
    ms = e0.elapsed_time(e1) / args.steps
    ms_all = [ms]
    if world > 1:
        import torch.distributed as dist

        tens = torch.tensor([ms], device=devc)
        gathered = [torch.zeros_like(tens) for _ in range(world)]
        dist.all_gather(gathered, tens)
        ms_all = [float(v.item()) for v in gathered]
    value, worst_ms = aggregate(ms_all, g.batch * g.n_img)
    err = mi.device_error()

    # ---- per-kernel times (same kernels through the single-kernel entry points, same shapes)
    kern = kernel_times(mi, torch, g, inp, t, devc, reps=max(20, min(200, args.steps)), sampler=sampler)
    sampler.stop()

    # ---- end to end through the public API with host buffers.  Every step copies its input
    # from pinned host memory and its output back to pinned host memory.  Pipelined (the value
    # reported): two device and two host buffer sets, the host-to-device copy of step i+1 and the
    # device-to-host copy of step i-1 run on their own streams while step i computes; events keep
    # each buffer's copy, forward and copy-back in order.  Serial (reported beside it): copy in,
    # forward, copy out on one stream.
    x_host = torch.from_numpy(np.ascontiguousarray(inp.x).view(np.int16)).view(torch.bfloat16).pin_memory()
    y_host = [torch.empty_like(x_host).pin_memory() for _ in range(2)]
    xin = [torch.empty_like(x) for _ in range(2)]
    yout = [torch.empty_like(x) for _ in range(2)]
    s_in = torch.cuda.Stream()
    s_out = torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_fwd = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_pipelined(n):
        s_in.wait_stream(stream)
        s_out.wait_stream(stream)
        for i in range(n):
            k = i & 1
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_fwd[k])  # forward i-2 has read xin[k]
                xin[k].copy_(x_host, non_blocking=True)
                ev_in[k].record(s_in)
            stream.wait_event(ev_in[k])
            if i >= 2:
                stream.wait_event(ev_out[k])  # yout[k] of step i-2 is back on the host
            blk.forward(layout, xin[k], yout[k], mod, cos, sin, mask, ws, stream=stream)
            ev_fwd[k].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_fwd[k])
                y_host[k].copy_(yout[k], non_blocking=True)
                ev_out[k].record(s_out)
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)

    def e2e_serial(n):
        for _ in range(n):
            xin[0].copy_(x_host, non_blocking=True)
            blk.forward(layout, xin[0], yout[0], mod, cos, sin, mask, ws, stream=stream)
            y_host[0].copy_(yout[0], non_blocking=True)

    e2e_steps = max(3, min(args.steps, 50))
    e2e_ms = {}
    for name, run in (("serial", e2e_serial), ("pipelined", e2e_pipelined)):
        run(2)
        torch.cuda.synchronize()
        barrier()
        e0.record(stream)
        run(e2e_steps)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        e2e_ms[name] = e0.elapsed_time(e1) / e2e_steps
    # the copied-back output is the forward's output
    if not torch.equal(y_host[(e2e_steps - 1) & 1], yout[(e2e_steps - 1) & 1].cpu()):
        raise SystemExit("end-to-end: the output copied to the host differs from the device output")
    serial_ms = e2e_ms["serial"]
    e2e_ms = e2e_ms["pipelined"]
    e2e_all = [e2e_ms]
    if world > 1:
        import torch.distributed as dist

        tens = torch.tensor([e2e_ms], device=devc)
        gathered = [torch.zeros_like(tens) for _ in range(world)]
        dist.all_gather(gathered, tens)
        e2e_all = [float(v.item()) for v in gathered]
    e2e_value, _ = aggregate(e2e_all, g.batch * g.n_img)
    xbytes = x_host.numel() * 2

    if rank == 0:
        peaks, peak_src = load_peaks()
        gemm_f, attn_f = flops_of(g)
        tflops = (gemm_f + attn_f) / (worst_ms * 1e-3) / 1e12
        dom = kern["gemm_gate_up_silu"]
        dom_flops = 2.0 * g.rows * 2 * g.mlp_inter * g.hidden
        achieved = dom_flops / (dom["ms"] * 1e-3) / 1e12
        peak = peaks["bf16_tflops"]
        traffic = _traffic_for("gemm_gate_up_silu")
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": worst_ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic: seeded N(0,1) activations, N(0,0.02) weights, N(0,0.1) modulation",
            "config": config_of(g),
            "attn_gemm_tflops": tflops, "pct_bf16_peak": tflops / peak,
            "pct_bf16_nominal": tflops / NOMINAL_PEAKS["bf16_tflops"],
            "roofline": {"bound": "tensor", "kernel": "gemm_gate_up_silu (tcgen05, fused SiLU gate)",
                         "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                         "peak_source": f"{peak_src} bf16_tflops (burst; kernel timed alone)",
                         "peak_nominal": NOMINAL_PEAKS["bf16_tflops"],
                         "frac_nominal": achieved / NOMINAL_PEAKS["bf16_tflops"],
                         "traffic": traffic},
            "kernels": {k: {"ms": v["ms"], **{kk: vv for kk, vv in v.items() if kk != "ms"}} for k, v in kern.items()},
            "cpu_baseline": None,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": xbytes, "d2h_bytes_per_step": xbytes,
                    "ms_per_step": max(e2e_all),
                    "copies": "pinned host buffers; copies of neighbouring steps overlap the forward on two "
                              "copy streams",
                    "serial_ms_per_step": serial_ms},
            "gpu_launches": args.steps * 7,
            "clocks": clocks,
            "device_error": err,
        }
        if not args.no_extras:
            line["extras"] = extras(mi, torch, devc, stream)
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(g, inp)
            line["cpu_baseline"]["other_configs"] = oracle_baselines()
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def _gpu_step_params(torch, g, seed, devc):
    """Seeded weights of a guided step drawn on the GPU with the synthetic recipe's distributions
    (24 full-size blocks are 5.4 GB; drawing them on the host would dominate the run)."""
    gen = torch.Generator(device=devc)
    gen.manual_seed(seed)
    H, I, C, B = g.hidden, g.mlp_inter, g.latent_ch, g.batch
    bf = torch.bfloat16

    def rn(*shape, std=1.0, mean=0.0):
        return (torch.randn(*shape, generator=gen, device=devc) * std + mean).to(bf)

    blocks = [dict(w_qkv=rn(3 * H, H, std=0.02), w_o=rn(H, H, std=0.02), w_gu=rn(2 * I, H, std=0.02),
                   w_d=rn(H, I, std=0.02), q_norm_w=rn(128, std=0.02, mean=1.0),
                   k_norm_w=rn(128, std=0.02, mean=1.0)) for _ in range(g.n_blocks)]
    return dict(blocks=blocks, mods=rn(g.n_blocks, 1, 6, H, std=0.1).expand(g.n_blocks, B, 6, H).contiguous(),
                w_in=rn(H, C, std=0.02), w_out=rn(C, H, std=0.02),
                mod_final=rn(1, 2, H, std=0.1).expand(B, 2, H).contiguous(), text=rn(B, g.text_pad, H),
                latent=torch.randn(g.n_img, C, generator=gen, device=devc).to(bf).float())


def _time_block(mi, torch, devc, name, reps=20):
    """A block forward of geometry `name` (in place, back to back), timed with CUDA events."""
    g = mi_synth.GEOMETRIES[name]
    inp = mi_synth.block_inputs(g, 0)

    def t(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(devc)

    w = inp.weights
    blk = mi.Block(t(w.w_qkv), t(w.w_o), t(w.w_gu), t(w.w_d), t(w.q_norm_w), t(w.k_norm_w), g.n_heads, g.eps)
    layout = mi.SeqLayout(g.batch, g.text_pad, g.grid_h, g.grid_w)
    x = t(inp.x)
    args = (t(inp.mod), torch.from_numpy(inp.rope_cos).to(devc), torch.from_numpy(inp.rope_sin).to(devc),
            torch.from_numpy(inp.key_mask).to(devc))
    ws = torch.empty(blk.workspace_size(g.batch, g.seq), dtype=torch.uint8, device=devc)
    stream = torch.cuda.current_stream()
    for _ in range(3):
        blk.forward(layout, x, x, *args, ws)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(reps):
        blk.forward(layout, x, x, *args, ws)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    gf, af = flops_of(g)
    return {"ms_per_block": ms, "image_tokens_per_s": g.batch * g.n_img / (ms * 1e-3),
            "tflops": (gf + af) / (ms * 1e-3) / 1e12, "rows": g.rows, "forwards": reps}


def extras(mi, torch, devc, stream):
    """The other workloads, timed with CUDA events: the 1200x880 block (63 + 55x75 rows), the
    long-sequence block (34 + 128x128 rows), one guided denoising step at 1024x1024 (24 blocks,
    batch 2: prompt and padded empty negative) and the 50-step Euler loop of that step (guidance 3,
    t linear in [1, 0]), replayed from a CUDA graph of one step."""
    out = {}
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    peaks, _ = load_peaks()
    for name in ("block_1200x880", "block_2048"):
        out[name] = _time_block(mi, torch, devc, name)
        out[name]["frac_bf16_peak"] = out[name]["tflops"] / peaks["bf16_tflops_sustained"]
        out[name]["peak"] = "bf16_tflops_sustained (a block is a long mixed step)"
        torch.cuda.empty_cache()
    # guided step and 50-step loop
    g = mi_synth.GEOMETRIES["step_1024_cfg"]
    prm = _gpu_step_params(torch, g, 7, devc)
    model = mi.Model(prm["blocks"], prm["w_in"], prm["w_out"], g.n_heads, g.eps)
    layout = mi.SeqLayout(g.batch, g.text_pad, g.grid_h, g.grid_w)
    ws = torch.empty(model.workspace_size(layout), dtype=torch.uint8, device=devc)
    cos, sin = (torch.from_numpy(a).to(devc) for a in mi_synth.rope_tables(g))
    mask = torch.from_numpy(mi_synth.key_mask(g)).to(devc)
    lat = prm["latent"].clone()
    ts = mi_synth.euler_schedule(50)
    dt = float(ts[1] - ts[0])

    def step():
        model.denoise_step(layout, lat, prm["text"], prm["mods"], prm["mod_final"], cos, sin, mask, dt, 3.0, ws)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    reps = 10
    e0.record(stream)
    for _ in range(reps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    # algorithmic work counts valid rows only (the padded negative rows run but are not credited)
    valid = sum(g.n_img + nt for nt in g.n_text)
    gemm_f = sum(2 * (g.n_img + nt) * (4 * g.hidden ** 2 + 3 * g.hidden * g.mlp_inter) for nt in g.n_text) * g.n_blocks
    attn_f = sum(4 * (g.n_img + nt) ** 2 * 128 * g.n_heads for nt in g.n_text) * g.n_blocks
    out["step_1024_cfg"] = {"ms_per_step": ms, "tflops": (gemm_f + attn_f) / (ms * 1e-3) / 1e12,
                            "blocks": g.n_blocks, "batch": g.batch, "valid_rows": valid}
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    lat.copy_(prm["latent"])
    graph.replay()
    torch.cuda.synchronize()
    lat.copy_(prm["latent"])
    gstream = torch.cuda.current_stream()
    e0.record(gstream)
    for _ in range(50):
        graph.replay()
    e1.record(gstream)
    torch.cuda.synchronize()
    out["loop_1024_cfg50"] = {"seconds": e0.elapsed_time(e1) * 1e-3, "steps": 50, "guidance": 3.0,
                              "launch": "one CUDA graph of one step, replayed 50 times",
                              "latent_finite": bool(torch.isfinite(lat).all().item())}
    err = mi.device_error()
    if err:
        out["device_error"] = err
    return out


L2_BYTES = 129e6  # GB300 L2


# replays of each kernel's graph; the per-launch time is taken from the median replay
KERNEL_REPLAYS = 5


def kernel_times(mi, torch, g, inp, t, devc, reps, sampler=None):
    """Device time of each kernel of the block, launched alone at the workload's shapes through the
    single-kernel entry points.  Every kernel cycles through enough separate buffer sets (inputs,
    weights and outputs) that the bytes touched between two uses of one set are at least three
    times the 129 MB L2: each launch reads its operands from HBM, as the first use inside a forward
    would, and pays for the write-back of earlier outputs.  Times are CUDA events around each of a
    few replays of a CUDA graph of those launches: the median replay, divided by the launch count."""
    R, H, I, nh, S, B = g.rows, g.hidden, g.mlp_inter, g.n_heads, g.seq, g.batch
    bf = torch.bfloat16
    w = inp.weights
    x = t(inp.x).view(R, H)
    mod = t(inp.mod)
    w_qkv, w_o, w_gu, w_d = t(w.w_qkv), t(w.w_o), t(w.w_gu), t(w.w_d)
    wq, wk = t(w.q_norm_w), t(w.k_norm_w)
    cos = torch.from_numpy(inp.rope_cos).to(devc)
    sin = torch.from_numpy(inp.rope_sin).to(devc)
    mask = torch.from_numpy(inp.key_mask).to(devc)
    # realistic operands for each kernel: run the chain once
    h = torch.empty(R, H, dtype=bf, device=devc)
    qkv = torch.empty(R, 3 * H, dtype=bf, device=devc)
    qp = torch.empty(B, nh, S, 128, dtype=bf, device=devc)
    kp = torch.empty_like(qp)
    o = torch.empty(R, H, dtype=bf, device=devc)
    x1 = torch.empty(R, H, dtype=bf, device=devc)
    h2 = torch.empty(R, H, dtype=bf, device=devc)
    m = torch.empty(R, I, dtype=bf, device=devc)
    mi.mod_rmsnorm(x, mod, 0, 1, h, B, S, g.eps)
    mi.gemm_qkv_rope(h, w_qkv, wq, wk, cos, sin, qp, kp, qkv, B, S, nh, g.eps)
    # the attention on the schedule the block forward uses (one CTA per SM, split query-tile pairs)
    attn_ws = torch.empty(mi.attention_workspace_size(B, S, nh), dtype=torch.uint8, device=devc)
    mi.attention(qp, kp, qkv, mask, o, B, S, nh, ws=attn_ws)
    mi.gemm_gated_residual(o, w_o, x, mod, 2, x1, S)
    mi.mod_rmsnorm(x1, mod, 3, 4, h2, B, S, g.eps)
    mi.gemm_silu_gate(h2, w_gu, m)
    torch.cuda.synchronize()

    def cl(a):
        return a.clone()

    def em(a):
        return torch.empty_like(a)

    _, attn_f = flops_of(g)
    # name: (buffers of one set, launch on a set, bytes a launch touches, algorithmic work)
    specs = {
        "mod_rmsnorm": (lambda: dict(x=cl(x), h=em(h)),
                        lambda b: mi.mod_rmsnorm(b["x"], mod, 0, 1, b["h"], B, S, g.eps),
                        4 * R * H, {"bytes": 4 * R * H}),
        "gemm_qkv_rope": (lambda: dict(h=cl(h), w=cl(w_qkv), qp=em(qp), kp=em(kp), qkv=em(qkv)),
                          lambda b: mi.gemm_qkv_rope(b["h"], b["w"], wq, wk, cos, sin, b["qp"], b["kp"], b["qkv"],
                                                     B, S, nh, g.eps),
                          2 * R * H + 6 * H * H + 6 * R * H, {"flops": 2.0 * R * 3 * H * H}),
        "attention": (lambda: dict(qp=cl(qp), kp=cl(kp), qkv=cl(qkv), o=em(o)),
                      lambda b: mi.attention(b["qp"], b["kp"], b["qkv"], mask, b["o"], B, S, nh, ws=attn_ws),
                      8 * R * H, {"flops": float(attn_f)}),
        "gemm_out_gated_residual": (lambda: dict(o=cl(o), w=cl(w_o), x=cl(x), y=em(x1)),
                                    lambda b: mi.gemm_gated_residual(b["o"], b["w"], b["x"], mod, 2, b["y"], S),
                                    6 * R * H + 2 * H * H, {"flops": 2.0 * R * H * H}),
        "gemm_gate_up_silu": (lambda: dict(h=cl(h2), w=cl(w_gu), m=em(m)),
                              lambda b: mi.gemm_silu_gate(b["h"], b["w"], b["m"]),
                              2 * R * H + 4 * I * H + 2 * R * I, {"flops": 2.0 * R * 2 * I * H}),
        "gemm_down_gated_residual": (lambda: dict(m=cl(m), w=cl(w_d), x=cl(x1), y=em(x1)),
                                     lambda b: mi.gemm_gated_residual(b["m"], b["w"], b["x"], mod, 5, b["y"], S),
                                     2 * R * I + 2 * H * I + 4 * R * H, {"flops": 2.0 * R * H * I}),
    }
    peaks, _ = load_peaks()
    out = {}
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    for name, (make, call, touched, work) in specs.items():
        n_sets = max(2, int(np.ceil(3 * L2_BYTES / touched)))
        sets = [make() for _ in range(n_sets)]
        rounds = max(1, int(np.ceil(reps / n_sets)))
        for b in sets:  # warm-up
            call(b)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(rounds):
                for b in sets:
                    call(b)
        graph.replay()
        torch.cuda.synchronize()
        gstream = torch.cuda.current_stream()
        t0 = time.time()
        per_replay = []
        for _ in range(KERNEL_REPLAYS):
            e0.record(gstream)
            graph.replay()
            e1.record(gstream)
            torch.cuda.synchronize()
            per_replay.append(e0.elapsed_time(e1))
        t1 = time.time()
        launches = rounds * n_sets
        ms = float(np.median(per_replay)) / launches
        del graph, sets
        ent = {"ms": ms}
        if "bytes" in work:
            gbs = work["bytes"] / (ms * 1e-3) / 1e9
            ent.update(gbs=gbs, frac_hbm_peak=gbs / peaks["hbm_gbs"], frac_hbm_nominal=gbs / NOMINAL_PEAKS["hbm_gbs"])
        else:
            tf = work["flops"] / (ms * 1e-3) / 1e12
            ent.update(tflops=tf, frac_bf16_peak=tf / peaks["bf16_tflops"],
                       frac_bf16_nominal=tf / NOMINAL_PEAKS["bf16_tflops"])
        ent["timing"] = (f"median over {KERNEL_REPLAYS} replays of one CUDA graph of {launches} launches cycling "
                         f"through {n_sets} buffer sets ({n_sets * touched / 1e6:.0f} MB touched per cycle, "
                         f"L2 129 MB), per launch")
        if sampler is not None:
            ck = sampler.summary(t0, t1)
            if ck:
                ent["sm_mhz"] = ck["sm_mhz"]
                ent["clock_reasons"] = ck["reasons"]
        out[name] = ent
    return out


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(mi_synth.GEOMETRIES))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip the long-sequence block and guided-step timings")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
