"""Benchmark of the log-mel front end on GB300.

Default workload: log_mel_from_stft on B=256 clips of F=3000 frames, NF=201
bins, NM=128 mel bands (the batch-of-30-second-clips shape), f32, synthetic
seeded inputs.  One step = one full call of the hot path over the batch.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  ``value`` is whole-job clips/s with inputs
already resident in HBM; ``e2e`` is the same metric through the library's
host-buffer call (lm_log_mel_from_stft_host / lm_mel_spectrogram_host): the
batch starts in page-locked host memory and the result ends there, with both
copies inside the timed region.  ``cpu_baseline`` times the CPU oracle on
the host cores on each workload's whole batch, and ``parity`` compares the
GPU result of the timed steps with that oracle output element by element.
``--impl reference`` times the CPU oracle (the plain double-precision
definition) on the host cores, on a bounded sample of the same workload per
step.

Under torchrun with N > 1 ranks each rank runs its own full batch on its own
GPU (independent replicas, weak scaling; no collective on the data path).
"""
from __future__ import annotations

import argparse
import json
import os
import pathlib
import statistics
import subprocess
import sys
import time

ROOT = pathlib.Path(__file__).resolve().parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))

METRIC = "log-mel clips/sec and achieved HBM GB/s vs GB300 peak (B=256 Whisper STFT)"
L2_BYTES = 129 * 2 ** 20  # GB300 L2
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, nominal


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int, device="cpu") -> float:
    """The largest of every rank's value (the slowest rank's time); the
    identity with one rank.  Needs an initialised process group when world > 1
    (NCCL with a CUDA device in the benchmark, gloo with "cpu" in the tests)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, units_per_rank: int, steps: int, total_ms: float) -> float:
    """Whole-job units per second: every rank processes its own batch each
    step (weak scaling) and the job takes the slowest rank's time."""
    return world * units_per_rank * steps / (total_ms / 1e3)


def _peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        try:
            d = json.loads(p.read_text())
            return float(d["hbm_gbs"]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


def _traffic_record():
    """dram bytes per launch of the main kernel from the committed ncu summary,
    valid only while the kernel source is unchanged since the capture."""
    import hashlib
    rec = ROOT / "profiles" / "traffic.json"
    if not rec.exists():
        return None
    try:
        d = json.loads(rec.read_text())
        csrc = ROOT / "log_mel_spectrogram_gb300" / "csrc"
        digest = hashlib.sha256((csrc / "stft_logmel.cu").read_bytes() + (csrc / "ptx.cuh").read_bytes())
        if digest.hexdigest() != d.get("source_sha256"):
            return None
        return d
    except Exception:
        return None


class ClockSampler:
    """Samples the SM clock, its maximum, the board power and the active
    clock-event reasons of one GPU while the timed regions run.

    NVML (the driver's libnvidia-ml, read-only queries) is polled every 2 ms
    from a thread, so even a region of a few milliseconds gets samples;
    where NVML cannot be loaded, nvidia-smi samples every 200 ms instead.
    Nothing here changes a setting of the GPU."""

    # nvmlClocksEventReasons bits
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}
    SMI_FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                  "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                  "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, pci_bus_id: str | None = None, interval_s: float = 0.002):
        self.gpu = gpu_index
        self.pci = pci_bus_id
        self.interval = interval_s
        self.rows = []
        self.windows = []
        self.source = None
        self.proc = None
        self.thread = None

    def _nvml_open(self):
        import ctypes
        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        h = ctypes.c_void_p()
        ok = False
        if self.pci:
            ok = nv.nvmlDeviceGetHandleByPciBusId_v2(self.pci.encode(), ctypes.byref(h)) == 0
        if not ok and nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.gpu), ctypes.byref(h)) != 0:
            raise RuntimeError("no NVML handle")
        try:
            reasons_fn = nv.nvmlDeviceGetCurrentClocksEventReasons
        except AttributeError:
            reasons_fn = nv.nvmlDeviceGetCurrentClocksThrottleReasons
        return nv, h, reasons_fn

    def _poll(self, nv, h, reasons_fn):
        import ctypes
        sm, mx, mw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop:
            t = time.time()
            if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(sm)) == 0 and \
                    nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                nv.nvmlDeviceGetPowerUsage(h, ctypes.byref(mw))
                reasons_fn(h, ctypes.byref(rs))
                self.rows.append({"t": t, "sm": float(sm.value), "max": float(mx.value),
                                  "power": mw.value / 1000.0,
                                  "reasons": [n for bit, n in self.REASONS.items() if rs.value & bit]})
            time.sleep(self.interval)

    def __enter__(self):
        import threading
        self._stop = False
        try:
            nv, h, reasons_fn = self._nvml_open()
            self.thread = threading.Thread(target=self._poll, args=(nv, h, reasons_fn), daemon=True)
            self.thread.start()
            self.source = "nvml, every 2 ms"
        except Exception:
            try:
                self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.SMI_FIELDS}",
                                              "--format=csv,noheader,nounits", "-lms", "200"],
                                             stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
                self.source = "nvidia-smi, every 200 ms"
            except Exception:
                self.proc = None
        return self

    def __exit__(self, *exc):
        self._stop = True
        if self.thread is not None:
            self.thread.join(timeout=5)
        if self.proc is not None:
            import datetime
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            for line in (out or "").splitlines():
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    names = [n for n, v in (("hw_slowdown", parts[6]), ("hw_thermal_slowdown", parts[7]),
                                            ("sw_thermal_slowdown", parts[8]), ("sw_power_cap", parts[9]))
                             if v.lower() == "active"]
                    self.rows.append({"t": ts, "sm": float(parts[2]), "max": float(parts[3]),
                                      "power": float(parts[4]), "reasons": names})
                except ValueError:
                    continue

    def mark(self, t0: float, t1: float):
        """Wall-clock bounds of a timed region; only samples inside some
        marked region count."""
        self.windows.append((t0, t1))

    def summary(self, windows=None):
        wins = windows if windows is not None else self.windows
        rows = [r for r in self.rows if any(w0 - 0.002 <= r["t"] <= w1 + 0.002 for w0, w1 in wins)]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0,
                    "source": self.source}
        reasons = sorted({n for r in rows for n in r["reasons"]})
        return {"sm_mhz": statistics.median(r["sm"] for r in rows), "sm_max_mhz": max(r["max"] for r in rows),
                "reasons": reasons, "samples": len(rows), "power_w_max": max(r["power"] for r in rows),
                "source": self.source}


def parity_errors(got, ref, tol: float) -> dict:
    """Elementwise comparison of a GPU result with the oracle's: the largest
    absolute error, the largest relative error (over elements with
    |oracle| >= 1e-2: log-mel outputs pass through zero), the relative
    Frobenius error, the largest ratio of an element's error to its allowance
    tol + tol |oracle| (<= 1 inside the gate), and whether every element is
    inside the gate."""
    import numpy as np
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    err = np.abs(g - r)
    big = np.abs(r) >= 1e-2
    allow = tol + tol * np.abs(r)
    return {"vs": "oracle, whole batch", "max_abs": float(err.max()),
            "max_rel": float((err[big] / np.abs(r[big])).max()) if big.any() else 0.0,
            "rel_fro": float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30)),
            "gate": f"|gpu - oracle| <= {tol:g} + {tol:g} |oracle|",
            "max_gate_ratio": float((err / allow).max()),
            "within_gate": bool(np.all(err <= allow))}


def cpu_baseline(stft_host, W_host, target_s: float = 12.0, sample_note: str = "", got=None) -> dict:
    """Times the oracle (as it stands) on the given clips, processed
    repeatedly until about target_s seconds of CPU work are done.  With `got`
    (the GPU result for the same clips) the dict also carries "parity"."""
    import oracle
    oracle.build()
    n_clips = stft_host.shape[0]
    done = 0
    t0 = time.perf_counter()
    while True:
        ref = oracle.log_mel_from_stft(stft_host, W_host)
        done += n_clips
        dt = time.perf_counter() - t0
        if dt >= target_s:
            break
    out = {"value": done / dt, "unit": "clips/s", "cores": oracle.num_threads(), "kind": "oracle",
           "sample": f"{done} clips ({n_clips} distinct clips{sample_note}, repeated) in {dt:.1f} s, dense "
                     "double-precision oracle, OpenMP over clips"}
    if got is not None:
        out["parity"] = parity_errors(got, ref, 1e-4)
    return out


def cpu_baseline_wave(w, x_host, got=None) -> dict:
    """Times the oracle once on the whole waveform batch; with `got` (the GPU
    result) the dict also carries "parity" (f16 output against the oracle
    rounded to f16, at 2e-3)."""
    import oracle
    oracle.build()
    t0 = time.perf_counter()
    ref = oracle.mel_spectrogram(x_host, w.sample_rate, w.n_fft, w.hop_length, w.n_mels, f_min=w.f_min,
                                 f_max=w.f_max, center=w.center, pad_mode=w.pad_mode, power=w.power,
                                 mel_scale=w.mel_scale, norm=w.norm, log_mel=w.log_mel, out_dtype=w.out_dtype)
    dt = time.perf_counter() - t0
    out = {"value": w.B / dt, "unit": "clips/s", "cores": oracle.num_threads(), "kind": "oracle",
           "sample": f"the whole batch ({w.B} clips) once in {dt:.1f} s: explicit padding and frames, O(N^2) "
                     "DFT, dense filterbank, double precision, OpenMP over clips"}
    if got is not None:
        out["parity"] = parity_errors(got, ref, 2e-3 if w.out_dtype == "f16" else 1e-4)
    return out


STFT_JOBS = ("stft_small", "stft_b8", "stft")
WAVE_JOBS = ("wave_whisper", "wave_pcm16")
# The five workloads in the order of the benchmark's configuration list:
# log_mel_from_stft at B=1/F=300/NM=80, B=8/F=3000/NM=80 and B=256/F=3000/NM=128
# (the headline), then the two mel_spectrogram workloads.
CONFIG_ORDER = ("stft_small", "stft_b8", "stft", "wave_whisper", "wave_pcm16")


class StftJob:
    """log_mel_from_stft on one of the three STFT workloads (or --batch B)."""

    def __init__(self, lm, workloads, dev, batch, name="stft"):
        import torch
        w = {"stft": workloads.WHISPER_STFT_B256, "stft_small": workloads.WHISPER_STFT_SMALL,
             "stft_b8": workloads.WHISPER_STFT}[name]
        if batch and batch != w.B:
            import dataclasses
            w = dataclasses.replace(w, B=batch, name=w.name.replace(f"b{w.B}_", f"b{batch}_"))
        self.name = name
        self.lm, self.w, self.dev = lm, w, dev
        self.stft, self.W = workloads.stft_workload_inputs(w, device=dev)
        self.out = torch.empty((w.B, w.F, w.NM), dtype=torch.float32, device=dev)
        self.ws = torch.empty(lm.log_mel_from_stft_workspace_size(w.B, w.F, w.NF, w.NM), dtype=torch.uint8,
                              device=dev)
        self.info = lm.describe_log_mel_from_stft(w.B, w.F, w.NF, w.NM)
        self.units = w.B
        self.bytes = w.canonical_bytes
        self.kernels = self.info["kernels"]
        # The headline batch streams 1.63 GB per step, 12x the L2; smaller
        # batches that could sit in L2 are flushed between steps.
        self.flush_l2 = w.canonical_bytes < 4 * L2_BYTES
        self.inputs = [self.stft, self.W]

    def step(self, inputs=None):
        stft, W = inputs if inputs is not None else (self.stft, self.W)
        self.lm.log_mel_from_stft(stft, W, out=self.out, workspace=self.ws)

    def error(self):
        return self.lm.workspace_error(self.ws)

    def host_setup(self):
        """Host copies of the inputs and a host output, both page-locked, and
        the device workspace of the host-buffer entry point."""
        import torch
        w = self.w
        self.h_stft = torch.empty(self.stft.shape, dtype=self.stft.dtype, pin_memory=True)
        self.h_stft.copy_(self.stft)
        self.h_out = torch.empty(self.out.shape, dtype=self.out.dtype, pin_memory=True)
        self.h_ws = torch.empty(self.lm.log_mel_from_stft_host_workspace_size(w.B, w.F, w.NF, w.NM),
                                dtype=torch.uint8, device=self.dev)
        return self.h_stft.numel() * self.h_stft.element_size(), self.h_out.numel() * self.h_out.element_size()

    def host_step(self):
        self.lm.log_mel_from_stft_host(self.h_stft, self.W, out=self.h_out, workspace=self.h_ws, synchronize=False)

    def host_check(self):
        return self.lm.workspace_error(self.h_ws) == 0 and bool(self.h_out.equal(self.out.cpu()))

    def host_api(self):
        return "log_mel_from_stft_host -> lm_log_mel_from_stft_host (chunked copy-in / kernel / copy-out pipeline)"

    def config(self):
        w, info = self.w, self.info
        return {"workload": w.name, "B": w.B, "F": w.F, "NF": w.NF, "NM": w.NM,
                "canonical_bytes_per_step": w.canonical_bytes,
                "l2": ("flushed between timed steps by writing 512 MB (outside the per-step events)" if self.flush_l2
                       else f"no flush: each step streams {w.canonical_bytes / 1e9:.2f} GB, more than 4x the L2"),
                "variant": (f"cluster x{info['cluster']}" if info.get("cluster") else
                            "resident" if info["resident"] else "twopass"), "grid": info["grid"],
                "frames_per_tile": info["frames_per_tile"], "stages": info["stages"], "lag": info["lag"]}

    def kernel_note(self):
        return ("stft_logmel_kernel (one cooperative launch per step, timed with the workspace memset that "
                "precedes it)")

    def roofline(self, mean_launch_s, min_launch_s, peak, peak_kind, trec=None):
        achieved = self.bytes / mean_launch_s / 1e9
        return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "peak_kind": peak_kind, "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
                "basis": "canonical bytes / mean per-step CUDA-event time (each step's event pair brackets the "
                         "workspace memset and the kernel)",
                "traffic": (trec["dram_bytes_per_launch"] if trec else None),
                "traffic_source": ("profiles/traffic.json" if trec else "stale or missing"),
                "kernel": self.kernel_note(), "launch_ms_mean": mean_launch_s * 1e3,
                "launch_ms_min": min_launch_s * 1e3}

    def cpu_baseline(self):
        w = self.w
        # the whole batch (256 clips take about a second on 16 cores), repeated
        # for a stable figure
        return cpu_baseline(self.stft.cpu().numpy(), self.W.cpu().numpy(), target_s=2.0 if w.B <= 8 else 10.0,
                            sample_note=": the whole batch", got=self.out.cpu().numpy())


class WaveJob:
    """mel_spectrogram on one of the two waveform workloads."""

    def __init__(self, lm, workloads, dev, name, batch=0):
        import torch
        w = {"wave_whisper": workloads.WAVE_WHISPER, "wave_pcm16": workloads.WAVE_PCM16}[name]
        if batch and batch != w.B:
            import dataclasses
            w = dataclasses.replace(w, B=batch, name=w.name.replace(f"_b{w.B}_", f"_b{batch}_"))
        self.name = name
        self.lm, self.w, self.dev = lm, w, dev
        self.x = workloads.wave_workload_inputs(w, device=dev)
        self.mel = lm.MelSpectrogram(sample_rate=w.sample_rate, n_fft=w.n_fft, hop_length=w.hop_length,
                                     n_mels=w.n_mels, f_min=w.f_min, f_max=w.f_max, center=w.center,
                                     pad_mode=w.pad_mode, power=w.power, mel_scale=w.mel_scale, norm=w.norm,
                                     log_mel=w.log_mel,
                                     dtype=torch.float16 if w.out_dtype == "f16" else torch.float32)
        self.ws = torch.empty(self.mel.workspace_size(w.B, w.T, dev), dtype=torch.uint8, device=dev)
        self.out = self.mel(self.x, workspace=self.ws)
        self.units = w.B
        self.bytes = w.canonical_bytes
        self.flops = wave_flops(w)
        # log plans: the transform and the clamp kernel (one launch with
        # LOGMEL_K3_EPILOGUE=fused on the register kernels, n_fft <= 1024)
        fused = os.environ.get("LOGMEL_K3_EPILOGUE") == "fused" and w.n_fft <= 1024
        self.kernels = 2 if (w.log_mel and not fused) else 1
        self.flush_l2 = True  # 14-28 MB per step fits in L2
        self.inputs = [self.x]

    def step(self, inputs=None):
        x = inputs[0] if inputs is not None else self.x
        self.mel(x, out=self.out, workspace=self.ws)

    def error(self):
        return self.lm.workspace_error(self.ws)

    def host_setup(self):
        import torch
        self.h_x = torch.empty(self.x.shape, dtype=self.x.dtype, pin_memory=True)
        self.h_x.copy_(self.x)
        self.h_out = torch.empty(self.out.shape, dtype=self.out.dtype, pin_memory=True)
        return self.h_x.numel() * self.h_x.element_size(), self.h_out.numel() * self.h_out.element_size()

    def host_step(self):
        self.mel.host(self.h_x, device=self.dev, out=self.h_out, synchronize=False)

    def host_check(self):
        return bool(self.h_out.equal(self.out.cpu()))

    def host_api(self):
        return "MelSpectrogram.host -> lm_mel_spectrogram_host (chunked copy-in / kernel / copy-out pipeline)"

    def config(self):
        w = self.w
        return {"workload": w.name, "B": w.B, "T": w.T, "sample_rate": w.sample_rate, "n_fft": w.n_fft,
                "hop_length": w.hop_length, "n_mels": w.n_mels, "mel_scale": w.mel_scale, "in": w.in_dtype,
                "out": w.out_dtype, "log_mel": w.log_mel, "canonical_bytes_per_step": w.canonical_bytes,
                "l2": "flushed between timed steps by writing 512 MB (outside the per-step events)"}

    def kernel_note(self):
        return "wave_mel_kernel" + (" + logmel_clamp_kernel" if self.w.log_mel else "")

    def roofline(self, mean_launch_s, min_launch_s, peak, peak_kind, trec=None):
        achieved = self.bytes / mean_launch_s / 1e9
        tflops = self.flops / mean_launch_s / 1e12
        return {"bound": "alu", "achieved": tflops, "peak": FP32_PEAK_TFLOPS, "unit": "TFLOP/s",
                "frac": tflops / FP32_PEAK_TFLOPS,
                "peak_kind": "derived: 152 SMs x 128 FP32 lanes x 2 flops x 2.07 GHz",
                "basis": "algorithmic flops (bench.wave_flops) / mean per-step CUDA-event time",
                "traffic": None, "kernel": self.kernel_note(),
                "hbm_gbs": achieved, "hbm_frac_of_measured": achieved / peak,
                "flops_per_step": self.flops,
                "launch_ms_mean": mean_launch_s * 1e3, "launch_ms_min": min_launch_s * 1e3}

    def cpu_baseline(self):
        return cpu_baseline_wave(self.w, self.x.cpu().numpy(), got=self.out.float().cpu().numpy())


# FP32 FMA peak of the GPU from its unit counts and clock: 152 SMs x 128
# FP32 lanes x 2 flops per FMA x 2.07 GHz.
FP32_PEAK_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


def wave_flops(w) -> float:
    """Algorithmic flops of one waveform step: per frame, the N/2-point
    complex FFT at 5 (N/2) log2(N/2), the real-input untangle and power at 10
    per bin, the window at 1 per sample, the mel projection at 2 per filter
    tap (triangles overlap in pairs: about 2 taps per bin) and one log per
    band on log plans."""
    import math
    M = w.n_fft // 2
    nf = M + 1
    per_frame = 5 * M * math.log2(M) + 10 * nf + w.n_fft + 2 * 2 * nf + (w.n_mels if w.log_mel else 0)
    return w.B * w.n_frames * per_frame


def make_job(lm, workloads, dev, name, batch=0):
    if name in STFT_JOBS:
        return StftJob(lm, workloads, dev, batch, name)
    return WaveJob(lm, workloads, dev, name, batch)


def timed_steps(job, run_step, steps, stream, flush, dev, clk=None, soak_s=0.0):
    """Runs `steps` steps, each bracketed by CUDA events on the launching
    stream (an L2 flush, when given, runs between steps outside the events).
    With soak_s > 0 the same step first runs back to back, untimed, for about
    that long, directly before the timed steps, so that the clock samples
    describe the state the timed steps run in.  Returns the per-step times
    (ms), the total (ms) and the wall-clock window."""
    import torch
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    wall0 = time.time()
    if soak_s > 0:
        # about soak_s of back-to-back steps, enqueued in bursts so the host
        # stays ahead of the GPU
        per = max(1, int(soak_s * 1e3 / 0.25))
        for _ in range(per):
            run_step()
    t_begin.record(stream)
    for i in range(steps):
        if flush is not None:
            flush.fill_(i & 0xFF)
        starts[i].record(stream)
        run_step()
        ends[i].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    wall1 = time.time()
    if clk is not None:
        clk.mark(wall0, wall1)
    launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = sum(launch_ms) if flush is not None else t_begin.elapsed_time(t_end)
    return launch_ms, total_ms, (wall0, wall1)


def run_ours(args, world, rank, local):
    import torch

    import __graft_entry__
    import workloads

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    if rank == 0:
        __graft_entry__.build()
    barrier()
    import log_mel_spectrogram_gb300 as lm

    job = make_job(lm, workloads, dev, args.workload, args.batch)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device=dev)

    for _ in range(args.warmup):
        job.step()
    torch.cuda.synchronize(dev)
    if job.error():
        raise RuntimeError("device error word set during warm-up")
    run_step = job.step
    if args.graph:
        # One step captured once and replayed: the same kernels, without the
        # per-call host work (argument checks, plan lookup, launch calls).
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            job.step()
        graph.replay()
        torch.cuda.synchronize(dev)
        run_step = graph.replay

    props = torch.cuda.get_device_properties(dev)
    pci = None
    try:
        pci = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0"
    except Exception:
        pass
    barrier()
    with ClockSampler(local, pci) as clk:
        time.sleep(0.05)  # the sampler is running before the timed region
        launch_ms, total_ms, head_win = timed_steps(job, run_step, args.steps, stream,
                                                    flush if job.flush_l2 else None, dev, clk,
                                                    soak_s=args.clock_soak)
        barrier()
        if job.error():
            raise RuntimeError("device error word set during the timed region")

        # Host-observed latency of one call: wall clock from the call to the
        # end of a synchronize, with the inputs warm in L2.  Reported beside
        # the device-timed throughput; it is what a B=1 caller waits for.
        lat = []
        for _ in range(min(args.steps, 200)):
            h0 = time.perf_counter()
            run_step()
            torch.cuda.synchronize(dev)
            lat.append((time.perf_counter() - h0) * 1e3)
        lat.sort()

        total_ms = max_over_ranks(total_ms, world, dev)
        ms_per_step = total_ms / args.steps
        value = job_throughput(world, job.units, args.steps, total_ms)

        # End to end through the public host-buffer call: every step copies
        # the batch in from page-locked host memory and the result back out,
        # inside the timed region (the library overlaps the two directions and
        # the kernels chunk by chunk).  Inputs stay in host memory; the filter
        # matrix is a device-resident parameter, as in a serving process.  The
        # value is the whole run's throughput; per-step times are reported
        # beside it, since one host stall on a shared machine can weigh on a
        # short run.
        e2e_steps = 0 if args.no_e2e else max(1, min(args.steps, 60))
        e2e_value = None
        h2d = d2h = 0
        e2e_ok = None
        e2e_steps_ms = []
        if e2e_steps:
            h2d, d2h = job.host_setup()
            for _ in range(max(1, args.warmup)):
                job.host_step()  # warm-up (the first creates the library's copy streams)
            torch.cuda.synchronize(dev)
            barrier()
            marks = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps + 1)]
            marks[0].record(stream)
            for i in range(e2e_steps):
                job.host_step()
                marks[i + 1].record(stream)
            torch.cuda.synchronize(dev)
            barrier()
            e2e_steps_ms = sorted(marks[i].elapsed_time(marks[i + 1]) for i in range(e2e_steps))
            e2e_ms = max_over_ranks(marks[0].elapsed_time(marks[-1]), world, dev)
            e2e_value = job_throughput(world, job.units, e2e_steps, e2e_ms)
            e2e_ok = job.host_check()
            if not e2e_ok:
                raise RuntimeError("host-buffer result differs from the device result")

        # The other workloads of the configuration list, each timed on its own
        # (L2 flushed between steps) with the oracle timed beside it.  One GPU
        # only: under torchrun each rank would repeat them to no purpose.
        configs = {}
        peak, peak_kind = _peaks()
        if world == 1 and not args.no_configs and not args.batch and args.workload == "stft":
            for name in CONFIG_ORDER:
                if name == args.workload:
                    continue
                cj = make_job(lm, workloads, dev, name)
                for _ in range(args.warmup):
                    cj.step()
                torch.cuda.synchronize(dev)
                c_ms, c_total, _ = timed_steps(cj, cj.step, args.config_steps, stream, flush, dev, clk)
                if cj.error():
                    raise RuntimeError(f"device error word set while timing {name}")
                c_mean = statistics.mean(c_ms) / 1e3
                configs[name] = {
                    "workload": cj.w.name, "value": cj.units * args.config_steps / (c_total / 1e3),
                    "unit": "clips/s", "steps": args.config_steps, "ms_per_step": c_total / args.config_steps,
                    "ms_per_step_min": min(c_ms), "ms_per_step_median": statistics.median(c_ms),
                    "gpu_launches": args.config_steps * cj.kernels, "config": cj.config(),
                    "roofline": cj.roofline(c_mean, min(c_ms) / 1e3, peak, peak_kind),
                }
                del cj
                torch.cuda.empty_cache()
        clocks_head = clk.summary([head_win])
        clocks_all = clk.summary()

    mean_launch_s = statistics.mean(launch_ms) / 1e3
    trec = _traffic_record() if args.workload == "stft" and not args.batch else None
    config = job.config()
    config["parallelism"] = f"replicas x{world}" if world > 1 else "single GPU"
    config["launch"] = "cuda graph replay" if args.graph else "eager library call"
    if args.clock_soak > 0:
        config["clock_soak"] = (f"{args.clock_soak:g} s of the same step back to back, untimed, directly before "
                                "the timed steps (clock samples cover both)")
    roof = job.roofline(mean_launch_s, min(launch_ms) / 1e3, peak, peak_kind, trec)
    result = {
        "metric": METRIC if args.workload == "stft" else f"{job.w.name} clips/sec",
        "value": value,
        "unit": "clips/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded, generated on the device; see workloads.py)",
        "achieved_hbm_gbs": job.bytes / mean_launch_s / 1e9,
        "config": config,
        "roofline": roof,
        "e2e": {"value": e2e_value, "unit": "clips/s", "steps": e2e_steps,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "api": job.host_api() if e2e_steps else None,
                "equals_device_result": e2e_ok,
                "step_ms": ({"min": e2e_steps_ms[0], "median": e2e_steps_ms[len(e2e_steps_ms) // 2],
                             "max": e2e_steps_ms[-1]} if e2e_steps_ms else None),
                "value_at_median_step": (world * job.units / (e2e_steps_ms[len(e2e_steps_ms) // 2] / 1e3)
                                         if e2e_steps_ms else None)},
        "host_latency_ms": {"median": lat[len(lat) // 2], "p90": lat[(9 * len(lat)) // 10], "samples": len(lat),
                            "launch": "cuda graph replay" if args.graph else "eager library call"},
        "gpu_launches": args.steps * job.kernels,
        "clocks": clocks_head,
        "clocks_all_timed_regions": clocks_all,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # The oracle's run on each whole batch doubles as a parity check of
        # the GPU result the timed steps produced.
        result["cpu_baseline"] = job.cpu_baseline()
        result["parity"] = result["cpu_baseline"].pop("parity", None)
        for name, entry in configs.items():
            cj = make_job(lm, workloads, dev, name)
            for _ in range(max(1, args.warmup)):
                cj.step()
            entry["cpu_baseline"] = cj.cpu_baseline()
            entry["parity"] = entry["cpu_baseline"].pop("parity", None)
            del cj
    if configs:
        head = {"workload": job.w.name, "value": value, "unit": "clips/s", "steps": args.steps,
                "ms_per_step": ms_per_step, "roofline": roof, "see": "the top-level keys of this line"}
        if "cpu_baseline" in result:
            head["cpu_baseline"] = result["cpu_baseline"]
            head["parity"] = result.get("parity")
        configs[args.workload] = head
        result["configs"] = {n: configs[n] for n in CONFIG_ORDER if n in configs}
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


SWEEP_NFFT = (64, 256, 512, 1024, 4096, 16384)


def run_sweep(args, world, rank, local):
    """The full-spectrum sweep of the flashmel page's performance section:
    hop = n_fft / 4, 128 mels, B = 32 clips of T = 160000 samples, one line
    per n_fft in the sweep list (f32 in and out, no log; 16 kHz, HTK 0-8 kHz).
    Each size is timed over --config-steps calls with L2 flushed in between,
    and the oracle is timed beside it on a bounded sample (whole clips, up to
    about a second of CPU work; its DFT is O(N^2))."""
    import dataclasses
    import torch

    import __graft_entry__
    import workloads
    import oracle
    if rank != 0:
        return
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    __graft_entry__.build()
    import log_mel_spectrogram_gb300 as lm
    oracle.build()
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device=dev)
    peak, peak_kind = _peaks()
    base = workloads.WaveWorkload("sweep", 32, 160000, 16000, 1024, 256, 128, 0.0, 8000.0, "htk", "f32", "f32",
                                  False, 1005)
    rows = []
    with ClockSampler(local) as clk:
        for n_fft in args.sweep_nfft:
            w = dataclasses.replace(base, name=f"sweep_b32_t160000_nfft{n_fft}_hop{n_fft // 4}_htk128",
                                    n_fft=n_fft, hop_length=n_fft // 4)
            job = WaveJob.__new__(WaveJob)
            job.name, job.lm, job.w, job.dev = "sweep", lm, w, dev
            job.x = workloads.wave_workload_inputs(w, device=dev)
            job.mel = lm.MelSpectrogram(sample_rate=w.sample_rate, n_fft=w.n_fft, hop_length=w.hop_length,
                                        n_mels=w.n_mels, f_min=w.f_min, f_max=w.f_max, center=w.center,
                                        pad_mode=w.pad_mode, power=w.power, mel_scale=w.mel_scale, log_mel=False)
            job.ws = torch.empty(job.mel.workspace_size(w.B, w.T, dev), dtype=torch.uint8, device=dev)
            job.out = job.mel(job.x, workspace=job.ws)
            job.units, job.bytes, job.flops, job.kernels, job.flush_l2 = w.B, w.canonical_bytes, wave_flops(w), 1, True
            for _ in range(args.warmup):
                job.step()
            torch.cuda.synchronize(dev)
            ms, total, _ = timed_steps(job, job.step, args.config_steps, stream, flush, dev, clk)
            if job.error():
                raise RuntimeError(f"device error word set in the sweep at n_fft {n_fft}")
            us = statistics.median(ms) * 1e3
            # oracle: one call on as many whole clips as it has threads (it
            # runs one clip per thread)
            x_host = job.x.cpu().numpy()
            done = min(w.B, max(1, oracle.num_threads()))
            t0 = time.perf_counter()
            oracle.mel_spectrogram(x_host[:done], w.sample_rate, w.n_fft, w.hop_length, w.n_mels, f_max=w.f_max)
            cpu_s = time.perf_counter() - t0
            rows.append({"n_fft": n_fft, "hop": n_fft // 4, "n_frames": w.n_frames, "us_per_call_median": us,
                         "us_per_call_min": min(ms) * 1e3, "clips_per_s": w.B / (us / 1e6),
                         "essential_bytes": w.canonical_bytes, "essential_gbs": w.canonical_bytes / (us / 1e6) / 1e9,
                         "hbm_frac_of_measured": w.canonical_bytes / (us / 1e6) / 1e9 / peak,
                         "tflops": job.flops / (us / 1e6) / 1e12,
                         "cpu_baseline": {"clips_per_s": done / cpu_s, "cores": oracle.num_threads(), "kind": "oracle",
                                          "sample": f"{done} whole clips in one call, {cpu_s:.2f} s"}})
            job.mel.close()
            del job
            torch.cuda.empty_cache()
    print(json.dumps({"metric": "full-spectrum sweep: us per call (B=32, T=160000, hop=n_fft/4, 128 mels)",
                      "value": next((r["clips_per_s"] for r in rows if r["n_fft"] == 1024), rows[0]["clips_per_s"]),
                      "unit": "clips/s",
                      "n_gpus": 1, "steps": args.config_steps, "warmup": args.warmup, "higher_is_better": True,
                      "dtype": "f32", "data": "synthetic (seeded sinusoids, workloads.wave_sines)",
                      "config": {"workload": "sweep", "B": 32, "T": 160000, "sample_rate": 16000, "n_mels": 128,
                                 "l2": "flushed between timed calls by writing 512 MB"},
                      "peak_hbm_gbs": peak, "peak_kind": peak_kind, "sweep": rows,
                      "clocks": clk.summary()}), flush=True)


def run_reference(args, world, rank):
    """The oracle timed on host cores, each step a bounded sample of clips."""
    if rank != 0:
        return
    import oracle
    import workloads
    oracle.build()
    w = workloads.WHISPER_STFT_B256
    clips = args.reference_clips
    stft, W = workloads.stft_inputs(clips, w.F, w.NF, w.NM, w.seed, device="cpu")
    stft_np, W_np = stft.numpy(), W.numpy()
    for _ in range(args.warmup):
        oracle.log_mel_from_stft(stft_np[:1], W_np)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.log_mel_from_stft(stft_np, W_np)
    dt = time.perf_counter() - t0
    value = clips * args.steps / dt
    cores = oracle.num_threads()
    sample = f"{clips} of {w.B} clips per step (F={w.F}, NF={w.NF}, NM={w.NM}), dense double-precision oracle"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "clips/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "F": w.F, "NF": w.NF, "NM": w.NM, "sampled_clips": clips},
        "cpu_baseline": {"value": value, "unit": "clips/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "clips/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def run_torch_eager(args, world, rank, local):
    """Context only: the per-clip definition composed from eager PyTorch ops
    on the same GPU (power, dense projection, log10, clip max, clamp,
    rescale), timed like the library call.  Not the reference arm."""
    import torch

    import workloads
    if rank != 0:
        return
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = workloads.WHISPER_STFT_B256
    stft, W = workloads.stft_workload_inputs(w, device=dev)

    def step():
        mag = torch.view_as_real(stft).square().sum(-1)
        mel = mag @ W.t()
        ls = torch.log10(mel.clamp_min(1e-10))
        hi = ls.amax(dim=(1, 2), keepdim=True)
        return (torch.maximum(ls, hi - 8.0) + 4.0) / 4.0

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        step()
    e1.record()
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / args.steps
    achieved = w.canonical_bytes / (ms / 1e3) / 1e9
    peak, peak_kind = _peaks()
    print(json.dumps({"impl": "torch_eager", "metric": METRIC, "value": w.B / (ms / 1e3), "unit": "clips/s",
                      "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
                      "higher_is_better": True, "dtype": "f32", "data": "synthetic",
                      "config": {"workload": w.name, "B": w.B, "F": w.F, "NF": w.NF, "NM": w.NM},
                      "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                                   "frac": achieved / peak, "peak_kind": peak_kind}}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference", "torch_eager"], default="ours",
                    help="ours (the library), reference (the CPU oracle), or torch_eager (context: the "
                         "definition as eager PyTorch ops on the GPU)")
    ap.add_argument("--reference-clips", type=int, default=16)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer leg (profiling runs)")
    ap.add_argument("--batch", type=int, default=0, help="override B (profiling runs on smaller cases)")
    ap.add_argument("--graph", action="store_true", help="replay one captured CUDA graph per step")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other four workloads of the configuration list (profiling runs)")
    ap.add_argument("--config-steps", type=int, default=200,
                    help="timed steps for each of the other workloads (L2 flushed between steps)")
    ap.add_argument("--clock-soak", type=float, default=1.0,
                    help="seconds of untimed back-to-back steps directly before the timed steps, so that the "
                         "clock samples describe a GPU under this load (0 = none)")
    ap.add_argument("--workload", choices=["stft", "stft_small", "stft_b8", "wave_whisper", "wave_pcm16", "sweep"],
                    default="stft",
                    help="stft (default, the headline: B=256, F=3000, NM=128), stft_small (B=1, F=300, NM=80), "
                         "stft_b8 (B=8, F=3000, NM=80), one of the waveform workloads, or sweep (n_fft 64..16384)")
    ap.add_argument("--sweep-nfft", type=lambda v: tuple(int(n) for n in v.split(",")), default=SWEEP_NFFT,
                    help="comma-separated n_fft values for --workload sweep (default: the page's sweep, "
                         + ",".join(map(str, SWEEP_NFFT)) + ")")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = _dist()
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    if args.impl == "torch_eager":
        run_torch_eager(args, world, rank, local)
        return
    if args.workload == "sweep":
        run_sweep(args, world, rank, local)
        return
    run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
