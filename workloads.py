"""Seeded synthetic inputs for the log-mel front end.

This module only draws inputs. It holds none of the log-mel arithmetic, so the
CUDA path and the CPU oracle can both be fed from it without sharing any of
the computation they are checked on.

Two families of input:

* Complex STFTs plus a dense triangular filterbank, drawn the way the KBench
  task spec "audio-mel-spectrogram-fused" builds its inputs (its
  ``make_inputs`` recipe): re and im are Gaussian, scaled by a spectral tilt
  exp(-k / (NF/3)) and a per-frame envelope 0.05 + U(0,1)^2; the NM filters
  are triangles between NM+2 equally spaced centres over bins 0..NF-1.
* Waveforms for the mel spectrogram path (the flashmel page's use case):
  a sum of three sinusoids with noise and a slow envelope (f32), or clipped
  Gaussian int16 PCM.

Everything is seeded; ``device`` chooses where torch draws the numbers.  The
same buffer is handed to the GPU path and the oracle, so the two never need
to agree on a random stream.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class StftWorkload:
    """A ``log_mel_from_stft`` problem: stft[B,F,NF] complex64, filters[NM,NF]."""
    name: str
    B: int
    F: int
    NF: int
    NM: int
    seed: int

    @property
    def canonical_bytes(self) -> int:
        # One read of the complex64 source, one write of the f32 result
        # (the byte count the KBench spec states from the shape alone).
        return self.B * self.F * self.NF * 8 + self.B * self.F * self.NM * 4


@dataclasses.dataclass(frozen=True)
class WaveWorkload:
    """A ``mel_spectrogram`` problem on a batch of waveforms."""
    name: str
    B: int
    T: int
    sample_rate: int
    n_fft: int
    hop_length: int
    n_mels: int
    f_min: float
    f_max: float
    mel_scale: str          # "htk" or "slaney"
    in_dtype: str           # "f32" or "i16"
    out_dtype: str          # "f32" or "f16"
    log_mel: bool
    seed: int
    center: bool = True
    pad_mode: str = "reflect"
    power: float = 2.0
    norm: str | None = None

    @property
    def n_frames(self) -> int:
        if self.center:
            return 1 + self.T // self.hop_length
        return 1 + (self.T - self.n_fft) // self.hop_length

    @property
    def canonical_bytes(self) -> int:
        in_b = 4 if self.in_dtype == "f32" else 2
        out_b = 4 if self.out_dtype == "f32" else 2
        return self.B * self.T * in_b + self.B * self.n_mels * self.n_frames * out_b


# The five workloads the front end is measured and checked on.  Seeds are
# 1000 + position.
WHISPER_STFT_SMALL = StftWorkload("stft_b1_f300_nf201_nm80", 1, 300, 201, 80, 1000)
WHISPER_STFT = StftWorkload("stft_b8_f3000_nf201_nm80", 8, 3000, 201, 80, 1001)
WHISPER_STFT_B256 = StftWorkload("stft_b256_f3000_nf201_nm128", 256, 3000, 201, 128, 1002)
WAVE_WHISPER = WaveWorkload("wave_f32_b8_t480000_nfft400_htk128_log", 8, 480000, 16000, 400, 160,
                            128, 0.0, 8000.0, "htk", "f32", "f32", True, 1003)
WAVE_PCM16 = WaveWorkload("wave_i16_b32_t220500_nfft1024_slaney128_f16", 32, 220500, 22050, 1024,
                          256, 128, 0.0, 11025.0, "slaney", "i16", "f16", False, 1004)

STFT_WORKLOADS = (WHISPER_STFT_SMALL, WHISPER_STFT, WHISPER_STFT_B256)
WAVE_WORKLOADS = (WAVE_WHISPER, WAVE_PCM16)

# Ragged / odd shapes the KBench spec lists for correctness (F ragged, small odd NF).
STFT_CORRECTNESS_SHAPES = ((3, 301, 201, 128), (5, 128, 65, 40), (2, 3000, 201, 128), (7, 97, 129, 80))


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def triangle_filters(NF: int, NM: int, device="cpu") -> torch.Tensor:
    """Dense [NM, NF] f32 filters: NM overlapping triangles between NM+2
    equally spaced centres over bins 0..NF-1 (the spec's input recipe)."""
    centres = torch.linspace(0, NF - 1, NM + 2, device=device)
    bins = torch.arange(NF, device=device, dtype=torch.float32).view(1, NF)
    lo = centres[:-2].view(NM, 1)
    mid = centres[1:-1].view(NM, 1)
    hi = centres[2:].view(NM, 1)
    left = (bins - lo) / (mid - lo).clamp(min=1e-6)
    right = (hi - bins) / (hi - mid).clamp(min=1e-6)
    return torch.minimum(left, right).clamp(min=0.0).contiguous()


def stft_inputs(B: int, F: int, NF: int, NM: int, seed: int, device="cpu"):
    """(stft [B,F,NF] complex64, mel_filters [NM,NF] f32), speech-tilted Gaussian."""
    g = _gen(seed, device)
    tilt = torch.exp(-torch.arange(NF, device=device, dtype=torch.float32) / (NF / 3.0)).view(1, 1, NF)
    env = 0.05 + torch.rand(B, F, 1, device=device, generator=g) ** 2
    re = torch.randn(B, F, NF, device=device, generator=g) * tilt * env
    im = torch.randn(B, F, NF, device=device, generator=g) * tilt * env
    stft = torch.complex(re, im)
    del re, im
    return stft.contiguous(), triangle_filters(NF, NM, device)


def stft_workload_inputs(w: StftWorkload, device="cpu"):
    return stft_inputs(w.B, w.F, w.NF, w.NM, w.seed, device)


def wave_sines(B: int, T: int, sample_rate: int, seed: int, device="cpu") -> torch.Tensor:
    """f32 [B,T]: 3 sinusoids (f ~ U(100,4000) Hz, a ~ U(0.1,0.5), phase ~ U(0,2pi))
    plus N(0, 0.01) noise, times a piecewise-linear envelope through U(0.2,1.0)
    knots every 0.5 s."""
    g = _gen(seed, device)
    f = 100.0 + 3900.0 * torch.rand(B, 3, 1, device=device, generator=g, dtype=torch.float64)
    a = 0.1 + 0.4 * torch.rand(B, 3, 1, device=device, generator=g, dtype=torch.float64)
    ph = 2 * math.pi * torch.rand(B, 3, 1, device=device, generator=g, dtype=torch.float64)
    t = torch.arange(T, device=device, dtype=torch.float64).view(1, 1, T) / sample_rate
    x = (a * torch.sin(2 * math.pi * f * t + ph)).sum(dim=1)
    x = x + 0.01 * torch.randn(B, T, device=device, generator=g, dtype=torch.float64)
    knot_step = sample_rate // 2
    n_knots = T // knot_step + 2
    knots = 0.2 + 0.8 * torch.rand(B, n_knots, device=device, generator=g, dtype=torch.float64)
    pos = torch.arange(T, device=device, dtype=torch.float64) / knot_step
    i0 = pos.floor().long()
    frac = (pos - i0).view(1, T)
    env = knots[:, i0] * (1 - frac) + knots[:, i0 + 1] * frac
    return (x * env).to(torch.float32).contiguous()


def wave_pcm16(B: int, T: int, seed: int, device="cpu") -> torch.Tensor:
    """i16 [B,T]: round-half-even(N(0,1) * 3000), clipped to the int16 range."""
    g = _gen(seed, device)
    x = torch.randn(B, T, device=device, generator=g, dtype=torch.float32) * 3000.0
    return torch.round(x).clamp(-32768, 32767).to(torch.int16).contiguous()


def wave_workload_inputs(w: WaveWorkload, device="cpu", B: int | None = None, T: int | None = None):
    B = w.B if B is None else B
    T = w.T if T is None else T
    if w.in_dtype == "f32":
        return wave_sines(B, T, w.sample_rate, w.seed, device)
    return wave_pcm16(B, T, w.seed, device)
