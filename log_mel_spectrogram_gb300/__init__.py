"""GB300-native log-mel front end: a thin torch binding over liblogmel.so.

Every step of both operations runs in the library's CUDA kernels; this module
only checks tensor arguments, allocates outputs and workspaces through torch
and passes raw pointers plus torch's current stream to the C ABI
(include/logmel.h).  There is no CPU fallback: calls fail when the library is
missing or the tensors are not on a CUDA device.

* ``log_mel_from_stft(stft, mel_filters)`` -- Whisper's log-mel spectrogram
  from a complex STFT (KBench "audio_mel_spectrogram_fused" spec).
* ``mel_spectrogram(wave, ...)`` / ``MelSpectrogram`` -- waveform to mel
  spectrogram with torchaudio-style arguments (flashmel page).
"""
from __future__ import annotations

import ctypes

import torch

from . import _native
from ._native import LogmelError

__all__ = ["log_mel_from_stft", "log_mel_from_stft_workspace_size", "workspace_error", "LogmelError",
           "describe_log_mel_from_stft",
           "library_path"]


def library_path():
    return _native.library_path()


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _require_cuda(t: torch.Tensor, name: str) -> None:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def log_mel_from_stft_workspace_size(B: int, F: int, NF: int, NM: int) -> int:
    n = ctypes.c_size_t()
    _native.check(_native.lib().lm_log_mel_from_stft_workspace_size(int(B), int(F), int(NF), int(NM),
                                                                    ctypes.byref(n)),
                  "lm_log_mel_from_stft_workspace_size")
    return int(n.value)


def log_mel_from_stft(stft: torch.Tensor, mel_filters: torch.Tensor, out: torch.Tensor | None = None,
                      workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """stft [B,F,NF] complex64, mel_filters [NM,NF] float32 -> [B,F,NM] float32."""
    _require_cuda(stft, "stft")
    _require_cuda(mel_filters, "mel_filters")
    if stft.dtype != torch.complex64 or stft.dim() != 3:
        raise ValueError("stft must be a [B, F, NF] complex64 tensor")
    if mel_filters.dtype != torch.float32 or mel_filters.dim() != 2 or mel_filters.shape[1] != stft.shape[2]:
        raise ValueError("mel_filters must be a [NM, NF] float32 tensor")
    B, F, NF = stft.shape
    NM = mel_filters.shape[0]
    if out is None:
        out = torch.empty((B, F, NM), dtype=torch.float32, device=stft.device)
    elif out.shape != (B, F, NM) or out.dtype != torch.float32 or not out.is_contiguous():
        raise ValueError("out must be a contiguous [B, F, NM] float32 tensor")
    ws_bytes = log_mel_from_stft_workspace_size(B, F, NF, NM)
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=stft.device)
    elif workspace.numel() * workspace.element_size() < ws_bytes:
        raise ValueError(f"workspace needs {ws_bytes} bytes")
    rc = _native.lib().lm_log_mel_from_stft(stft.data_ptr(), mel_filters.data_ptr(), out.data_ptr(), B, F, NF,
                                            NM, workspace.data_ptr(),
                                            workspace.numel() * workspace.element_size(),
                                            _stream_handle(stream))
    _native.check(rc, "lm_log_mel_from_stft")
    return out


def describe_log_mel_from_stft(B: int, F: int, NF: int, NM: int) -> dict:
    """How the library will launch this shape on the current device."""
    info = _native.StftLaunchInfo()
    _native.check(_native.lib().lm_log_mel_from_stft_describe(B, F, NF, NM, ctypes.byref(info)),
                  "lm_log_mel_from_stft_describe")
    return {name: getattr(info, name) for name, _ in info._fields_}


def workspace_error(workspace: torch.Tensor, stream=None) -> int:
    """Synchronise and return the workspace's device error word (0 = none)."""
    v = ctypes.c_uint32()
    _native.lib().lm_workspace_error(workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                     ctypes.byref(v), _stream_handle(stream))
    return int(v.value)
