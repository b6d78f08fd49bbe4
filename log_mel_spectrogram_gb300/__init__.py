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

import collections
import ctypes
import threading
import weakref

import torch

from . import _native
from ._native import LogmelError

__all__ = ["log_mel_from_stft", "log_mel_from_stft_workspace_size", "workspace_error", "LogmelError",
           "pack_mel_filters", "log_mel_from_stft_host", "log_mel_from_stft_host_workspace_size",
           "describe_log_mel_from_stft", "MelSpectrogram", "mel_spectrogram", "library_path",
           "log_mel_from_stft_op", "mel_spectrogram_op"]


def library_path():
    return _native.library_path()


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _no_grad_inputs(*tensors: torch.Tensor) -> None:
    """Inference only: a tensor that requires grad under grad mode is refused."""
    if torch.is_grad_enabled() and any(t.requires_grad for t in tensors):
        raise RuntimeError("log_mel_spectrogram_gb300 ops are inference-only: inputs must not require grad "
                           "(use torch.no_grad() or detach())")


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


def pack_mel_filters(mel_filters: torch.Tensor, stream=None) -> torch.Tensor:
    """Packs a [NM, NF] float32 CUDA filter matrix once (each band's first
    nonzero bin, width and first 8 weights; lm_mel_filters_pack) so that
    log_mel_from_stft calls with it skip the per-call derivation.  Returns the
    pack as a uint8 CUDA tensor, filled in stream order."""
    _require_cuda(mel_filters, "mel_filters")
    if mel_filters.dtype != torch.float32 or mel_filters.dim() != 2:
        raise ValueError("mel_filters must be a [NM, NF] float32 tensor")
    NM, NF = mel_filters.shape
    n = ctypes.c_size_t()
    _native.check(_native.lib().lm_mel_filters_pack_size(NF, NM, ctypes.byref(n)), "lm_mel_filters_pack_size")
    packed = torch.empty(n.value, dtype=torch.uint8, device=mel_filters.device)
    _native.check(_native.lib().lm_mel_filters_pack(mel_filters.data_ptr(), NF, NM, packed.data_ptr(), n.value,
                                                    _stream_handle(stream)), "lm_mel_filters_pack")
    return packed


# Packs made on behalf of callers, one per live filter tensor and version
# (torch bumps a tensor's version on every in-place write, views included);
# an entry goes when its tensor is freed.  Never filled during graph capture.
_PACKS: collections.OrderedDict = collections.OrderedDict()
_PACKS_MAX = 32
_PACK_FINALIZERS: set = set()
_PACKS_LOCK = threading.RLock()  # host threads may call concurrently


def _drop_packs(tid: int) -> None:
    with _PACKS_LOCK:
        _PACK_FINALIZERS.discard(tid)
        for k in [k for k in _PACKS if k[0] == tid]:
            del _PACKS[k]


def _cached_pack(mel_filters: torch.Tensor, stream) -> torch.Tensor:
    if torch.cuda.is_current_stream_capturing():
        return pack_mel_filters(mel_filters, stream)
    try:
        version = mel_filters._version
    except RuntimeError:  # inference tensors keep no version counter: no cache
        return None
    tid = id(mel_filters)
    key = (tid, version, mel_filters.data_ptr(), tuple(mel_filters.shape), mel_filters.device.index)
    with _PACKS_LOCK:
        hit = _PACKS.get(key)
        if hit is not None:
            _PACKS.move_to_end(key)
            return hit
        for k in [k for k in _PACKS if k[0] == tid]:
            del _PACKS[k]
        packed = pack_mel_filters(mel_filters, stream)
        _PACKS[key] = packed
        if tid not in _PACK_FINALIZERS:
            weakref.finalize(mel_filters, _drop_packs, tid)
            _PACK_FINALIZERS.add(tid)
        while len(_PACKS) > _PACKS_MAX:
            _PACKS.popitem(last=False)
    return packed


def log_mel_from_stft(stft: torch.Tensor, mel_filters: torch.Tensor, out: torch.Tensor | None = None,
                      workspace: torch.Tensor | None = None, stream=None, packed=None) -> torch.Tensor:
    """stft [B,F,NF] complex64, mel_filters [NM,NF] float32 -> [B,F,NM] float32.

    packed: None (default) packs mel_filters once per tensor version and
    reuses the pack; a tensor from pack_mel_filters(mel_filters) uses that
    pack; False derives supports and weights from the dense matrix every call."""
    _no_grad_inputs(stft, mel_filters)
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
    ws_len = workspace.numel() * workspace.element_size()
    if packed is None:
        packed = _cached_pack(mel_filters, stream)
        if packed is None:
            packed = False
    if packed is False:
        rc = _native.lib().lm_log_mel_from_stft(stft.data_ptr(), mel_filters.data_ptr(), out.data_ptr(), B, F,
                                                NF, NM, workspace.data_ptr(), ws_len, _stream_handle(stream))
        _native.check(rc, "lm_log_mel_from_stft")
        return out
    if not isinstance(packed, torch.Tensor) or not packed.is_cuda:
        raise ValueError("packed must be None, False or a tensor from pack_mel_filters")
    rc = _native.lib().lm_log_mel_from_stft_packed(stft.data_ptr(), mel_filters.data_ptr(), packed.data_ptr(),
                                                   out.data_ptr(), B, F, NF, NM, workspace.data_ptr(), ws_len,
                                                   _stream_handle(stream))
    _native.check(rc, "lm_log_mel_from_stft_packed")
    return out


def _require_host(t: torch.Tensor, name: str) -> None:
    if not isinstance(t, torch.Tensor) or t.device.type != "cpu":
        raise ValueError(f"{name} must be a CPU tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _host_output(shape, dtype, like: torch.Tensor, out: torch.Tensor | None) -> torch.Tensor:
    if out is None:
        return torch.empty(shape, dtype=dtype, pin_memory=like.is_pinned())
    _require_host(out, "out")
    if tuple(out.shape) != tuple(shape) or out.dtype != dtype:
        raise ValueError(f"out must be a contiguous {tuple(shape)} {dtype} CPU tensor")
    return out


def log_mel_from_stft_host_workspace_size(B: int, F: int, NF: int, NM: int, chunk_clips: int = 0) -> int:
    n = ctypes.c_size_t()
    _native.check(_native.lib().lm_log_mel_from_stft_host_workspace_size(int(B), int(F), int(NF), int(NM),
                                                                         int(chunk_clips), ctypes.byref(n)),
                  "lm_log_mel_from_stft_host_workspace_size")
    return int(n.value)


def log_mel_from_stft_host(stft: torch.Tensor, mel_filters: torch.Tensor, out: torch.Tensor | None = None,
                           workspace: torch.Tensor | None = None, stream=None, packed=None, chunk_clips: int = 0,
                           synchronize: bool = True) -> torch.Tensor:
    """log_mel_from_stft for a batch in host memory: stft [B,F,NF] complex64
    on the CPU (pinned, for the copies to overlap the kernels), mel_filters
    [NM,NF] float32 on the GPU that computes -> [B,F,NM] float32 on the CPU.

    The library pipelines chunks of whole clips through device staging slots
    (lm_log_mel_from_stft_host).  With synchronize=False the result is
    complete only once the stream reaches the end of the call's work."""
    _no_grad_inputs(stft, mel_filters)
    _require_host(stft, "stft")
    _require_cuda(mel_filters, "mel_filters")
    if stft.dtype != torch.complex64 or stft.dim() != 3:
        raise ValueError("stft must be a [B, F, NF] complex64 tensor")
    if mel_filters.dtype != torch.float32 or mel_filters.dim() != 2 or mel_filters.shape[1] != stft.shape[2]:
        raise ValueError("mel_filters must be a [NM, NF] float32 tensor")
    B, F, NF = stft.shape
    NM = mel_filters.shape[0]
    out = _host_output((B, F, NM), torch.float32, stft, out)
    with torch.cuda.device(mel_filters.device):
        ws_bytes = log_mel_from_stft_host_workspace_size(B, F, NF, NM, chunk_clips)
        if workspace is None:
            workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=mel_filters.device)
        elif not workspace.is_cuda or workspace.numel() * workspace.element_size() < ws_bytes:
            raise ValueError(f"workspace must be a CUDA tensor of at least {ws_bytes} bytes")
        if packed is None:
            packed = _cached_pack(mel_filters, stream)
        if packed is False:
            packed = None
        if packed is not None and (not isinstance(packed, torch.Tensor) or not packed.is_cuda):
            raise ValueError("packed must be None, False or a tensor from pack_mel_filters")
        rc = _native.lib().lm_log_mel_from_stft_host(
            stft.data_ptr(), mel_filters.data_ptr(), packed.data_ptr() if packed is not None else None,
            out.data_ptr(), B, F, NF, NM, int(chunk_clips), workspace.data_ptr(),
            workspace.numel() * workspace.element_size(), _stream_handle(stream))
        _native.check(rc, "lm_log_mel_from_stft_host")
        if synchronize:
            (stream or torch.cuda.current_stream()).synchronize()
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


class MelSpectrogram:
    """Waveform -> mel spectrogram with torchaudio MelSpectrogram argument names
    (window fixed to periodic Hann, onesided).  Holds one library plan per
    CUDA device.  ``log_mel=True`` adds log10(max(x, 1e-10)), the per-clip
    clamp at max - 8 and the (x + 4) / 4 rescale."""

    def __init__(self, sample_rate: int = 16000, n_fft: int = 400, win_length: int | None = None,
                 hop_length: int | None = None, f_min: float = 0.0, f_max: float | None = None, pad: int = 0,
                 n_mels: int = 128, power: float = 2.0, normalized: bool = False, center: bool = True,
                 pad_mode: str = "reflect", norm: str | None = None, mel_scale: str = "htk",
                 log_mel: bool = False, dtype: torch.dtype = torch.float32):
        self.params = _native.MelParams(
            sample_rate=int(sample_rate), n_fft=int(n_fft), win_length=int(win_length or 0),
            hop_length=int(hop_length if hop_length is not None else (win_length or n_fft) // 2),
            n_mels=int(n_mels), f_min=float(f_min), f_max=float(f_max if f_max is not None else 0.0),
            pad=int(pad), center=int(bool(center)), pad_mode=_native.PAD_MODES[pad_mode], power=float(power),
            normalized=int(bool(normalized)), mel_scale=_native.MEL_SCALES[mel_scale],
            slaney_norm=int(norm == "slaney"), log_mel=int(bool(log_mel)))
        if dtype not in (torch.float32, torch.float16):
            raise ValueError("dtype must be torch.float32 or torch.float16")
        self.dtype = dtype
        self.n_mels = int(n_mels)
        self._plans: dict[int, int] = {}

    def _plan(self, device: torch.device) -> int:
        idx = device.index if device.index is not None else torch.cuda.current_device()
        plan = self._plans.get(idx)
        if plan is None:
            with torch.cuda.device(idx):
                handle = ctypes.c_void_p()
                _native.check(_native.lib().lm_mel_plan_create(ctypes.byref(self.params), ctypes.byref(handle)),
                              "lm_mel_plan_create")
            plan = self._plans[idx] = handle.value
        return plan

    def n_frames(self, T: int) -> int:
        if not self._plans:
            self._plan(torch.device("cuda", torch.cuda.current_device()))
        n = ctypes.c_int64()
        _native.check(_native.lib().lm_mel_n_frames(next(iter(self._plans.values())), int(T), ctypes.byref(n)),
                      "lm_mel_n_frames")
        return int(n.value)

    def workspace_size(self, B: int, T: int, device=None) -> int:
        """Bytes of device workspace a call on B clips of T samples needs
        (lm_mel_workspace_size); pass such a tensor as ``workspace`` to read
        its device error word afterwards with workspace_error()."""
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        need = ctypes.c_size_t()
        _native.check(_native.lib().lm_mel_workspace_size(self._plan(dev), int(B), int(T), ctypes.byref(need)),
                      "lm_mel_workspace_size")
        return max(int(need.value), 16)

    def __call__(self, wave: torch.Tensor, out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                 stream=None) -> torch.Tensor:
        _no_grad_inputs(wave)
        _require_cuda(wave, "wave")
        if wave.dtype == torch.int16:
            in_code = _native.DTYPES["i16"]
        elif wave.dtype == torch.float32:
            in_code = _native.DTYPES["f32"]
        else:
            raise ValueError("wave must be float32 or int16")
        lead = wave.shape[:-1]
        T = wave.shape[-1]
        w2 = wave.reshape(-1, T)
        B = w2.shape[0]
        with torch.cuda.device(wave.device):
            plan = self._plan(wave.device)
            nfr = ctypes.c_int64()
            _native.check(_native.lib().lm_mel_n_frames(plan, T, ctypes.byref(nfr)), "lm_mel_n_frames")
            shape = (B, self.n_mels, nfr.value)
            if out is None:
                out = torch.empty(shape, dtype=self.dtype, device=wave.device)
            elif tuple(out.shape) != shape or out.dtype != self.dtype or not out.is_contiguous():
                raise ValueError(f"out must be a contiguous {shape} {self.dtype} tensor")
            need = ctypes.c_size_t()
            _native.check(_native.lib().lm_mel_workspace_size(plan, B, T, ctypes.byref(need)), "lm_mel_workspace_size")
            if workspace is None:
                workspace = torch.empty(max(need.value, 16), dtype=torch.uint8, device=wave.device)
            out_code = _native.DTYPES["f16" if self.dtype == torch.float16 else "f32"]
            rc = _native.lib().lm_mel_spectrogram(plan, w2.data_ptr(), in_code, B, T, out.data_ptr(), out_code,
                                                  workspace.data_ptr(),
                                                  workspace.numel() * workspace.element_size(),
                                                  _stream_handle(stream))
            _native.check(rc, "lm_mel_spectrogram")
        return out.reshape(*lead, self.n_mels, nfr.value)

    def host(self, wave: torch.Tensor, device=None, out: torch.Tensor | None = None,
             workspace: torch.Tensor | None = None, stream=None, chunk_clips: int = 0,
             synchronize: bool = True) -> torch.Tensor:
        """The same transform for waveforms in host memory (pinned, for the
        copies to overlap the kernels), computed on `device` (default: the
        current CUDA device) and returned in host memory
        (lm_mel_spectrogram_host).  With synchronize=False the result is
        complete only once the stream reaches the end of the call's work."""
        _no_grad_inputs(wave)
        _require_host(wave, "wave")
        if wave.dtype == torch.int16:
            in_code = _native.DTYPES["i16"]
        elif wave.dtype == torch.float32:
            in_code = _native.DTYPES["f32"]
        else:
            raise ValueError("wave must be float32 or int16")
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        lead = wave.shape[:-1]
        T = wave.shape[-1]
        w2 = wave.reshape(-1, T)
        B = w2.shape[0]
        with torch.cuda.device(dev):
            plan = self._plan(dev)
            nfr = ctypes.c_int64()
            _native.check(_native.lib().lm_mel_n_frames(plan, T, ctypes.byref(nfr)), "lm_mel_n_frames")
            out = _host_output((B, self.n_mels, nfr.value), self.dtype, wave, out)
            out_code = _native.DTYPES["f16" if self.dtype == torch.float16 else "f32"]
            need = ctypes.c_size_t()
            _native.check(_native.lib().lm_mel_spectrogram_host_workspace_size(
                plan, B, T, in_code, out_code, int(chunk_clips), ctypes.byref(need)),
                "lm_mel_spectrogram_host_workspace_size")
            if workspace is None:
                workspace = torch.empty(need.value, dtype=torch.uint8, device=dev)
            elif not workspace.is_cuda or workspace.numel() * workspace.element_size() < need.value:
                raise ValueError(f"workspace must be a CUDA tensor of at least {need.value} bytes")
            rc = _native.lib().lm_mel_spectrogram_host(plan, w2.data_ptr(), in_code, B, T, out.data_ptr(), out_code,
                                                       int(chunk_clips), workspace.data_ptr(),
                                                       workspace.numel() * workspace.element_size(),
                                                       _stream_handle(stream))
            _native.check(rc, "lm_mel_spectrogram_host")
            if synchronize:
                (stream or torch.cuda.current_stream()).synchronize()
        return out.reshape(*lead, self.n_mels, nfr.value)

    def close(self) -> None:
        for plan in self._plans.values():
            _native.lib().lm_mel_plan_destroy(plan)
        self._plans.clear()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def mel_spectrogram(wave: torch.Tensor, **kwargs) -> torch.Tensor:
    """One-shot functional form of MelSpectrogram (builds a plan per call)."""
    m = MelSpectrogram(**kwargs)
    try:
        out = m(wave)
        torch.cuda.current_stream(wave.device).synchronize()
        return out
    finally:
        m.close()


# ---------------------------------------------------------------------------
# torch integration: custom ops with shape-only fake implementations, so that
# torch.compile(fullgraph=True) traces through the library calls.  Inference
# only: a tensor that requires grad under grad mode is rejected.
# ---------------------------------------------------------------------------

@torch.library.custom_op("logmel_gb300::log_mel_from_stft", mutates_args=())
def log_mel_from_stft_op(stft: torch.Tensor, mel_filters: torch.Tensor) -> torch.Tensor:
    """Custom-op form of log_mel_from_stft (same arguments and result)."""
    _no_grad_inputs(stft, mel_filters)
    return log_mel_from_stft(stft.contiguous(), mel_filters.contiguous())


@log_mel_from_stft_op.register_fake
def _(stft, mel_filters):
    return stft.new_empty((stft.shape[0], stft.shape[1], mel_filters.shape[0]), dtype=torch.float32)


_OP_PLANS: dict = {}


def _op_frames(T: int, n_fft: int, hop: int, pad: int, center: bool) -> int:
    length = T + 2 * pad + (2 * (n_fft // 2) if center else 0)
    return 0 if length < n_fft else 1 + (length - n_fft) // hop


@torch.library.custom_op("logmel_gb300::mel_spectrogram", mutates_args=())
def mel_spectrogram_op(wave: torch.Tensor, sample_rate: int, n_fft: int, win_length: int, hop_length: int,
                       f_min: float, f_max: float, pad: int, n_mels: int, power: float, normalized: bool,
                       center: bool, pad_mode: str, norm: str, mel_scale: str, log_mel: bool,
                       half: bool) -> torch.Tensor:
    """Custom-op form of MelSpectrogram(...)(wave); plans are cached per argument set."""
    _no_grad_inputs(wave)
    key = (sample_rate, n_fft, win_length, hop_length, f_min, f_max, pad, n_mels, power, normalized, center,
           pad_mode, norm, mel_scale, log_mel, half)
    m = _OP_PLANS.get(key)
    if m is None:
        m = _OP_PLANS[key] = MelSpectrogram(
            sample_rate=sample_rate, n_fft=n_fft, win_length=win_length or None, hop_length=hop_length,
            f_min=f_min, f_max=f_max if f_max > 0 else None, pad=pad, n_mels=n_mels, power=power,
            normalized=normalized, center=center, pad_mode=pad_mode, norm=norm or None, mel_scale=mel_scale,
            log_mel=log_mel, dtype=torch.float16 if half else torch.float32)
    return m(wave.contiguous())


@mel_spectrogram_op.register_fake
def _(wave, sample_rate, n_fft, win_length, hop_length, f_min, f_max, pad, n_mels, power, normalized, center,
      pad_mode, norm, mel_scale, log_mel, half):
    nfr = _op_frames(wave.shape[-1], n_fft, hop_length, pad, center)
    return wave.new_empty((*wave.shape[:-1], n_mels, nfr), dtype=torch.float16 if half else torch.float32)


def _refuse_backward(ctx, inputs, output):
    raise RuntimeError("log_mel_spectrogram_gb300 ops are inference-only: inputs must not require grad "
                       "(use torch.no_grad() or detach())")


def _no_backward(ctx, grad):
    raise RuntimeError("log_mel_spectrogram_gb300 ops have no backward")


log_mel_from_stft_op.register_autograd(_no_backward, setup_context=_refuse_backward)
mel_spectrogram_op.register_autograd(_no_backward, setup_context=_refuse_backward)
