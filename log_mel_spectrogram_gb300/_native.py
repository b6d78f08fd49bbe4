"""ctypes view of liblogmel.so (declarations mirror include/logmel.h).

Loading fails loudly when the library has not been built: there is no
fallback implementation of any operation.
"""
from __future__ import annotations

import ctypes
import pathlib
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

LM_OK = 0
STATUS_NAMES = {0: "LM_OK", 1: "LM_ERR_INVALID_ARG", 2: "LM_ERR_UNSUPPORTED", 3: "LM_ERR_MISALIGNED",
                4: "LM_ERR_CUDA", 5: "LM_ERR_OUT_OF_MEMORY", 6: "LM_ERR_DEVICE_FAULT", 7: "LM_ERR_WORKSPACE"}
DTYPES = {"f32": 0, "i16": 1, "f16": 2}
PAD_MODES = {"reflect": 0, "constant": 1, "replicate": 2, "circular": 3}
MEL_SCALES = {"htk": 0, "slaney": 1}


class LogmelError(RuntimeError):
    def __init__(self, status: int, what: str, cuda_error: int = 0):
        self.status = status
        self.cuda_error = cuda_error
        msg = f"{what}: {STATUS_NAMES.get(status, status)}"
        if cuda_error:
            msg += f" (cudaError {cuda_error})"
        super().__init__(msg)


class StftLaunchInfo(ctypes.Structure):
    _fields_ = [("resident", ctypes.c_int32), ("kernels", ctypes.c_int32), ("grid", ctypes.c_int32),
                ("frames_per_tile", ctypes.c_int32), ("stages", ctypes.c_int32), ("lag", ctypes.c_int32),
                ("smem_bytes", ctypes.c_int64), ("cluster", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class MelParams(ctypes.Structure):
    _fields_ = [("sample_rate", ctypes.c_int32), ("n_fft", ctypes.c_int32), ("win_length", ctypes.c_int32),
                ("hop_length", ctypes.c_int32), ("n_mels", ctypes.c_int32), ("f_min", ctypes.c_float),
                ("f_max", ctypes.c_float), ("pad", ctypes.c_int32), ("center", ctypes.c_int32),
                ("pad_mode", ctypes.c_int32), ("power", ctypes.c_float), ("normalized", ctypes.c_int32),
                ("mel_scale", ctypes.c_int32), ("slaney_norm", ctypes.c_int32), ("log_mel", ctypes.c_int32)]


def library_path() -> pathlib.Path:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """The loaded library.  Raises if liblogmel.so is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if not path.exists():
            raise RuntimeError(f"liblogmel.so is not built ({path}); run __graft_entry__.build() "
                               "or python -m log_mel_spectrogram_gb300.build")
        _lib = _declare(ctypes.CDLL(str(path)))
        return _lib


def _declare(L: ctypes.CDLL) -> ctypes.CDLL:
    """Argument and result types of every entry point (include/logmel.h)."""
    i64, i32, u32, sz, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32, ctypes.c_size_t, ctypes.c_void_p
    L.lm_status_string.argtypes = [ctypes.c_int]
    L.lm_status_string.restype = ctypes.c_char_p
    L.lm_last_cuda_error.restype = ctypes.c_int
    L.lm_version.restype = ctypes.c_int
    L.lm_log_mel_from_stft_workspace_size.argtypes = [i64, i64, i32, i32, ctypes.POINTER(sz)]
    L.lm_log_mel_from_stft_workspace_size.restype = ctypes.c_int
    L.lm_log_mel_from_stft.argtypes = [vp, vp, vp, i64, i64, i32, i32, vp, sz, vp]
    L.lm_log_mel_from_stft.restype = ctypes.c_int
    L.lm_log_mel_from_stft_describe.argtypes = [i64, i64, i32, i32, ctypes.POINTER(StftLaunchInfo)]
    L.lm_log_mel_from_stft_describe.restype = ctypes.c_int
    L.lm_mel_filters_pack_size.argtypes = [i32, i32, ctypes.POINTER(sz)]
    L.lm_mel_filters_pack_size.restype = ctypes.c_int
    L.lm_mel_filters_pack.argtypes = [vp, i32, i32, vp, sz, vp]
    L.lm_mel_filters_pack.restype = ctypes.c_int
    L.lm_log_mel_from_stft_packed.argtypes = [vp, vp, vp, vp, i64, i64, i32, i32, vp, sz, vp]
    L.lm_log_mel_from_stft_packed.restype = ctypes.c_int
    L.lm_workspace_error.argtypes = [vp, sz, ctypes.POINTER(u32), vp]
    L.lm_workspace_error.restype = ctypes.c_int
    L.lm_log_mel_from_stft_noalloc.argtypes = [vp, vp, vp, i64, i64, i32, i32, vp]
    L.lm_log_mel_from_stft_noalloc.restype = ctypes.c_int
    L.lm_log_mel_from_stft_noalloc_error.argtypes = [ctypes.POINTER(u32), i32, vp]
    L.lm_log_mel_from_stft_noalloc_error.restype = ctypes.c_int
    L.lm_debug_log_mel_from_stft_withhold.argtypes = [vp, vp, vp, i64, i64, i32, i32, vp, sz, i64,
                                                      ctypes.c_uint64, vp]
    L.lm_debug_log_mel_from_stft_withhold.restype = ctypes.c_int
    L.lm_mel_plan_create.argtypes = [ctypes.POINTER(MelParams), ctypes.POINTER(vp)]
    L.lm_mel_plan_create.restype = ctypes.c_int
    L.lm_mel_plan_destroy.argtypes = [vp]
    L.lm_mel_plan_destroy.restype = ctypes.c_int
    L.lm_mel_n_frames.argtypes = [vp, i64, ctypes.POINTER(i64)]
    L.lm_mel_n_frames.restype = ctypes.c_int
    L.lm_mel_workspace_size.argtypes = [vp, i64, i64, ctypes.POINTER(sz)]
    L.lm_mel_workspace_size.restype = ctypes.c_int
    L.lm_mel_spectrogram.argtypes = [vp, vp, i32, i64, i64, vp, i32, vp, sz, vp]
    L.lm_mel_spectrogram.restype = ctypes.c_int
    L.lm_log_mel_from_stft_host_workspace_size.argtypes = [i64, i64, i32, i32, i64, ctypes.POINTER(sz)]
    L.lm_log_mel_from_stft_host_workspace_size.restype = ctypes.c_int
    L.lm_log_mel_from_stft_host.argtypes = [vp, vp, vp, vp, i64, i64, i32, i32, i64, vp, sz, vp]
    L.lm_log_mel_from_stft_host.restype = ctypes.c_int
    L.lm_mel_spectrogram_host_workspace_size.argtypes = [vp, i64, i64, i32, i32, i64, ctypes.POINTER(sz)]
    L.lm_mel_spectrogram_host_workspace_size.restype = ctypes.c_int
    L.lm_mel_spectrogram_host.argtypes = [vp, vp, i32, i64, i64, vp, i32, i64, vp, sz, vp]
    L.lm_mel_spectrogram_host.restype = ctypes.c_int
    return L


_checked = None


def checked_lib() -> ctypes.CDLL:
    """The bounds-checked debug variant (-DLOGMEL_CHECKED): every computed
    global-memory index is tested against its buffer, and one outside sets
    bit 8 of the error word and skips the access.  Built on first use."""
    global _checked
    with _lock:
        if _checked is None:
            _checked = _declare(ctypes.CDLL(str(_build.build(checked=True))))
        return _checked


def check(status: int, what: str) -> None:
    if status != LM_OK:
        raise LogmelError(status, what, lib().lm_last_cuda_error() if status == 4 else 0)
