"""Python access to the CPU oracle (``oracle/logmel_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The product package never
imports this module, and this module never imports the product package.

The C source is compiled on demand with gcc (``-O2 -fopenmp``) into
``oracle/_build/liblogmel_oracle.so``; ``build()`` does it explicitly.
"""
from __future__ import annotations

import ctypes
import os
import pathlib
import subprocess
import threading

import numpy as np

_HERE = pathlib.Path(__file__).resolve().parent
_SRC = _HERE / "logmel_oracle.c"
_OUT_DIR = _HERE / "_build"
_LIB_PATH = _OUT_DIR / "liblogmel_oracle.so"
_lock = threading.Lock()
_lib = None

PAD_MODES = {"reflect": 0, "constant": 1, "replicate": 2, "circular": 3}
MEL_SCALES = {"htk": 0, "slaney": 1}


def build(force: bool = False) -> pathlib.Path:
    """Compile the oracle into a shared library (no-op when up to date)."""
    _OUT_DIR.mkdir(exist_ok=True)
    if not force and _LIB_PATH.exists() and _LIB_PATH.stat().st_mtime >= _SRC.stat().st_mtime:
        return _LIB_PATH
    tmp = _LIB_PATH.with_suffix(f".{os.getpid()}.tmp")
    cmd = ["gcc", "-O2", "-std=c11", "-D_DEFAULT_SOURCE", "-fPIC", "-shared", "-fopenmp",
           str(_SRC), "-o", str(tmp), "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(str(path))
            i64, i32, dbl, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
            L.oracle_num_threads.restype = i32
            L.oracle_log_mel_from_stft.argtypes = [vp, vp, i64, i64, i64, i64, vp]
            L.oracle_log_mel_from_stft.restype = i32
            L.oracle_log_mel_from_stft_wrong.argtypes = [vp, vp, i64, i64, i64, i64, i32, i32, vp]
            L.oracle_log_mel_from_stft_wrong.restype = i32
            L.oracle_hz_to_mel.argtypes = [dbl, i32]
            L.oracle_hz_to_mel.restype = dbl
            L.oracle_mel_to_hz.argtypes = [dbl, i32]
            L.oracle_mel_to_hz.restype = dbl
            L.oracle_mel_filterbank.argtypes = [i64, dbl, dbl, i64, dbl, i32, i32, vp]
            L.oracle_mel_filterbank.restype = i32
            L.oracle_hann_window.argtypes = [i64, vp]
            L.oracle_hann_window.restype = i32
            L.oracle_n_frames.argtypes = [i64, i64, i64, i32]
            L.oracle_n_frames.restype = i64
            L.oracle_power_spectrogram.argtypes = [vp, i64, i64, i64, i32, i32, dbl, vp]
            L.oracle_power_spectrogram.restype = i32
            L.oracle_f64_to_f16.argtypes = [dbl]
            L.oracle_f64_to_f16.restype = ctypes.c_uint16
            L.oracle_mel_spectrogram.argtypes = [vp, i32, i64, i64, i64, i64, i64, i64, dbl, dbl,
                                                 i32, i32, dbl, i32, i32, i32, i32, vp]
            L.oracle_mel_spectrogram.restype = i32
            L.oracle_power_spectrogram_ex.argtypes = [vp, i64, i64, i64, i64, i64, i32, i32, i32, dbl, vp]
            L.oracle_power_spectrogram_ex.restype = i32
            L.oracle_mel_spectrogram_ex.argtypes = [vp, i32, i64, i64, i64, i64, i64, i64, i64, i64, dbl, dbl,
                                                    i32, i32, i32, dbl, i32, i32, i32, i32, vp]
            L.oracle_mel_spectrogram_ex.restype = i32
            _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


def num_threads() -> int:
    return int(lib().oracle_num_threads())


def log_mel_from_stft(stft: np.ndarray, mel_filters: np.ndarray) -> np.ndarray:
    """stft [B,F,NF] complex64, mel_filters [NM,NF] f32 -> out [B,F,NM] f32."""
    stft = np.ascontiguousarray(stft, dtype=np.complex64)
    W = np.ascontiguousarray(mel_filters, dtype=np.float32)
    B, F, NF = stft.shape
    NM = W.shape[0]
    assert W.shape == (NM, NF)
    out = np.empty((B, F, NM), dtype=np.float32)
    _check(lib().oracle_log_mel_from_stft(_ptr(stft), _ptr(W), B, F, NF, NM, _ptr(out)),
           "log_mel_from_stft")
    return out


def log_mel_from_stft_wrong(stft: np.ndarray, mel_filters: np.ndarray, scope: str = "clip",
                            bf16_projection: bool = False) -> np.ndarray:
    """A deliberately wrong variant (per-frame / per-batch clamp, bf16 projection)."""
    stft = np.ascontiguousarray(stft, dtype=np.complex64)
    W = np.ascontiguousarray(mel_filters, dtype=np.float32)
    B, F, NF = stft.shape
    NM = W.shape[0]
    out = np.empty((B, F, NM), dtype=np.float32)
    code = {"clip": 0, "frame": 1, "batch": 2}[scope]
    _check(lib().oracle_log_mel_from_stft_wrong(_ptr(stft), _ptr(W), B, F, NF, NM, code,
                                                int(bf16_projection), _ptr(out)), "wrong variant")
    return out


def hz_to_mel(f: float, scale: str) -> float:
    return float(lib().oracle_hz_to_mel(float(f), MEL_SCALES[scale]))


def mel_to_hz(m: float, scale: str) -> float:
    return float(lib().oracle_mel_to_hz(float(m), MEL_SCALES[scale]))


def mel_filterbank(n_freqs: int, f_min: float, f_max: float, n_mels: int, sample_rate: float,
                   scale: str = "htk", norm: str | None = None) -> np.ndarray:
    fb = np.empty((n_mels, n_freqs), dtype=np.float64)
    _check(lib().oracle_mel_filterbank(n_freqs, f_min, f_max, n_mels, float(sample_rate),
                                       MEL_SCALES[scale], int(norm == "slaney"), _ptr(fb)),
           "mel_filterbank")
    return fb


def hann_window(n: int) -> np.ndarray:
    w = np.empty(n, dtype=np.float64)
    _check(lib().oracle_hann_window(n, _ptr(w)), "hann_window")
    return w


def n_frames(T: int, n_fft: int, hop: int, center: bool = True) -> int:
    return int(lib().oracle_n_frames(T, n_fft, hop, int(center)))


def power_spectrogram(x: np.ndarray, n_fft: int, hop: int, center: bool = True,
                      pad_mode: str = "reflect", power: float = 2.0, win_length: int | None = None,
                      pad: int = 0, normalized: bool = False) -> np.ndarray:
    """[n_frames, n_fft/2+1] float64 power spectrogram of one signal."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    nfr = n_frames(x.shape[0] + 2 * pad, n_fft, hop, center)
    spec = np.empty((nfr, n_fft // 2 + 1), dtype=np.float64)
    if win_length is None and pad == 0 and not normalized:
        rc = lib().oracle_power_spectrogram(_ptr(x), x.shape[0], n_fft, hop, int(center), PAD_MODES[pad_mode],
                                            float(power), _ptr(spec))
    else:
        rc = lib().oracle_power_spectrogram_ex(_ptr(x), x.shape[0], n_fft, int(win_length or 0), hop, int(pad),
                                               int(center), PAD_MODES[pad_mode], int(normalized), float(power),
                                               _ptr(spec))
    _check(rc, "power_spectrogram")
    return spec


def f64_to_f16_bits(v: float) -> int:
    return int(lib().oracle_f64_to_f16(float(v)))


def mel_spectrogram(wave: np.ndarray, sample_rate: int, n_fft: int, hop_length: int, n_mels: int,
                    f_min: float = 0.0, f_max: float | None = None, center: bool = True,
                    pad_mode: str = "reflect", power: float = 2.0, mel_scale: str = "htk",
                    norm: str | None = None, log_mel: bool = False,
                    out_dtype: str = "f32", win_length: int | None = None, pad: int = 0,
                    normalized: bool = False) -> np.ndarray:
    """wave [B,T] f32 or i16 -> [B, n_mels, n_frames] f32 or f16."""
    wave = np.ascontiguousarray(wave)
    if wave.dtype == np.int16:
        in_code = 1
    else:
        wave = wave.astype(np.float32, copy=False)
        in_code = 0
    B, T = wave.shape
    if f_max is None:
        f_max = sample_rate / 2.0
    nfr = n_frames(T + 2 * pad, n_fft, hop_length, center)
    if out_dtype == "f16":
        out = np.empty((B, n_mels, nfr), dtype=np.uint16)
        out_code = 2
    else:
        out = np.empty((B, n_mels, nfr), dtype=np.float32)
        out_code = 0
    if win_length is None and pad == 0 and not normalized:
        rc = lib().oracle_mel_spectrogram(_ptr(wave), in_code, B, T, sample_rate, n_fft, hop_length, n_mels,
                                          float(f_min), float(f_max), int(center), PAD_MODES[pad_mode],
                                          float(power), MEL_SCALES[mel_scale], int(norm == "slaney"),
                                          int(log_mel), out_code, _ptr(out))
    else:
        rc = lib().oracle_mel_spectrogram_ex(_ptr(wave), in_code, B, T, sample_rate, n_fft, int(win_length or 0),
                                             hop_length, int(pad), n_mels, float(f_min), float(f_max),
                                             int(center), PAD_MODES[pad_mode], int(normalized), float(power),
                                             MEL_SCALES[mel_scale], int(norm == "slaney"), int(log_mel),
                                             out_code, _ptr(out))
    _check(rc, "mel_spectrogram")
    if out_dtype == "f16":
        return out.view(np.float16)
    return out
