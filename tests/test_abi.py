"""The C-ABI library builds, loads and exports what include/logmel.h declares,
and rejects bad arguments on the host before touching a GPU."""
import ctypes
import pathlib
import re
import subprocess

import pytest

ROOT = pathlib.Path(__file__).resolve().parents[1]
HEADER = ROOT / "include" / "logmel.h"


@pytest.fixture(scope="module")
def L():
    from log_mel_spectrogram_gb300 import build, _native
    build.build()
    return _native.lib()


def declared_functions():
    text = HEADER.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lm_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for must in ("lm_log_mel_from_stft", "lm_log_mel_from_stft_workspace_size", "lm_mel_plan_create",
                 "lm_mel_spectrogram", "lm_mel_plan_destroy", "lm_workspace_error", "lm_status_string"):
        assert must in names


def test_every_declared_symbol_is_exported(L):
    from log_mel_spectrogram_gb300 import build
    out = subprocess.run(["nm", "-D", "--defined-only", str(build.LIB)], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        getattr(L, n)  # resolvable through ctypes too


def test_library_is_built_for_sm_103a():
    from log_mel_spectrogram_gb300 import build
    assert any("compute_103a,code=sm_103a" in a for a in build.ARCH)


def test_status_strings(L):
    for code in range(0, 9):
        s = L.lm_status_string(code)
        assert s and isinstance(s, bytes)
    assert L.lm_status_string(0) == b"LM_OK"
    assert L.lm_version() >= 100


def test_workspace_size(L):
    n = ctypes.c_size_t()
    assert L.lm_log_mel_from_stft_workspace_size(256, 3000, 201, 128, ctypes.byref(n)) == 0
    # header + one u32 per 25-frame tile (120 per clip; 20 consumer warps x 5 frames)
    assert n.value >= 16 + 4 * 256 * 120 and n.value % 256 == 0
    assert L.lm_log_mel_from_stft_workspace_size(-1, 10, 201, 128, ctypes.byref(n)) == 1
    assert L.lm_log_mel_from_stft_workspace_size(2, 10, 201, 600, ctypes.byref(n)) == 2


def _call(L, stft=0x10000, filt=0x20000, out=0x30000000, B=2, F=3, NF=201, NM=80, ws=0x40000, ws_bytes=1 << 20):
    return L.lm_log_mel_from_stft(stft, filt, out, B, F, NF, NM, ws, ws_bytes, None)


def test_argument_validation_needs_no_gpu(L):
    # Every one of these is rejected before any CUDA call (the pointers are
    # never dereferenced), so they run on a machine without a GPU.
    assert _call(L, B=-1) == 1
    assert _call(L, F=-5) == 1
    assert _call(L, NF=0) == 1
    assert _call(L, NM=0) == 1
    assert _call(L, NM=513) == 2
    assert _call(L, NF=9000) == 2
    assert _call(L, stft=0) == 1
    assert _call(L, ws=0) == 7
    assert _call(L, stft=0x10004) == 3      # complex64 source must be 8-byte aligned
    assert _call(L, stft=0x10002) == 3
    assert _call(L, out=0x30000002) == 3
    assert _call(L, ws_bytes=8) == 7
    assert _call(L, out=0x10000 + 64) == 1  # output overlapping the input
    assert _call(L, B=0) == 0               # nothing to do
    assert _call(L, F=0) == 0


def test_mel_plan_validation(L):
    from log_mel_spectrogram_gb300 import _native
    plan = ctypes.c_void_p()
    assert L.lm_mel_plan_create(None, ctypes.byref(plan)) == 1
    p = _native.MelParams(sample_rate=16000, n_fft=400, hop_length=160, n_mels=128, f_max=8000.0, center=1,
                          power=2.0)
    assert L.lm_mel_plan_create(ctypes.byref(p), None) == 1


def test_filter_pack_validation_needs_no_gpu(L):
    n = ctypes.c_size_t()
    assert L.lm_mel_filters_pack_size(201, 128, ctypes.byref(n)) == 0
    # header, {first, width} per band (padded to 16 bytes), 8 weights per band
    assert n.value == 16 + 1024 + 32 * 128 and n.value % 16 == 0
    assert L.lm_mel_filters_pack_size(201, 81, ctypes.byref(n)) == 0
    assert n.value == 16 + 656 + 32 * 81
    assert L.lm_mel_filters_pack_size(0, 80, ctypes.byref(n)) == 1
    assert L.lm_mel_filters_pack_size(201, 600, ctypes.byref(n)) == 2
    assert L.lm_mel_filters_pack(None, 201, 80, 0x10000, 1 << 20, None) == 1
    assert L.lm_mel_filters_pack(0x20000, 201, 80, 0x10008, 1 << 20, None) == 3   # pack not 16-byte aligned
    assert L.lm_mel_filters_pack(0x20000, 201, 80, 0x10000, 64, None) == 7        # pack too small
    # the packed call validates like the dense one, plus a null or misaligned pack
    assert L.lm_log_mel_from_stft_packed(0x10000, 0x20000, None, 0x30000000, 2, 3, 201, 80, 0x40000, 1 << 20,
                                         None) == 1
    assert L.lm_log_mel_from_stft_packed(0x10000, 0x20000, 0x50008, 0x30000000, 2, 3, 201, 80, 0x40000,
                                         1 << 20, None) == 3


def _host_ws(L, B, F, NF, NM, chunk=0):
    n = ctypes.c_size_t()
    st = L.lm_log_mel_from_stft_host_workspace_size(B, F, NF, NM, chunk, ctypes.byref(n))
    return st, n.value


def test_host_pipeline_workspace_size(L):
    # default chunk: whole clips filling about 32 MB of input, here 6 Whisper clips
    in_clip, out_clip = 3000 * 201 * 8, 3000 * 128 * 4
    st, n = _host_ws(L, 256, 3000, 201, 128)
    assert st == 0 and n % 256 == 0
    assert n >= 3 * 6 * (in_clip + out_clip) and n < 3 * 7 * (in_clip + out_clip)
    st, n1 = _host_ws(L, 256, 3000, 201, 128, 1)
    assert st == 0 and 3 * (in_clip + out_clip) <= n1 < n
    st, nb = _host_ws(L, 2, 3000, 201, 128, 64)   # a chunk never exceeds the batch
    assert st == 0 and nb < n
    # a small batch runs in at least three chunks: 8 clips -> 3 per chunk
    st, n8 = _host_ws(L, 8, 3000, 201, 128)
    _, n3 = _host_ws(L, 8, 3000, 201, 128, 3)
    assert st == 0 and n8 == n3
    assert _host_ws(L, -1, 10, 201, 128)[0] == 1
    assert _host_ws(L, 2, 10, 201, 128, -1)[0] == 1
    assert _host_ws(L, 2, 10, 201, 600)[0] == 2
    assert L.lm_log_mel_from_stft_host_workspace_size(2, 10, 201, 128, 0, None) == 1
    n = ctypes.c_size_t()
    assert L.lm_mel_spectrogram_host_workspace_size(None, 2, 1000, 0, 0, 0, ctypes.byref(n)) == 1


def _host_call(L, stft=0x10000, filt=0x20000, packed=None, out=0x30000000, B=2, F=3, NF=201, NM=80, chunk=0,
               ws=0x40000, ws_bytes=1 << 26):
    return L.lm_log_mel_from_stft_host(stft, filt, packed, out, B, F, NF, NM, chunk, ws, ws_bytes, None)


def test_host_pipeline_validation_needs_no_gpu(L):
    # rejected before any CUDA call: the pointers are never dereferenced
    assert _host_call(L, B=-1) == 1
    assert _host_call(L, NM=600) == 2
    assert _host_call(L, chunk=-2) == 1
    assert _host_call(L, stft=0) == 1
    assert _host_call(L, out=0) == 1
    assert _host_call(L, ws=0) == 7
    assert _host_call(L, ws=0x40010) == 3        # workspace must be 256-byte aligned
    assert _host_call(L, filt=0x20002) == 3
    assert _host_call(L, packed=0x50008) == 3
    assert _host_call(L, ws_bytes=1024) == 7
    assert _host_call(L, out=0x10000 + 8) == 1   # host output overlapping the host input
    assert _host_call(L, B=0) == 0
    assert _host_call(L, F=0) == 0
    assert L.lm_mel_spectrogram_host(None, 0x10000, 0, 2, 1000, 0x30000000, 0, 0, 0x40000, 1 << 26, None) == 1


def test_eight_byte_aligned_source_passes_validation(L):
    # A complex64 view one element into its allocation is 8 bytes off a
    # 16-byte boundary: validation accepts it, and without a GPU the call
    # then stops at the first CUDA call (LM_ERR_CUDA), never at alignment.
    assert _call(L, stft=0x10008) not in (1, 3, 7)


def test_fault_injection_entry_validation_needs_no_gpu(L):
    f = L.lm_debug_log_mel_from_stft_withhold
    args = (0x10000, 0x20000, 0x30000000, 2, 3, 201, 80, 0x40000, 1 << 20)
    assert f(*args, -1, 1000000, None) == 1            # no tile to withhold
    assert f(*args, 0, 10, None) == 1                  # wait limit below 100 us
    assert f(*args, 0, 10 ** 10, None) == 1            # above the regular 2 s
    assert f(0x10004, *args[1:], 0, 1000000, None) == 3  # validated like the regular call
    assert f(*args[:3], -1, 3, 201, 80, 0x40000, 1 << 20, 0, 1000000, None) == 1


def test_noalloc_validation_needs_no_gpu(L):
    assert L.lm_log_mel_from_stft_noalloc(None, None, None, -1, 10, 201, 80, None) == 1
    assert L.lm_log_mel_from_stft_noalloc(None, None, None, 2, 10, 201, 600, None) == 2
    assert L.lm_log_mel_from_stft_noalloc(None, None, None, 0, 10, 201, 80, None) == 0
    # larger than the scratch the library holds: refused before any pointer is used
    assert L.lm_log_mel_from_stft_noalloc(None, None, None, 512, 20000, 201, 128, None) == 7
    assert L.lm_log_mel_from_stft_noalloc_error(None, 0, None) == 1


def test_forced_plan_allocation_failure_needs_no_gpu(L, monkeypatch):
    # LOGMEL_FAULT=plan_alloc: the plan's first device allocation fails as if
    # the device were out of memory, before any CUDA call is made for it.
    from log_mel_spectrogram_gb300 import _native
    p = _native.MelParams(sample_rate=16000, n_fft=400, hop_length=160, n_mels=128, f_max=8000.0, center=1,
                          power=2.0)
    plan = ctypes.c_void_p(1234)
    monkeypatch.setenv("LOGMEL_FAULT", "plan_alloc")
    assert L.lm_mel_plan_create(ctypes.byref(p), ctypes.byref(plan)) == 5   # LM_ERR_OUT_OF_MEMORY
    assert plan.value is None
    monkeypatch.setenv("LOGMEL_FAULT", "plan_alloc:1")
    assert L.lm_mel_plan_create(ctypes.byref(p), ctypes.byref(plan)) == 5
    # invalid parameters are still reported first
    bad = _native.MelParams(sample_rate=16000, n_fft=401, hop_length=160, n_mels=128, center=1, power=2.0)
    assert L.lm_mel_plan_create(ctypes.byref(bad), ctypes.byref(plan)) == 2
