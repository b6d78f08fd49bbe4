"""The bounds-checked debug build (-DLOGMEL_CHECKED).

compute-sanitizer is not available on the GPU pool, so the library has a
debug variant in which every computed global-memory index of the kernels (bulk
copy ranges, sample loads, output and slot stores, clip words) is tested
against its buffer: an index outside sets bit 8 of the device error word and
the access is skipped.  These tests run the main code paths through that
variant on ragged and edge shapes, through the C ABI, and require the error
word to stay 0 and the results to match the regular library's: bit for bit on
the STFT path and the generic waveform kernel, and within 1e-5 (2e-3 for f16
output) on the register kernels, whose code the checks' extra branches and
register pressure change (the compiler contracts some products into FMAs
differently).
"""
import ctypes

import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

LM_ERR_BOUNDS_BIT = 8


@pytest.fixture(scope="module")
def libs():
    import __graft_entry__
    __graft_entry__.build()
    from log_mel_spectrogram_gb300 import _native
    return _native.lib(), _native.checked_lib()


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _error_word(L, ws):
    v = ctypes.c_uint32(0xffffffff)
    L.lm_workspace_error(ws.data_ptr(), ws.numel(), ctypes.byref(v), _stream())
    return v.value


def _stft_call(L, stft, W, ws_offset=0):
    B, F, NF = stft.shape
    NM = W.shape[0]
    n = ctypes.c_size_t()
    assert L.lm_log_mel_from_stft_workspace_size(B, F, NF, NM, ctypes.byref(n)) == 0
    raw = torch.empty(n.value + 256, dtype=torch.uint8, device="cuda")
    ws = raw[ws_offset:ws_offset + n.value]
    out = torch.empty((B, F, NM), dtype=torch.float32, device="cuda")
    rc = L.lm_log_mel_from_stft(stft.data_ptr(), W.data_ptr(), out.data_ptr(), B, F, NF, NM, ws.data_ptr(),
                                n.value, _stream())
    assert rc == 0
    return out, _error_word(L, ws)


@pytest.mark.parametrize("variant", ["auto", "resident", "twopass", "cluster"])
@pytest.mark.parametrize("shape", [(3, 301, 201, 128), (7, 97, 129, 80), (8, 3000, 201, 80), (2, 5, 1, 1)])
def test_stft_paths_stay_in_bounds(libs, variant, shape, monkeypatch):
    reg, chk = libs
    monkeypatch.setenv("LOGMEL_K1_VARIANT", variant)
    B, F, NF, NM = shape
    stft, W = workloads.stft_inputs(B, F, NF, NM, seed=sum(shape))
    big = torch.view_as_real(stft).cuda().reshape(-1)
    # an 8-byte-aligned view (the tensor starts 8 bytes past a 16-byte boundary)
    src = torch.empty(big.numel() + 2, dtype=torch.float32, device="cuda")
    src[2:] = big
    view = torch.view_as_complex(src[2:].view(B, F, NF, 2))
    W = W.cuda()
    try:
        got, err = _stft_call(chk, view, W, ws_offset=0)
    except AssertionError:
        pytest.skip(f"variant {variant} does not take shape {shape}")
    ref, _ = _stft_call(reg, view, W)
    assert err == 0, f"error word {err:#x}"
    assert torch.equal(got, ref)


def _mel_call(L, params, wave, dtype_code_in, dtype_out, T):
    handle = ctypes.c_void_p()
    assert L.lm_mel_plan_create(ctypes.byref(params), ctypes.byref(handle)) == 0
    try:
        nfr = ctypes.c_int64()
        assert L.lm_mel_n_frames(handle, T, ctypes.byref(nfr)) == 0
        B = wave.shape[0]
        need = ctypes.c_size_t()
        assert L.lm_mel_workspace_size(handle, B, T, ctypes.byref(need)) == 0
        ws = torch.empty(max(need.value, 16), dtype=torch.uint8, device="cuda")
        out = torch.empty((B, params.n_mels, nfr.value), dtype=dtype_out, device="cuda")
        out_code = 2 if dtype_out == torch.float16 else 0
        rc = L.lm_mel_spectrogram(handle, wave.data_ptr(), dtype_code_in, B, T, out.data_ptr(), out_code,
                                  ws.data_ptr(), ws.numel(), _stream())
        assert rc == 0
        return out, _error_word(L, ws)
    finally:
        L.lm_mel_plan_destroy(handle)


@pytest.mark.parametrize("n_fft,hop,pad_mode,center,log_mel,i16,f16,epilogue", [
    (400, 160, "reflect", True, True, False, False, "separate"),   # register kernel, two launches
    (400, 160, "reflect", True, True, False, False, "fused"),      # register kernel, one launch
    (1024, 256, "reflect", True, False, True, True, "separate"),   # register kernel, i16 in, f16 out
    (256, 64, "constant", True, True, False, False, "fused"),      # register kernel, edge index pass
    (512, 128, "circular", True, False, True, False, "separate"),
    (64, 16, "replicate", False, False, False, False, "separate"),
    (2048, 512, "reflect", True, True, False, False, "separate"),  # generic kernel, staged spans
    (8192, 2048, "reflect", True, False, True, True, "separate"),  # generic kernel, in place
])
def test_waveform_paths_stay_in_bounds(libs, n_fft, hop, pad_mode, center, log_mel, i16, f16, epilogue,
                                       monkeypatch):
    import log_mel_spectrogram_gb300 as lm
    reg, chk = libs
    monkeypatch.setenv("LOGMEL_K3_EPILOGUE", epilogue)
    T = 3 * n_fft + 333
    m = lm.MelSpectrogram(sample_rate=16000, n_fft=n_fft, hop_length=hop, n_mels=64, f_max=8000.0,
                          pad_mode=pad_mode, center=center, log_mel=log_mel,
                          dtype=torch.float16 if f16 else torch.float32)
    x = (workloads.wave_pcm16(3, T, seed=n_fft) if i16 else workloads.wave_sines(3, T, 16000, seed=n_fft)).cuda()
    code_in = 1 if i16 else 0
    got, err = _mel_call(chk, m.params, x, code_in, torch.float16 if f16 else torch.float32, T)
    ref, _ = _mel_call(reg, m.params, x, code_in, torch.float16 if f16 else torch.float32, T)
    m.close()
    assert err == 0, f"error word {err:#x}"
    tol = 2e-3 if f16 else 1e-5
    g, r = got.double(), ref.double()
    assert torch.all((g - r).abs() <= tol + tol * r.abs()), float((g - r).abs().max())
    if n_fft > 1024:
        assert torch.equal(got, ref)  # the generic kernel: the same bits
