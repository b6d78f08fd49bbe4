"""The allocation-free entry point, lm_log_mel_from_stft_noalloc.

Some callers cannot allocate device memory: a real-time audio thread where
cudaMalloc may block or synchronise the device, or an application that owns
all device memory.  This entry point runs the same kernel with its scratch in
a fixed array inside the library.  These checks call it through the C ABI on
calls in a row with different shapes: a large one, a smaller one (whose clip
maxima would read the larger call's leftover tile slots if the scratch were
not cleared), then the large one again.  Each result is compared with the
CPU oracle at the f32 gate and, bit for bit, with the regular entry point
(which takes a caller workspace).  The sticky error word must read zero.

The file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

ATOL = RTOL = 1e-4
LM_ERR_WORKSPACE = 7


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build()
    from log_mel_spectrogram_gb300 import _native
    return _native.lib()


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _regular(L, stft, W):
    B, F, NF = stft.shape
    NM = W.shape[0]
    n = ctypes.c_size_t()
    assert L.lm_log_mel_from_stft_workspace_size(B, F, NF, NM, ctypes.byref(n)) == 0
    ws = torch.empty(n.value, dtype=torch.uint8, device="cuda")
    out = torch.empty((B, F, NM), dtype=torch.float32, device="cuda")
    rc = L.lm_log_mel_from_stft(stft.data_ptr(), W.data_ptr(), out.data_ptr(), B, F, NF, NM, ws.data_ptr(),
                                n.value, _stream())
    assert rc == 0
    return out


def _noalloc(L, stft, W):
    B, F, NF = stft.shape
    NM = W.shape[0]
    out = torch.empty((B, F, NM), dtype=torch.float32, device="cuda")
    rc = L.lm_log_mel_from_stft_noalloc(stft.data_ptr(), W.data_ptr(), out.data_ptr(), B, F, NF, NM, _stream())
    assert rc == 0
    return out


def _error_word(L, clear=1):
    v = ctypes.c_uint32(0xffffffff)
    rc = L.lm_log_mel_from_stft_noalloc_error(ctypes.byref(v), clear, _stream())
    assert rc == (0 if v.value == 0 else 6)
    return v.value


def test_noalloc_matches_oracle_and_regular_on_calls_in_a_row(L, oracle_mod):
    cases = (((7, 777, 201, 128), 32), ((3, 301, 201, 80), 31), ((7, 777, 201, 128), 33))
    for (B, F, NF, NM), seed in cases:
        stft, W = workloads.stft_inputs(B, F, NF, NM, seed=seed)
        stft[1, F // 2:] *= 1e-6  # make the clip floor matter
        s, w = stft.cuda(), W.cuda()
        got = _noalloc(L, s, w)
        ref_dev = _regular(L, s, w)
        torch.cuda.synchronize()
        assert _error_word(L) == 0
        ref = oracle_mod.log_mel_from_stft(stft.numpy(), W.numpy()).astype(np.float64)
        g = got.cpu().numpy().astype(np.float64)
        assert np.all(np.abs(g - ref) <= ATOL + RTOL * np.abs(ref)), (B, F, NF, NM)
        assert torch.equal(got, ref_dev)


def test_noalloc_rejects_problems_larger_than_its_scratch(L):
    # 512 clips x 20000 frames needs far more than the fixed scratch; the
    # call must refuse before touching any pointer (all are null here).
    rc = L.lm_log_mel_from_stft_noalloc(None, None, None, 512, 20000, 201, 128, None)
    assert rc == LM_ERR_WORKSPACE
