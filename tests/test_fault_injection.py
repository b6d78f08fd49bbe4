"""A bounded wait that runs out ends the kernel cleanly.

lm_debug_log_mel_from_stft_withhold keeps one tile's maximum from ever being
published, so the CTAs that wait for that clip's maximum give up after a
short limit instead of the regular 2 s.  The checks: the call completes, the
workspace's device error word carries the clip-timeout bit, clips that no
aborting CTA touched are still exact, and the next regular call on the same
GPU is exact again (the context stayed usable).  Nothing here faults, traps
or hangs the GPU: the only failure is a wait that nothing completes.
"""
import ctypes
import time

import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

ATOL = RTOL = 1e-4
CLIP_TIMEOUT_BIT = 2
LM_ERR_DEVICE_FAULT = 6


@pytest.fixture(scope="module")
def lm():
    import __graft_entry__
    __graft_entry__.build()
    import log_mel_spectrogram_gb300
    return log_mel_spectrogram_gb300


def _close(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return np.all(np.abs(got - ref) <= ATOL + RTOL * np.abs(ref))


def _withhold(lm, stft, W, out, ws, tile, wait_ns):
    from log_mel_spectrogram_gb300 import _native
    B, F, NF = stft.shape
    NM = W.shape[0]
    rc = _native.lib().lm_debug_log_mel_from_stft_withhold(
        stft.data_ptr(), W.data_ptr(), out.data_ptr(), B, F, NF, NM, ws.data_ptr(), ws.numel(), tile, wait_ns,
        torch.cuda.current_stream().cuda_stream)
    assert rc == 0


@pytest.mark.parametrize("shape,tile", [((4, 600, 201, 128), 30), ((8, 3000, 201, 80), 500)], ids=str)
def test_withheld_tile_times_out_and_reports(lm, oracle_mod, shape, tile, monkeypatch):
    # the fault entry runs the one-CTA-per-SM kernel; describe that one
    monkeypatch.setenv("LOGMEL_K1_VARIANT", "resident")
    B, F, NF, NM = shape
    info = lm.describe_log_mel_from_stft(B, F, NF, NM)
    assert info["resident"] == 1
    tpc = -(-F // info["frames_per_tile"])
    stft, W = workloads.stft_inputs(B, F, NF, NM, seed=400 + B)
    s, w = stft.cuda(), W.cuda()
    ref = oracle_mod.log_mel_from_stft(stft.numpy(), W.numpy())
    ws = torch.empty(lm.log_mel_from_stft_workspace_size(B, F, NF, NM), dtype=torch.uint8, device="cuda")
    out = torch.zeros(B, F, NM, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    _withhold(lm, s, w, out, ws, tile, 2_000_000)  # 2 ms limit
    err = lm.workspace_error(ws)                   # synchronises
    elapsed = time.perf_counter() - t0
    assert err & CLIP_TIMEOUT_BIT, err
    assert elapsed < 1.5, elapsed                  # gave up long before the regular 2 s
    v = ctypes.c_uint32()
    from log_mel_spectrogram_gb300 import _native
    assert _native.lib().lm_workspace_error(ws.data_ptr(), ws.numel(), ctypes.byref(v), None) == LM_ERR_DEVICE_FAULT
    got = out.cpu().numpy()
    if B * tpc <= info["grid"]:
        # one tile per CTA: only the CTAs of the withheld tile's clip gave up
        bad_clip = tile // tpc
        for b in range(B):
            if b != bad_clip:
                assert _close(got[b], ref[b]), b
    # the GPU is still fine: a regular call on the same workspace is exact
    out2 = lm.log_mel_from_stft(s, w, workspace=ws)
    assert lm.workspace_error(ws) == 0
    assert _close(out2.cpu().numpy(), ref)


@pytest.mark.parametrize("n_fft,k", [(400, 1), (400, 3), (400, 7), (16384, 7)])
def test_forced_plan_allocation_failure_frees_what_was_allocated(lm, monkeypatch, n_fft, k):
    # LOGMEL_FAULT=plan_alloc:k fails the k-th device allocation of a plan:
    # the call reports LM_ERR_OUT_OF_MEMORY and frees the k - 1 before it.
    # (At 400 points the 7th is the shared-memory table image; at 16384 it
    # is the filterbank image of the in-place kernel.)
    from log_mel_spectrogram_gb300 import _native
    p = _native.MelParams(sample_rate=16000, n_fft=n_fft, hop_length=n_fft // 4, n_mels=128, f_max=8000.0,
                          center=1, power=2.0)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    monkeypatch.setenv("LOGMEL_FAULT", f"plan_alloc:{k}")
    plan = ctypes.c_void_p(1234)
    for _ in range(50):
        assert _native.lib().lm_mel_plan_create(ctypes.byref(p), ctypes.byref(plan)) == 5
        assert plan.value is None
    free1, _ = torch.cuda.mem_get_info()
    assert free0 - free1 < 2 ** 21  # nothing left behind by 50 failed creations
    monkeypatch.delenv("LOGMEL_FAULT")
    m = lm.MelSpectrogram(sample_rate=16000, n_fft=400, hop_length=160, n_mels=128, f_max=8000.0)
    x = workloads.wave_sines(1, 8000, 16000, seed=1, device="cuda")
    assert m(x).shape == (1, 128, 51)
    m.close()
