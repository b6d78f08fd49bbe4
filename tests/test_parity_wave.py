"""GPU parity of the waveform -> mel spectrogram path against the CPU oracle.

Gates: f32 output |gpu - oracle| <= 1e-4 + 1e-4 |oracle|; f16 output is
compared with the oracle rounded to f16, |gpu - ref16| <= 2e-3 + 2e-3 |ref16|.
Inputs come from workloads.py and are identical on both sides.
"""
import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lm():
    import __graft_entry__
    __graft_entry__.build()
    import log_mel_spectrogram_gb300
    return log_mel_spectrogram_gb300


def _gate(got, ref, tol):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    err = np.abs(got - ref)
    bad = err > tol + tol * np.abs(ref)
    assert not bad.any(), (f"{bad.sum()} of {bad.size} outside tolerance; max err {err.max():.3g} at "
                           f"{np.unravel_index(np.argmax(err), err.shape)}")


def _run(lm, oracle_mod, wave, sample_rate, n_fft, hop, n_mels, f_min=0.0, f_max=None, center=True,
         pad_mode="reflect", power=2.0, mel_scale="htk", norm=None, log_mel=False, out_dtype="f32",
         win_length=None, pad=0, normalized=False):
    m = lm.MelSpectrogram(sample_rate=sample_rate, n_fft=n_fft, hop_length=hop, n_mels=n_mels, f_min=f_min,
                          f_max=f_max, center=center, pad_mode=pad_mode, power=power, mel_scale=mel_scale,
                          norm=norm, log_mel=log_mel, win_length=win_length, pad=pad, normalized=normalized,
                          dtype=torch.float16 if out_dtype == "f16" else torch.float32)
    got = m(wave.cuda())
    torch.cuda.synchronize()
    ref = oracle_mod.mel_spectrogram(wave.numpy(), sample_rate, n_fft, hop, n_mels, f_min=f_min, f_max=f_max,
                                     center=center, pad_mode=pad_mode, power=power, mel_scale=mel_scale,
                                     norm=norm, log_mel=log_mel, out_dtype=out_dtype, win_length=win_length,
                                     pad=pad, normalized=normalized)
    m.close()
    tol = 2e-3 if out_dtype == "f16" else 1e-4
    _gate(got.float().cpu().numpy(), ref.astype(np.float64), tol)
    return got


def test_whisper_sines_small(lm, oracle_mod):
    w = workloads.WAVE_WHISPER
    x = workloads.wave_workload_inputs(w, B=2, T=16000 * 3)
    _run(lm, oracle_mod, x, 16000, 400, 160, 128, f_max=8000.0, log_mel=True)
    _run(lm, oracle_mod, x, 16000, 400, 160, 128, f_max=8000.0, log_mel=False)


def test_pcm16_slaney_small(lm, oracle_mod):
    w = workloads.WAVE_PCM16
    x = workloads.wave_workload_inputs(w, B=3, T=22050)
    _run(lm, oracle_mod, x, 22050, 1024, 256, 128, f_max=11025.0, mel_scale="slaney", out_dtype="f16")
    _run(lm, oracle_mod, x, 22050, 1024, 256, 128, f_max=11025.0, mel_scale="slaney", out_dtype="f32")


@pytest.mark.parametrize("n_fft", [64, 128, 256, 512, 2048, 4096])
def test_power_of_two_sizes(lm, oracle_mod, n_fft):
    x = workloads.wave_sines(2, max(4 * n_fft, 3000), 16000, seed=n_fft)
    _run(lm, oracle_mod, x, 16000, n_fft, n_fft // 4, 40 if n_fft <= 128 else 80, f_max=8000.0)


@pytest.mark.parametrize("n_fft", [8192, 16384])
def test_large_fft_sizes(lm, oracle_mod, n_fft):
    # Past 4096 points the transform runs in place, one frame per tile: the
    # window and untangle twiddles are read from global memory, interior
    # frames load aligned sample pairs directly (clip 1 of an odd T starts
    # unaligned and gathers), and the filterbank image is copied into the
    # transform's buffer for the projection where it fits (128 and 80 bands;
    # 256 bands at 8192 points do not fit and read the global tables).  Seven
    # frames a clip keep the oracle's direct DFT to a few seconds.
    T = 3 * n_fft + 77
    x = workloads.wave_sines(2, T, 22050, seed=n_fft)
    _run(lm, oracle_mod, x, 22050, n_fft, n_fft // 2, 128, f_max=11025.0, mel_scale="slaney", norm="slaney")
    _run(lm, oracle_mod, x, 22050, n_fft, n_fft // 2, 80, f_max=8000.0, log_mel=True)
    xi = workloads.wave_pcm16(2, T, seed=n_fft + 1)
    _run(lm, oracle_mod, xi, 16000, n_fft, n_fft // 2, 256, f_max=8000.0, out_dtype="f16")


@pytest.mark.parametrize("pad_mode", ["reflect", "constant", "replicate", "circular"])
def test_pad_modes(lm, oracle_mod, pad_mode):
    x = workloads.wave_sines(2, 3333, 16000, seed=7)
    _run(lm, oracle_mod, x, 16000, 400, 160, 64, f_max=8000.0, pad_mode=pad_mode)


def test_center_false_power_one_norm_fmin(lm, oracle_mod):
    x = workloads.wave_sines(3, 5000, 16000, seed=9)
    _run(lm, oracle_mod, x, 16000, 400, 100, 80, f_min=60.0, f_max=7600.0, center=False, power=1.0)
    _run(lm, oracle_mod, x, 16000, 512, 128, 96, mel_scale="slaney", norm="slaney")
    _run(lm, oracle_mod, x, 16000, 256, 37, 256, f_max=8000.0)  # odd hop, 256 bands


def test_short_and_ragged_signals(lm, oracle_mod):
    # T just above n_fft / 2 (the least reflect padding allows): one or two frames
    x = workloads.wave_sines(2, 201, 16000, seed=3)
    _run(lm, oracle_mod, x, 16000, 400, 160, 40, f_max=8000.0)
    x = workloads.wave_pcm16(1, 700, seed=4)
    _run(lm, oracle_mod, x, 22050, 1024, 256, 64, mel_scale="slaney", log_mel=True)


def test_silence_and_log_window(lm, oracle_mod):
    x = workloads.wave_sines(3, 8000, 16000, seed=5)
    x[1] = 0.0
    x[2, 4000:] *= 1e-6
    got = _run(lm, oracle_mod, x, 16000, 400, 160, 128, f_max=8000.0, log_mel=True).cpu()
    assert torch.all(got[1] == -1.5)
    mx = got.amax(dim=(1, 2))
    assert torch.all(got.amin(dim=(1, 2)) >= mx - 2.0 - 1e-5)


def test_whisper_full_size_every_clip(lm, oracle_mod):
    # 8 x 480000 f32, n_fft 400, hop 160, 128 HTK bands, log: the whole batch
    # on the GPU and in the oracle.
    w = workloads.WAVE_WHISPER
    x = workloads.wave_workload_inputs(w)
    m = lm.MelSpectrogram(sample_rate=16000, n_fft=400, hop_length=160, n_mels=128, f_max=8000.0, log_mel=True)
    got = m(x.cuda())
    torch.cuda.synchronize()
    assert got.shape == (8, 128, 3001)
    ref = oracle_mod.mel_spectrogram(x.numpy(), 16000, 400, 160, 128, f_max=8000.0, log_mel=True)
    _gate(got.cpu().numpy(), ref, 1e-4)
    m.close()


def test_pcm16_full_size_every_clip(lm, oracle_mod):
    # 32 x 220500 int16, n_fft 1024, hop 256, 128 Slaney bands, f16 output:
    # the whole batch on the GPU and in the oracle.
    w = workloads.WAVE_PCM16
    x = workloads.wave_workload_inputs(w)
    m = lm.MelSpectrogram(sample_rate=22050, n_fft=1024, hop_length=256, n_mels=128, f_max=11025.0,
                          mel_scale="slaney", dtype=torch.float16)
    got = m(x.cuda())
    torch.cuda.synchronize()
    assert got.shape == (32, 128, 862) and got.dtype == torch.float16
    ref = oracle_mod.mel_spectrogram(x.numpy(), 22050, 1024, 256, 128, f_max=11025.0, mel_scale="slaney",
                                     out_dtype="f16")
    _gate(got.float().cpu().numpy(), ref.astype(np.float64), 2e-3)
    m.close()


def test_unaligned_input_and_long_hop_fallbacks(lm, oracle_mod):
    # A waveform view starting 4 bytes past a 16-byte boundary cannot be bulk
    # copied, and a hop this long makes a tile's sample span too big for shared
    # memory: both take the per-sample path and must agree with the oracle.
    base = workloads.wave_sines(1, 24001, 16000, seed=12)
    x = base[0, 1:].reshape(2, 12000)  # contiguous, but the storage offset is one float
    got_ref = _run(lm, oracle_mod, x.contiguous(), 16000, 400, 160, 64, f_max=8000.0)
    m = lm.MelSpectrogram(sample_rate=16000, n_fft=400, hop_length=160, n_mels=64, f_max=8000.0)
    xs = base.cuda()[0, 1:24001].view(2, 12000)
    assert xs.data_ptr() % 16 == 4
    got = m(xs)
    torch.cuda.synchronize()
    assert torch.equal(got.cpu(), got_ref.cpu())
    m.close()
    y = workloads.wave_sines(2, 40000, 16000, seed=13)
    _run(lm, oracle_mod, y, 16000, 400, 3000, 64, f_max=8000.0)


@pytest.mark.parametrize("win_length,pad,normalized,center,pad_mode,n_fft",
                         [(300, 0, False, True, "reflect", 400), (400, 37, False, True, "reflect", 400),
                          (400, 0, True, True, "constant", 400), (256, 11, True, False, "reflect", 512),
                          (333, 5, True, True, "replicate", 400), (1024, 300, False, True, "circular", 1024),
                          (700, 64, True, True, "reflect", 1024)])
def test_full_torchaudio_argument_set(lm, oracle_mod, win_length, pad, normalized, center, pad_mode, n_fft):
    # win_length < n_fft (window centred with zeros around it), `pad` zeros
    # before centre padding, the "window" normalisation, every pad mode.
    x = workloads.wave_sines(2, 6000, 16000, seed=win_length + pad)
    _run(lm, oracle_mod, x, 16000, n_fft, n_fft // 4, 64, f_max=8000.0, center=center, pad_mode=pad_mode,
         win_length=win_length, pad=pad, normalized=normalized)
    p = workloads.wave_pcm16(1, 4000, seed=pad)
    _run(lm, oracle_mod, p, 16000, n_fft, n_fft // 4, 48, mel_scale="slaney", norm="slaney", out_dtype="f16",
         win_length=win_length, pad=pad, normalized=normalized, center=center, pad_mode=pad_mode)


@pytest.mark.parametrize("in_dtype", ["f32", "i16"])
def test_odd_hop_and_odd_span_head(lm, oracle_mod, in_dtype):
    # An odd hop makes every other frame's sample pairs unaligned in the span
    # buffer (the scalar framing path); an odd leading pad offsets the whole
    # span by one sample.
    x = workloads.wave_sines(2, 9000, 16000, seed=41) if in_dtype == "f32" else workloads.wave_pcm16(2, 9000, seed=41)
    _run(lm, oracle_mod, x, 16000, 400, 161, 80, f_max=8000.0)
    _run(lm, oracle_mod, x, 16000, 512, 127, 64, f_max=8000.0, pad=3)


def test_repeat_calls_are_bitwise_identical(lm):
    # Tiles are claimed dynamically; the result must not depend on which CTA
    # computed which tile.
    x = workloads.wave_sines(4, 48000, 16000, seed=3).cuda()
    for log_mel in (False, True):
        m = lm.MelSpectrogram(sample_rate=16000, n_fft=400, hop_length=160, n_mels=128, f_max=8000.0,
                              log_mel=log_mel)
        a = m(x)
        b = m(x)
        torch.cuda.synchronize()
        assert torch.equal(a, b)
        m.close()


@pytest.mark.parametrize("n_fft,hop,sr,f_max", [(400, 160, 16000, 8000.0), (1024, 256, 22050, 11025.0),
                                                (64, 16, 16000, 8000.0), (256, 64, 16000, 8000.0)])
def test_fused_and_separate_log_epilogues_agree(lm, oracle_mod, monkeypatch, n_fft, hop, sr, f_max):
    # With LOGMEL_K3_EPILOGUE=fused the register kernels floor and rescale
    # log plans in the same launch (the clip maximum gathered across CTAs);
    # by default (separate) the clamp kernel runs after them.  Both give the
    # same bits, and the oracle's values.
    x = workloads.wave_sines(5, 37000, sr, seed=n_fft + 5)
    x[2, 20000:] *= 1e-5  # the clip floor matters
    args = dict(sample_rate=sr, n_fft=n_fft, hop_length=hop, n_mels=128, f_max=f_max, log_mel=True)
    m = lm.MelSpectrogram(**args)
    monkeypatch.setenv("LOGMEL_K3_EPILOGUE", "fused")
    fused = m(x.cuda())
    monkeypatch.setenv("LOGMEL_K3_EPILOGUE", "separate")
    sep = m(x.cuda())
    torch.cuda.synchronize()
    m.close()
    assert torch.equal(fused, sep)
    ref = oracle_mod.mel_spectrogram(x.numpy(), sr, n_fft, hop, 128, f_max=f_max, log_mel=True)
    _gate(fused.cpu().numpy(), ref, 1e-4)


def test_fused_log_epilogue_many_tiles_per_cta(lm, oracle_mod, monkeypatch):
    # 442 clips of 10 s: 14,144 tiles of 32 frames, about 31 per CTA of the
    # 400-point kernel, so CTAs that run out of tiles to compute rescale
    # finished clips for a long time while others still compute; the result
    # must equal the separate clamp kernel's, bit for bit.
    x = workloads.wave_sines(442, 160000, 16000, seed=77, device="cuda")
    args = dict(sample_rate=16000, n_fft=400, hop_length=160, n_mels=128, f_max=8000.0, log_mel=True)
    m = lm.MelSpectrogram(**args)
    ws = torch.empty(m.workspace_size(442, 160000), dtype=torch.uint8, device="cuda")
    monkeypatch.setenv("LOGMEL_K3_EPILOGUE", "fused")
    fused = m(x, workspace=ws)
    assert lm.workspace_error(ws) == 0
    monkeypatch.setenv("LOGMEL_K3_EPILOGUE", "separate")
    sep = m(x, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(fused, sep)
    for b in (0, 441):
        ref = oracle_mod.mel_spectrogram(x[b:b + 1].cpu().numpy(), 16000, 400, 160, 128, f_max=8000.0, log_mel=True)
        _gate(fused[b:b + 1].cpu().numpy(), ref, 1e-4)
    m.close()


@pytest.mark.parametrize("n_fft,hop,sr,f_max,log_mel,epilogue", [
    (400, 160, 16000, 8000.0, True, "fused"),      # register kernel, fused log epilogue
    (400, 160, 16000, 8000.0, True, "separate"),   # register kernel, clamp kernel after it
    (1024, 256, 22050, 11025.0, False, "auto"),    # register kernel, no log
    (2048, 512, 22050, 11025.0, True, "auto"),     # generic kernel, clamp kernel after it
])
def test_workspace_garbage_reuse_and_offset(lm, oracle_mod, monkeypatch, n_fft, hop, sr, f_max, log_mel, epilogue):
    """A call clears its error word, tile counter and clip words itself (no
    memset in front of it): the workspace is filled with random bytes, then
    used by calls in a row whose clip maxima differ, and once through a view
    4 bytes off an 8-byte boundary (the memset path); every result is checked
    against the oracle."""
    monkeypatch.setenv("LOGMEL_K3_EPILOGUE", epilogue)
    dev = torch.device("cuda")
    B, T = 5, 6 * sr // 2
    m = lm.MelSpectrogram(sample_rate=sr, n_fft=n_fft, hop_length=hop, n_mels=80, f_max=f_max, log_mel=log_mel)
    n = m.workspace_size(B, T)
    raw = torch.empty(n + 512, dtype=torch.uint8, device=dev)
    g = torch.Generator(device="cpu").manual_seed(78)
    raw.copy_(torch.randint(1, 256, (n + 512,), dtype=torch.uint8, generator=g))
    o8 = (-raw.data_ptr()) % 256
    for k, (scale, off) in enumerate(((1.0, o8), (1e-3, o8), (10.0, o8), (1.0, o8 + 4))):
        x = workloads.wave_sines(B, T, sr, seed=90 + k) * scale
        ws = raw[off:off + n]
        got = m(x.to(dev), workspace=ws)
        assert lm.workspace_error(ws) == 0
        ref = oracle_mod.mel_spectrogram(x.numpy(), sr, n_fft, hop, 80, f_max=f_max, log_mel=log_mel)
        _gate(got.float().cpu().numpy(), ref.astype(np.float64), 1e-4)
    m.close()


def test_large_sizes_repeat_between_other_kernels(lm, oracle_mod):
    """Calls at 8192 and 16384 points, interleaved with register-kernel calls
    that leave other data in shared memory, give the same bits every time
    (a CTA may not read its own shared-memory state before it is set), and
    the first result of each matches the oracle."""
    dev = torch.device("cuda")
    T = 3 * 16384 + 77
    x = workloads.wave_sines(2, T, 16000, seed=71)
    xd = x.to(dev)
    other = lm.MelSpectrogram(sample_rate=16000, n_fft=1024, hop_length=256, n_mels=128, f_max=8000.0, log_mel=True)
    big = {n: lm.MelSpectrogram(sample_rate=16000, n_fft=n, hop_length=n // 2, n_mels=128, f_max=8000.0)
           for n in (8192, 16384)}
    first = {}
    for _ in range(12):
        for n, m in big.items():
            other(xd)
            got = m(xd)
            if n not in first:
                first[n] = got.clone()
                ref = oracle_mod.mel_spectrogram(x.numpy(), 16000, n, n // 2, 128, f_max=8000.0)
                _gate(got.cpu().numpy(), ref.astype(np.float64), 1e-4)
            else:
                assert torch.equal(got, first[n]), n
    for m in (other, *big.values()):
        m.close()


@pytest.mark.parametrize("n_fft,win_length,pad,normalized,center,pad_mode,power", [
    (4096, 3000, 0, True, True, "circular", 2.0),      # generic kernel, Stockham, tables in shared memory
    (8192, 5000, 100, True, False, "constant", 1.0),   # in place, no centre padding, magnitude
    (16384, 16384, 37, False, True, "replicate", 2.0),  # in place, replicate padding after `pad` zeros
])
def test_large_sizes_argument_surface(lm, oracle_mod, n_fft, win_length, pad, normalized, center, pad_mode, power):
    # The torchaudio argument surface on the large-size paths; a few frames a
    # clip keep the oracle's direct DFT to seconds.
    T = 2 * n_fft + 500
    x = workloads.wave_sines(2, T, 16000, seed=n_fft + 9)
    _run(lm, oracle_mod, x, 16000, n_fft, n_fft // 4, 96, f_max=8000.0, center=center, pad_mode=pad_mode,
         power=power, win_length=win_length, pad=pad, normalized=normalized)
