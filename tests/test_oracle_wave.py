"""Pins for the oracle's waveform -> mel spectrogram path.

The flashmel page fixes the shape of the computation (torchaudio-style
MelSpectrogram: center/reflect framing, periodic Hann, one-sided FFT,
|X|^power, HTK or Slaney mel filterbank, int16 input scaled by 1/32768, f16
output).  These checks pin each stage of the oracle to something other than
itself: library routines the stage reduces to (numpy's rFFT, torch.stft in
float64, numpy's float16 rounding), closed forms (Hann spectrum lines,
Parseval, mel-scale anchor points) and invariants (partition of unity).
"""
import cmath
import math

import numpy as np
import pytest
import torch

import workloads


def test_dft_brute_force_small(oracle_mod):
    # One frame, no padding: |sum_j x_j w_j e^{-2 pi i j k / N}|^2 summed in Python.
    rng = np.random.default_rng(11)
    for N in (2, 4, 8, 12, 16):
        x = rng.standard_normal(N)
        spec = oracle_mod.power_spectrogram(x, N, N, center=False)
        assert spec.shape == (1, N // 2 + 1)
        w = [0.5 - 0.5 * math.cos(2 * math.pi * j / N) for j in range(N)]
        for k in range(N // 2 + 1):
            X = sum(x[j] * w[j] * cmath.exp(-2j * math.pi * j * k / N) for j in range(N))
            assert abs(spec[0, k] - abs(X) ** 2) <= 1e-12 * (1 + abs(X) ** 2)


@pytest.mark.parametrize("N", [400, 1024, 64])
def test_dft_matches_numpy_rfft(oracle_mod, N):
    rng = np.random.default_rng(N)
    x = rng.standard_normal(3 * N)
    hop = N
    spec = oracle_mod.power_spectrogram(x, N, hop, center=False)
    w = np.hanning(N + 1)[:-1]  # numpy's symmetric window of N+1 points, truncated = periodic Hann
    for t in range(spec.shape[0]):
        X = np.fft.rfft(x[t * hop: t * hop + N] * w)
        np.testing.assert_allclose(spec[t], np.abs(X) ** 2, rtol=1e-10, atol=1e-9)


@pytest.mark.parametrize("pad_mode", ["reflect", "constant", "replicate", "circular"])
@pytest.mark.parametrize("n_fft,hop", [(400, 160), (64, 16), (1024, 256)])
def test_power_spectrogram_matches_torch_stft(oracle_mod, pad_mode, n_fft, hop):
    rng = np.random.default_rng(5)
    T = 3 * n_fft + 37
    x = rng.standard_normal(T)
    spec = oracle_mod.power_spectrogram(x, n_fft, hop, center=True, pad_mode=pad_mode)
    xt = torch.from_numpy(x)
    win = torch.hann_window(n_fft, periodic=True, dtype=torch.float64)
    X = torch.stft(xt, n_fft, hop_length=hop, window=win, center=True, pad_mode=pad_mode,
                   return_complex=True, onesided=True)
    ref = (X.abs() ** 2).T.numpy()
    assert spec.shape == ref.shape
    np.testing.assert_allclose(spec, ref, rtol=1e-9, atol=1e-9)


def test_center_false_framing(oracle_mod):
    rng = np.random.default_rng(9)
    x = rng.standard_normal(1000)
    spec = oracle_mod.power_spectrogram(x, 64, 24, center=False)
    win = torch.hann_window(64, periodic=True, dtype=torch.float64)
    X = torch.stft(torch.from_numpy(x), 64, hop_length=24, window=win, center=False,
                   return_complex=True)
    np.testing.assert_allclose(spec, (X.abs() ** 2).T.numpy(), rtol=1e-9, atol=1e-9)


def test_parseval(oracle_mod):
    # sum_k c_k |X_k|^2 = N sum_j (x_j w_j)^2 with c_0 = c_{N/2} = 1, else 2.
    rng = np.random.default_rng(2)
    for N in (400, 1024):
        x = rng.standard_normal(N)
        spec = oracle_mod.power_spectrogram(x, N, N, center=False)[0]
        c = np.full(N // 2 + 1, 2.0)
        c[0] = c[-1] = 1.0
        w = oracle_mod.hann_window(N)
        assert math.isclose((c * spec).sum(), N * np.sum((x * w) ** 2), rel_tol=1e-11)


def test_hann_spectrum_lines(oracle_mod):
    # A cosine on bin k0 through a periodic Hann window has exactly three
    # lines: |X_k0| = A N/4 and |X_k0+-1| = A N/8; everything else is zero.
    N, k0, A = 400, 37, 0.7
    j = np.arange(4 * N)
    x = A * np.cos(2 * np.pi * k0 * j / N + 0.3)
    spec = oracle_mod.power_spectrogram(x, N, 160, center=True)
    interior = spec[3]  # frame 3 starts at 3*160 - 200 = 280 >= 0: no padding in it
    amp = np.sqrt(interior)
    assert math.isclose(amp[k0], A * N / 4, rel_tol=1e-9)
    assert math.isclose(amp[k0 - 1], A * N / 8, rel_tol=1e-9)
    assert math.isclose(amp[k0 + 1], A * N / 8, rel_tol=1e-9)
    rest = np.delete(amp, [k0 - 1, k0, k0 + 1])
    assert rest.max() < 1e-9 * A * N


def test_dc_input(oracle_mod):
    # Constant c: X_0 = c N/2 (the window's sum), |X_1| = c N/4, the rest 0.
    N, c = 64, 1.25
    spec = oracle_mod.power_spectrogram(np.full(N, c), N, N, center=False)[0]
    assert math.isclose(math.sqrt(spec[0]), c * N / 2, rel_tol=1e-12)
    assert math.isclose(math.sqrt(spec[1]), c * N / 4, rel_tol=1e-12)
    assert np.sqrt(spec[2:]).max() < 1e-10


def test_hann_window_values(oracle_mod):
    # Periodic Hann: w_0 = 0, w_{N/2} = 1, w_{N/4} = 1/2, symmetric about N/2.
    w = oracle_mod.hann_window(400)
    assert w[0] == 0.0 and math.isclose(w[200], 1.0) and math.isclose(w[100], 0.5)
    np.testing.assert_allclose(w[1:], w[1:][::-1], atol=1e-15)
    np.testing.assert_allclose(w, torch.hann_window(400, periodic=True, dtype=torch.float64).numpy(),
                               atol=1e-15)


def test_n_frames_closed_form(oracle_mod):
    assert oracle_mod.n_frames(480000, 400, 160, True) == 3001
    assert oracle_mod.n_frames(220500, 1024, 256, True) == 862
    assert oracle_mod.n_frames(1000, 64, 24, False) == 1 + (1000 - 64) // 24
    assert oracle_mod.n_frames(30, 64, 24, False) == 0


def test_mel_scale_anchor_points(oracle_mod):
    # HTK: mel(0) = 0, mel(6300 Hz) = 2595 exactly (1 + 6300/700 = 10).
    assert oracle_mod.hz_to_mel(0.0, "htk") == 0.0
    assert math.isclose(oracle_mod.hz_to_mel(6300.0, "htk"), 2595.0, rel_tol=1e-14)
    # Slaney: 200/3 Hz per mel up to 1 kHz = mel 15; then 27 mels per factor 6.4.
    assert math.isclose(oracle_mod.hz_to_mel(200.0 / 3.0, "slaney"), 1.0, rel_tol=1e-14)
    assert math.isclose(oracle_mod.hz_to_mel(1000.0, "slaney"), 15.0, rel_tol=1e-14)
    assert math.isclose(oracle_mod.hz_to_mel(6400.0, "slaney"), 42.0, rel_tol=1e-14)
    assert math.isclose(oracle_mod.hz_to_mel(6400.0 * 6.4, "slaney"), 69.0, rel_tol=1e-14)
    for scale in ("htk", "slaney"):
        for f in (0.0, 55.0, 999.0, 1000.0, 1234.5, 11025.0):
            assert math.isclose(oracle_mod.mel_to_hz(oracle_mod.hz_to_mel(f, scale), scale), f,
                                rel_tol=1e-12, abs_tol=1e-9)


@pytest.mark.parametrize("n_fft,sr,f_max,scale", [(400, 16000, 8000.0, "htk"),
                                                   (1024, 22050, 11025.0, "slaney"),
                                                   (512, 16000, 7600.0, "htk")])
def test_filterbank_triangles(oracle_mod, n_fft, sr, f_max, scale):
    n_freqs, n_mels = n_fft // 2 + 1, 128 if n_fft != 512 else 40
    fb = oracle_mod.mel_filterbank(n_freqs, 0.0, f_max, n_mels, sr, scale)
    assert fb.min() >= 0.0 and fb.max() <= 1.0 + 1e-12
    bin_hz = np.arange(n_freqs) * (sr / 2) / (n_freqs - 1)
    m = np.linspace(oracle_mod.hz_to_mel(0.0, scale), oracle_mod.hz_to_mel(f_max, scale), n_mels + 2)
    f_pts = np.array([oracle_mod.mel_to_hz(v, scale) for v in m])
    for n in range(n_mels):
        nz = np.nonzero(fb[n])[0]
        if nz.size == 0:
            # an empty row has no bin strictly inside its triangle
            assert not np.any((bin_hz > f_pts[n]) & (bin_hz < f_pts[n + 2]))
            continue
        assert np.all(np.diff(nz) == 1)                       # one contiguous support
        d = np.diff(fb[n, nz[0]: nz[-1] + 1])
        peak = int(np.argmax(fb[n]))
        assert np.all(d[: peak - nz[0]] >= -1e-12) and np.all(d[peak - nz[0]:] <= 1e-12)
        assert abs(bin_hz[peak] - f_pts[n + 1]) <= (sr / 2) / (n_freqs - 1) + 1e-9
        assert np.all((bin_hz[nz] > f_pts[n]) & (bin_hz[nz] < f_pts[n + 2]))
    # partition of unity between the first and the last centre
    s = fb.sum(axis=0)
    inside = (bin_hz >= f_pts[1]) & (bin_hz <= f_pts[n_mels])
    np.testing.assert_allclose(s[inside], 1.0, atol=1e-12)


def test_whisper_htk_has_empty_low_bands(oracle_mod):
    # 128 HTK bands over 0-8 kHz on 40 Hz bins: the lowest triangles are
    # narrower than a bin and some fall between bins, leaving all-zero rows.
    fb = oracle_mod.mel_filterbank(201, 0.0, 8000.0, 128, 16000, "htk")
    empty = np.where(fb.sum(axis=1) == 0)[0]
    assert empty.size > 0 and empty.max() < 20


def test_slaney_norm_unit_area(oracle_mod):
    # norm='slaney' scales each triangle to unit area; for triangles many bins
    # wide the Riemann sum over bins approaches that area.
    sr, n_fft = 22050, 1024
    n_freqs = n_fft // 2 + 1
    df = (sr / 2) / (n_freqs - 1)
    fb = oracle_mod.mel_filterbank(n_freqs, 0.0, 11025.0, 128, sr, "slaney", norm="slaney")
    raw = oracle_mod.mel_filterbank(n_freqs, 0.0, 11025.0, 128, sr, "slaney")
    checked = 0
    for n in range(128):
        width = np.count_nonzero(raw[n])
        if width >= 20:
            assert abs(fb[n].sum() * df - 1.0) < 0.02
            checked += 1
        nz = raw[n] > 0
        if nz.any():  # same shape, one positive factor per row
            ratio = fb[n][nz] / raw[n][nz]
            np.testing.assert_allclose(ratio, ratio[0], rtol=1e-12)
    assert checked > 10


def test_f16_rounding_matches_numpy(oracle_mod):
    rng = np.random.default_rng(1)
    vals = list(rng.standard_normal(2000) * 10.0 ** rng.integers(-9, 5, 2000))
    vals += [0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e6, -1e6, 2.0 ** -24, 2.0 ** -25,
             3 * 2.0 ** -26, 2.0 ** -14, 2.0 ** -14 - 2.0 ** -25, 1.0 + 2.0 ** -11,
             1.0 + 3 * 2.0 ** -11, 2049.0, 2051.0, -1.5, 0.1]
    with np.errstate(over="ignore"):  # values from 65520 up round to infinity on purpose
        for v in vals:
            assert oracle_mod.f64_to_f16_bits(v) == int(np.array(v, dtype=np.float64)
                                                        .astype(np.float16).view(np.uint16)), v


def test_int16_input_is_scaled(oracle_mod):
    # i16 PCM is x / 32768; that value is exact in f32, so both inputs agree.
    pcm = workloads.wave_pcm16(2, 3000, 4).numpy()
    a = oracle_mod.mel_spectrogram(pcm, 22050, 256, 64, 32, mel_scale="slaney")
    b = oracle_mod.mel_spectrogram(pcm.astype(np.float32) / 32768.0, 22050, 256, 64, 32,
                                   mel_scale="slaney")
    assert np.array_equal(a, b)


def test_pure_tone_lands_in_its_band(oracle_mod):
    sr, f0 = 16000, 1000.0
    t = np.arange(8000) / sr
    x = (0.5 * np.sin(2 * np.pi * f0 * t)).astype(np.float32)[None]
    mel = oracle_mod.mel_spectrogram(x, sr, 400, 160, 128, f_max=8000.0)
    band = int(np.argmax(mel[0, :, 20]))
    m = np.linspace(0, oracle_mod.hz_to_mel(8000.0, "htk"), 130)
    centre = oracle_mod.mel_to_hz(m[band + 1], "htk")
    spacing = oracle_mod.mel_to_hz(m[band + 2], "htk") - centre
    assert abs(centre - f0) <= spacing


def test_log_path_window_and_silence(oracle_mod):
    x = workloads.wave_sines(2, 16000, 16000, 3).numpy()
    x[1] = 0.0
    out = oracle_mod.mel_spectrogram(x, 16000, 400, 160, 128, f_max=8000.0, log_mel=True)
    mx = out[0].max()
    assert out[0].min() >= mx - 2.0 - 1e-6
    assert np.all(out[1] == np.float32(-1.5))  # silence: log10(1e-10) = -10 -> -1.5


def test_f16_output_is_rounded_f32_path(oracle_mod):
    pcm = workloads.wave_pcm16(1, 5000, 8).numpy()
    a = oracle_mod.mel_spectrogram(pcm, 22050, 1024, 256, 128, mel_scale="slaney", out_dtype="f16")
    b = oracle_mod.mel_spectrogram(pcm, 22050, 1024, 256, 128, mel_scale="slaney", out_dtype="f32")
    # f32 rounding then f16 rounding can differ from direct f16 rounding by at
    # most one f16 ulp; values this far from the range limits stay finite.
    assert np.all(np.isfinite(a.astype(np.float32)))
    np.testing.assert_allclose(a.astype(np.float64), b.astype(np.float64), rtol=2 ** -10, atol=0)


@pytest.mark.parametrize("win_length,pad,normalized,center,pad_mode",
                         [(300, 0, False, True, "reflect"), (400, 37, False, True, "reflect"),
                          (400, 0, True, True, "constant"), (256, 11, True, False, "reflect"),
                          (333, 5, True, True, "replicate")])
def test_power_spectrogram_full_argument_set(oracle_mod, win_length, pad, normalized, center, pad_mode):
    # torchaudio's Spectrogram: zero `pad` first, then torch.stft with a periodic
    # Hann of win_length centred in n_fft, and for normalized=True ("window")
    # a division of X by sqrt(sum w^2).  torch.stft in float64 is the reference.
    rng = np.random.default_rng(win_length + pad)
    n_fft, hop, T = 400, 128, 2100
    x = rng.standard_normal(T)
    spec = oracle_mod.power_spectrogram(x, n_fft, hop, center=center, pad_mode=pad_mode, win_length=win_length,
                                        pad=pad, normalized=normalized)
    xt = torch.nn.functional.pad(torch.from_numpy(x)[None], (pad, pad), mode="constant")[0]
    win = torch.hann_window(win_length, periodic=True, dtype=torch.float64)
    X = torch.stft(xt, n_fft, hop_length=hop, win_length=win_length, window=win, center=center,
                   pad_mode=pad_mode, return_complex=True, onesided=True)
    if normalized:
        X = X / win.pow(2).sum().sqrt()
    ref = (X.abs() ** 2).T.numpy()
    assert spec.shape == ref.shape
    np.testing.assert_allclose(spec, ref, rtol=1e-9, atol=1e-9)


def test_pad_changes_frame_count(oracle_mod):
    x = workloads.wave_sines(1, 1000, 16000, 2).numpy()
    out = oracle_mod.mel_spectrogram(x, 16000, 400, 160, 40, pad=80)
    assert out.shape == (1, 40, 1 + (1000 + 160) // 160)


@pytest.mark.parametrize("center,normalized,win_length,pad_mode",
                         [(True, False, None, "reflect"), (False, False, None, "reflect"),
                          (True, True, None, "constant"), (True, True, 300, "reflect"),
                          (False, False, 256, "reflect"), (True, False, None, "circular")])
def test_magnitude_spectrogram_matches_torch_stft(oracle_mod, center, normalized, win_length, pad_mode):
    # power = 1 is the magnitude |X| (torchaudio's Spectrogram with power=1),
    # not the power and not its square root taken twice: torch.stft in
    # float64, its .abs(), pins the oracle's power != 2 branch for the plain
    # and the full-argument entry points alike.
    rng = np.random.default_rng(17 + (win_length or 0))
    n_fft, hop, T = 400, 100, 3 * 400 + 51
    x = rng.standard_normal(T)
    spec = oracle_mod.power_spectrogram(x, n_fft, hop, center=center, pad_mode=pad_mode, power=1.0,
                                        win_length=win_length, normalized=normalized)
    wl = win_length or n_fft
    win = torch.hann_window(wl, periodic=True, dtype=torch.float64)
    X = torch.stft(torch.from_numpy(x), n_fft, hop_length=hop, win_length=wl, window=win, center=center,
                   pad_mode=pad_mode, return_complex=True, onesided=True)
    if normalized:
        X = X / win.pow(2).sum().sqrt()
    ref = X.abs().T.numpy()
    assert spec.shape == ref.shape
    np.testing.assert_allclose(spec, ref, rtol=1e-9, atol=1e-9)
    # the power-2 result is the square of the magnitude, element by element
    spec2 = oracle_mod.power_spectrogram(x, n_fft, hop, center=center, pad_mode=pad_mode, power=2.0,
                                         win_length=win_length, normalized=normalized)
    np.testing.assert_allclose(spec2, ref ** 2, rtol=1e-9, atol=1e-9)


def test_mel_spectrogram_power_one_is_filterbank_times_magnitude(oracle_mod):
    # The magnitude branch end to end, in the configuration the GPU parity
    # test uses it (center=False, f_min=60, f_max=7600, hop 100): the
    # filterbank (pinned above on its own) applied to torch.stft's |X|.
    x = workloads.wave_sines(1, 5000, 16000, seed=9)
    got = oracle_mod.mel_spectrogram(x.numpy(), 16000, 400, 100, 80, f_min=60.0, f_max=7600.0, center=False,
                                     power=1.0)
    fb = oracle_mod.mel_filterbank(201, 60.0, 7600.0, 80, 16000, scale="htk")
    win = torch.hann_window(400, periodic=True, dtype=torch.float64)
    X = torch.stft(x[0].double(), 400, hop_length=100, window=win, center=False, return_complex=True,
                   onesided=True)
    ref = fb @ X.abs().numpy()
    assert got.shape == (1,) + ref.shape
    # the oracle rounds its output to f32 once
    np.testing.assert_allclose(got[0].astype(np.float64), ref, rtol=2 ** -23, atol=1e-12)
