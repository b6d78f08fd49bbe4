"""Pins for the oracle's log_mel_from_stft against facts fixed outside it.

Each check comes from the KBench task spec "audio_mel_spectrogram_fused.py"
(its per-clip definition and its correctness notes) or from the mathematics
of the definition, not from re-running the oracle's own formula.
"""
import pathlib

import numpy as np
import pytest

import workloads

GOLDEN = pathlib.Path(__file__).resolve().parent / "golden"


def _read_golden(path):
    blocks, cur = {}, None
    for line in path.read_text().splitlines():
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        head = line.split()
        if head[0].isalpha():
            cur = head[0]
            blocks[cur] = {"shape": tuple(int(x) for x in head[1:]), "vals": []}
        else:
            blocks[cur]["vals"].extend(float(x) for x in head)
    return {k: np.array(v["vals"]).reshape(v["shape"]) for k, v in blocks.items()}


def _small_inputs(B=3, F=37, NF=65, NM=40, seed=7):
    stft, W = workloads.stft_inputs(B, F, NF, NM, seed)
    return stft.numpy(), W.numpy()


def test_worked_example(oracle_mod):
    g = _read_golden(GOLDEN / "stft_worked_example.txt")
    ri = g["stft"]  # [B, F, NF, 2] (re, im)
    stft = (ri[..., 0] + 1j * ri[..., 1]).astype(np.complex64)
    out = oracle_mod.log_mel_from_stft(stft, g["filters"].astype(np.float32))
    np.testing.assert_allclose(out, g["expected"], rtol=0, atol=1e-6)


def test_all_zero_clip_is_minus_one_and_a_half(oracle_mod):
    # mel = 0 everywhere -> floored at 1e-10 -> log = -10 = hi -> (-10+4)/4.
    stft, W = _small_inputs(B=2)
    stft[1] = 0
    out = oracle_mod.log_mel_from_stft(stft, W)
    assert np.all(out[1] == np.float32(-1.5))
    assert not np.all(out[0] == np.float32(-1.5))


def test_outputs_lie_in_the_80db_window(oracle_mod):
    # Every output lies in [max_out - 2, max_out] and max_out = (hi + 4)/4 is reached.
    stft, W = _small_inputs()
    out = oracle_mod.log_mel_from_stft(stft, W).astype(np.float64)
    for b in range(out.shape[0]):
        mx = out[b].max()
        assert out[b].min() >= mx - 2.0 - 1e-6
    # a clip whose dynamic range is wider than 80 dB actually hits the floor
    stft2 = stft.copy()
    stft2[0, : stft.shape[1] // 2] *= 1e-6  # 120 dB quieter frames
    out2 = oracle_mod.log_mel_from_stft(stft2, W).astype(np.float64)
    mx = out2[0].max()
    assert np.isclose(out2[0].min(), mx - 2.0, atol=1e-6)
    assert np.sum(np.isclose(out2[0], mx - 2.0, atol=1e-6)) > 10


def test_scaling_shifts_every_output(oracle_mod):
    # stft * 10 multiplies the power by 100: log10 moves by +2 everywhere,
    # and so does the clip floor, so every output moves by exactly +2/4.
    stft, W = _small_inputs()
    a = oracle_mod.log_mel_from_stft(stft, W).astype(np.float64)
    b = oracle_mod.log_mel_from_stft(stft * np.float32(10.0), W).astype(np.float64)
    np.testing.assert_allclose(b - a, 0.5, atol=2e-6)


def test_clips_are_independent(oracle_mod):
    # The floor is per clip: changing clip 1 must leave clip 0 bit-identical.
    stft, W = _small_inputs()
    a = oracle_mod.log_mel_from_stft(stft, W)
    stft2 = stft.copy()
    stft2[1] *= np.float32(1e5)
    b = oracle_mod.log_mel_from_stft(stft2, W)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[2], b[2])
    assert not np.array_equal(a[1], b[1])


def test_frame_permutation_commutes(oracle_mod):
    # The definition is per frame except for the clip max, which is order
    # free: permuting frames permutes the output rows.
    stft, W = _small_inputs()
    perm = np.random.default_rng(0).permutation(stft.shape[1])
    a = oracle_mod.log_mel_from_stft(stft, W)
    b = oracle_mod.log_mel_from_stft(stft[:, perm], W)
    assert np.array_equal(a[:, perm], b)


def test_projection_is_linear_in_power(oracle_mod):
    # With a single nonzero filter tap, each band is log10 of one bin's power:
    # an identity filterbank on NF = NM reduces to log10(re^2 + im^2).
    rng = np.random.default_rng(3)
    NF = 17
    stft = (rng.standard_normal((1, 5, NF)) + 1j * rng.standard_normal((1, 5, NF))).astype(np.complex64)
    W = np.eye(NF, dtype=np.float32)
    out = oracle_mod.log_mel_from_stft(stft, W).astype(np.float64)
    p = np.abs(stft.astype(np.complex128)) ** 2
    ls = np.log10(np.maximum(p, 1e-10))
    ref = (np.maximum(ls, ls.max() - 8.0) + 4.0) / 4.0
    np.testing.assert_allclose(out, ref, atol=1e-6)


def test_partition_of_unity_of_the_input_filters():
    # The spec's linspace triangles sum to one on every bin between the first
    # and the last centre: the generator that both sides share is what it says.
    NF, NM = 201, 80
    W = workloads.triangle_filters(NF, NM).numpy().astype(np.float64)
    centres = np.linspace(0, NF - 1, NM + 2)
    s = W.sum(axis=0)
    inside = (np.arange(NF) >= centres[1]) & (np.arange(NF) <= centres[-2])
    np.testing.assert_allclose(s[inside], 1.0, atol=1e-5)
    assert W.min() >= 0 and W.max() <= 1.0 + 1e-6


def _gate(a, b, atol=1e-4, rtol=1e-4):
    return bool(np.all(np.abs(a.astype(np.float64) - b) <= atol + rtol * np.abs(b)))


def test_wrong_variants_fail_the_gate(oracle_mod):
    # The spec says its tolerance catches a per-frame or per-batch clamp and a
    # bf16 projection.  Plant each mistake in the oracle and check the gate
    # rejects it on inputs where the floor is active.
    stft, W = _small_inputs(B=3, F=64, NF=129, NM=80)
    stft[0, 32:] *= np.float32(1e-5)   # quiet half-clip: 100 dB down
    stft[2] *= np.float32(1e-5)        # a whole quiet clip
    ref = oracle_mod.log_mel_from_stft(stft, W).astype(np.float64)
    same = oracle_mod.log_mel_from_stft_wrong(stft, W, scope="clip")
    assert _gate(same, ref)
    for kw in ({"scope": "frame"}, {"scope": "batch"}, {"bf16_projection": True}):
        bad = oracle_mod.log_mel_from_stft_wrong(stft, W, **kw)
        assert not _gate(bad, ref), kw
        if "scope" in kw:  # the clamp mistakes also fail the relative-Frobenius gate
            fro = np.linalg.norm(bad - ref) / np.linalg.norm(ref)
            assert fro > 1e-4, (kw, fro)
