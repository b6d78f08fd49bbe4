"""GPU parity of log_mel_from_stft against the CPU oracle.

Gate (elementwise): |gpu - oracle| <= 1e-4 + 1e-4 |oracle|, the f32
tolerance the log-mel front end is specified at; the KBench spec's
relative-Frobenius gate (1e-4) is checked too.  Inputs come from the seeded
generators in workloads.py and are identical on both sides.
"""
import os

import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

ATOL = RTOL = 1e-4


@pytest.fixture(scope="module")
def lm():
    import __graft_entry__
    __graft_entry__.build()
    import log_mel_spectrogram_gb300
    return log_mel_spectrogram_gb300


def _compare(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape
    err = np.abs(got - ref)
    bad = err > ATOL + RTOL * np.abs(ref)
    assert not bad.any(), (f"{bad.sum()} of {bad.size} outside tolerance; max err {err.max():.3g} "
                           f"at {np.unravel_index(np.argmax(err), err.shape)}")
    fro = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    assert fro <= 1e-4
    return err.max()


def _run(lm, oracle_mod, stft, W, check_ws=True):
    dev = torch.device("cuda")
    ws = torch.empty(lm.log_mel_from_stft_workspace_size(*stft.shape, W.shape[0]), dtype=torch.uint8, device=dev)
    out = lm.log_mel_from_stft(stft.to(dev), W.to(dev), workspace=ws)
    if check_ws:
        assert lm.workspace_error(ws) == 0
    got = out.cpu().numpy()
    ref = oracle_mod.log_mel_from_stft(stft.numpy(), W.numpy())
    return got, ref


@pytest.mark.parametrize("w", workloads.STFT_WORKLOADS[:2], ids=lambda w: w.name)
def test_small_workloads(lm, oracle_mod, w):
    stft, W = workloads.stft_workload_inputs(w)
    _compare(*_run(lm, oracle_mod, stft, W))


@pytest.mark.parametrize("shape", workloads.STFT_CORRECTNESS_SHAPES, ids=str)
def test_correctness_shapes(lm, oracle_mod, shape):
    B, F, NF, NM = shape
    stft, W = workloads.stft_inputs(B, F, NF, NM, seed=B * 1000 + F)
    _compare(*_run(lm, oracle_mod, stft, W))


@pytest.mark.parametrize("shape", [(1, 1, 201, 80), (3, 1, 201, 128), (2, 5, 1, 1), (1, 7, 3, 2), (4, 33, 64, 40),
                                   (3, 17, 401, 80), (5, 9, 129, 512), (2, 50, 2049, 128), (9, 3, 7, 300)],
                         ids=str)
@pytest.mark.parametrize("variant", ["auto", "nocluster"])
def test_edge_shapes(lm, oracle_mod, shape, variant, monkeypatch):
    # F = 1, NF = 1, NM = 1, even NF (every tile aligned), odd B*F*NF (the
    # tensor ends 8 bytes past a 16-byte boundary), NM up to 512, big NF; on
    # the variant small batches pick (one cluster per clip) and without it.
    monkeypatch.setenv("LOGMEL_K1_VARIANT", variant)
    B, F, NF, NM = shape
    stft, W = workloads.stft_inputs(B, F, NF, NM, seed=11 + B + F + NF)
    _compare(*_run(lm, oracle_mod, stft, W))


def test_silent_clip_and_floor(lm, oracle_mod):
    stft, W = workloads.stft_inputs(3, 200, 201, 128, seed=5)
    stft[1] = 0                      # silent clip: every output -1.5
    stft[2, 100:] *= 1e-6            # 120 dB drop: the floor is active
    got, ref = _run(lm, oracle_mod, stft, W)
    _compare(got, ref)
    assert np.all(got[1] == np.float32(-1.5))
    assert np.isclose(got[2].min(), got[2].max() - 2.0, atol=1e-5)


def test_zero_and_wide_filter_rows(lm, oracle_mod):
    # rows with no support (mel = 0 -> -10), and rows wider than the
    # register taps (the dense tail path): a random dense nonnegative matrix.
    stft, W = workloads.stft_inputs(2, 90, 201, 64, seed=8)
    W = W.clone()
    W[3] = 0
    W[10] = 0
    _compare(*_run(lm, oracle_mod, stft, W))
    Wd = torch.rand(64, 201, generator=torch.Generator().manual_seed(3))
    _compare(*_run(lm, oracle_mod, stft, Wd))
    Ww = workloads.triangle_filters(401, 10)  # ~80-bin triangles
    s2, _ = workloads.stft_inputs(2, 40, 401, 10, seed=9)
    _compare(*_run(lm, oracle_mod, s2, Ww))


@pytest.mark.parametrize("variant", ["resident", "twopass", "cluster"])
def test_variants_agree(lm, oracle_mod, variant, monkeypatch):
    monkeypatch.setenv("LOGMEL_K1_VARIANT", variant)
    stft, W = workloads.stft_inputs(6, 777, 201, 128, seed=21)
    _compare(*_run(lm, oracle_mod, stft, W))


def test_filters_only_four_byte_aligned(lm, oracle_mod):
    # A filter view 4 bytes into its allocation: the prologue's scalar path.
    stft, W = workloads.stft_inputs(3, 301, 201, 128, seed=31)
    Wbig = torch.zeros(W.numel() + 1)
    Wbig[1:] = W.flatten()
    Wv = Wbig[1:].view(W.shape)
    dev = torch.device("cuda")
    Wd = torch.zeros(W.numel() + 1, device=dev)
    Wd[1:] = W.flatten().to(dev)
    out = lm.log_mel_from_stft(stft.to(dev), Wd[1:].view(W.shape))
    ref = oracle_mod.log_mel_from_stft(stft.numpy(), Wv.numpy())
    _compare(out.cpu().numpy(), ref)


@pytest.mark.parametrize("shape", [(3, 301, 201, 128), (2, 100, 201, 81), (2, 50, 65, 7), (1, 40, 3, 2),
                                   (2, 90, 201, 64)], ids=str)
def test_packed_filters_match_dense(lm, oracle_mod, shape):
    # Supports and first taps from a pack, from the per-call cache, or from
    # the dense matrix: the same bits.  Odd NM exercises the pack's padding;
    # the last case has dense random rows (every band wider than 8 taps).
    B, F, NF, NM = shape
    stft, W = workloads.stft_inputs(B, F, NF, NM, seed=60 + NM)
    if NM == 64:
        W = torch.rand(NM, NF, generator=torch.Generator().manual_seed(4))
        W[5] = 0
    dev = torch.device("cuda")
    s, w = stft.to(dev), W.to(dev)
    dense = lm.log_mel_from_stft(s, w, packed=False)
    ws = torch.empty(lm.log_mel_from_stft_workspace_size(B, F, NF, NM), dtype=torch.uint8, device=dev)
    explicit = lm.log_mel_from_stft(s, w, packed=lm.pack_mel_filters(w), workspace=ws)
    assert lm.workspace_error(ws) == 0
    cached = lm.log_mel_from_stft(s, w)
    cached2 = lm.log_mel_from_stft(s, w)
    assert torch.equal(dense, explicit) and torch.equal(dense, cached) and torch.equal(dense, cached2)
    _compare(dense.cpu().numpy(), oracle_mod.log_mel_from_stft(stft.numpy(), W.numpy()))


def test_pack_follows_in_place_filter_changes(lm, oracle_mod):
    stft, W = workloads.stft_inputs(2, 120, 201, 80, seed=71)
    s, w = stft.cuda(), W.cuda()
    a = lm.log_mel_from_stft(s, w)
    w.mul_(3.0)                        # bumps the tensor's version: a new pack
    b = lm.log_mel_from_stft(s, w)
    _compare(b.cpu().numpy(), oracle_mod.log_mel_from_stft(stft.numpy(), (W * 3.0).numpy()))
    assert not torch.equal(a, b)


def test_mismatched_pack_is_reported_and_not_used(lm, oracle_mod):
    stft, W = workloads.stft_inputs(2, 100, 201, 80, seed=72)
    _, W2 = workloads.stft_inputs(1, 1, 201, 64, seed=73)
    dev = torch.device("cuda")
    s, w = stft.to(dev), W.to(dev)
    wrong = lm.pack_mel_filters(W2.to(dev))              # a pack made for 64 bands
    ws = torch.empty(lm.log_mel_from_stft_workspace_size(2, 100, 201, 80), dtype=torch.uint8, device=dev)
    out = lm.log_mel_from_stft(s, w, packed=wrong, workspace=ws)
    assert lm.workspace_error(ws) == 4                  # bit 4: the pack did not match; dense matrix used
    _compare(out.cpu().numpy(), oracle_mod.log_mel_from_stft(stft.numpy(), W.numpy()))


def test_deterministic_and_stream_aware(lm):
    stft, W = workloads.stft_inputs(4, 500, 201, 80, seed=2, device="cuda")
    a = lm.log_mel_from_stft(stft, W)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        b = lm.log_mel_from_stft(stft, W)
    s.synchronize()
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_empty_batch(lm):
    stft = torch.zeros(0, 10, 201, dtype=torch.complex64, device="cuda")
    W = torch.ones(80, 201, device="cuda")
    assert lm.log_mel_from_stft(stft, W).shape == (0, 10, 80)
    stft = torch.zeros(2, 0, 201, dtype=torch.complex64, device="cuda")
    assert lm.log_mel_from_stft(stft, W).shape == (2, 0, 80)


def test_full_size_headline_every_clip(lm, oracle_mod):
    # B=256, F=3000, NF=201, NM=128, launched exactly as the benchmark does;
    # the oracle recomputes every clip (in slices, to bound host memory).
    w = workloads.WHISPER_STFT_B256
    stft, W = workloads.stft_workload_inputs(w, device="cuda")
    ws = torch.empty(lm.log_mel_from_stft_workspace_size(w.B, w.F, w.NF, w.NM), dtype=torch.uint8, device="cuda")
    out = lm.log_mel_from_stft(stft, W, workspace=ws)
    assert lm.workspace_error(ws) == 0
    W_np = W.cpu().numpy()
    for b0 in range(0, w.B, 32):
        ref = oracle_mod.log_mel_from_stft(stft[b0:b0 + 32].cpu().numpy(), W_np)
        _compare(out[b0:b0 + 32].cpu().numpy(), ref)
    assert torch.isfinite(out).all()


@pytest.mark.parametrize("shape", [(3, 301, 201, 128), (2, 50, 64, 40), (6, 777, 201, 80), (1, 1, 1, 1),
                                   (1, 1, 2, 1), (2, 3, 5, 3)], ids=str)
@pytest.mark.parametrize("variant", ["auto", "resident", "twopass"])
def test_source_eight_bytes_off_a_boundary(lm, oracle_mod, shape, variant, monkeypatch):
    # A contiguous complex64 view one element into its allocation starts 8
    # bytes past a 16-byte boundary: the first tile's first value is copied
    # by hand.  An even element count also ends 8 bytes past a boundary.
    B, F, NF, NM = shape
    if variant == "resident" and not lm.describe_log_mel_from_stft(B, F, NF, NM)["resident"]:
        variant = "nocluster"  # a shape whose clips span too many steps for the resident mode
    monkeypatch.setenv("LOGMEL_K1_VARIANT", variant)
    stft, W = workloads.stft_inputs(B, F, NF, NM, seed=90 + B + F + NF)
    big = torch.zeros(B * F * NF + 1, dtype=torch.complex64, device="cuda")
    big[1:] = stft.flatten().cuda()
    view = big[1:].view(B, F, NF)
    assert view.data_ptr() % 16 == 8 and view.is_contiguous()
    ws = torch.empty(lm.log_mel_from_stft_workspace_size(B, F, NF, NM), dtype=torch.uint8, device="cuda")
    for packed in (None, False):
        out = lm.log_mel_from_stft(view, W.cuda(), workspace=ws, packed=packed)
        assert lm.workspace_error(ws) == 0
        _compare(out.cpu().numpy(), oracle_mod.log_mel_from_stft(stft.numpy(), W.numpy()))


def test_batch_view_of_a_larger_tensor(lm, oracle_mod):
    # stft[1:] of a [3, 301, 201] batch: 301 * 201 is odd, so the view starts
    # 8 bytes off a 16-byte boundary.
    stft, W = workloads.stft_inputs(3, 301, 201, 128, seed=93)
    s = stft.cuda()
    v = s[1:]
    assert v.data_ptr() % 16 == 8
    out = lm.log_mel_from_stft(v, W.cuda())
    _compare(out.cpu().numpy(), oracle_mod.log_mel_from_stft(stft[1:].numpy(), W.numpy()))


def test_small_batches_run_one_cluster_per_clip(lm, oracle_mod, monkeypatch):
    # B = 7 Whisper clips: the device runs every clip's cluster of 16 CTAs at
    # once, keeping 112 SMs busy, so the library picks the cluster variant;
    # the one-CTA-per-SM kernel gives the same values.  Every clip is checked
    # against the oracle.
    import dataclasses
    w = dataclasses.replace(workloads.WHISPER_STFT, B=7)
    info = lm.describe_log_mel_from_stft(w.B, w.F, w.NF, w.NM)
    assert 8 <= info["cluster"] <= 16 and info["kernels"] == 1
    stft, W = workloads.stft_workload_inputs(w, device="cuda")
    ws = torch.empty(lm.log_mel_from_stft_workspace_size(w.B, w.F, w.NF, w.NM), dtype=torch.uint8, device="cuda")
    out = lm.log_mel_from_stft(stft, W, workspace=ws)
    assert lm.workspace_error(ws) == 0
    _compare(out.cpu().numpy(), oracle_mod.log_mel_from_stft(stft.cpu().numpy(), W.cpu().numpy()))
    monkeypatch.setenv("LOGMEL_K1_VARIANT", "nocluster")
    assert lm.describe_log_mel_from_stft(w.B, w.F, w.NF, w.NM)["cluster"] == 0
    other = lm.log_mel_from_stft(stft, W, workspace=ws)
    _compare(other.cpu().numpy(), out.cpu().numpy())


@pytest.mark.parametrize("variant", ["resident", "twopass", "auto"])
def test_workspace_garbage_reuse_and_offset(lm, oracle_mod, variant, monkeypatch):
    """A result may depend neither on what the workspace held before nor on
    an earlier call with the same workspace: the workspace is filled with
    random bytes, then used by calls in a row whose clip maxima differ (the
    quieter batch would take the louder one's maxima from any stale slot),
    and once through a view 4 bytes off an 8-byte boundary."""
    monkeypatch.setenv("LOGMEL_K1_VARIANT", variant)
    dev = torch.device("cuda")
    B, F, NF, NM = 5, 700, 201, 80
    n = lm.log_mel_from_stft_workspace_size(B, F, NF, NM)
    raw = torch.empty(n + 64, dtype=torch.uint8, device=dev)
    g = torch.Generator(device="cpu").manual_seed(77)
    raw.copy_(torch.randint(1, 256, (n + 64,), dtype=torch.uint8, generator=g))
    base = raw.data_ptr() % 256
    o8 = (-base) % 256  # a 256-byte aligned start
    for k, (scale, off) in enumerate(((1.0, o8), (1e-3, o8), (10.0, o8), (1.0, o8 + 4))):
        stft, W = workloads.stft_inputs(B, F, NF, NM, seed=40 + k)
        stft = stft * scale
        ws = raw[off:off + n]
        out = lm.log_mel_from_stft(stft.to(dev), W.to(dev), workspace=ws)
        assert lm.workspace_error(ws) == 0
        _compare(out.cpu().numpy(), oracle_mod.log_mel_from_stft(stft.numpy(), W.numpy()))


@pytest.mark.parametrize("variant", ["resident", "twopass", "cluster"])
def test_floor_rewrites_in_every_variant(lm, oracle_mod, variant, monkeypatch):
    """Values below the clip floor, spread over early, middle and last tiles
    of every clip (resident mode stores every value as (v + 4) / 4 when
    computed and stores the ones below the floor again once the clip maximum
    is known, both during the stream and in the tail)."""
    monkeypatch.setenv("LOGMEL_K1_VARIANT", variant)
    B, F = (5, 700) if variant == "cluster" else (8, 3000)
    stft, W = workloads.stft_inputs(B, F, 201, 80, seed=61)
    for b in range(B):
        for f0 in range(37 * b % 120, F, 240):
            stft[b, f0:f0 + 90] *= 1e-6  # 120 dB down: far below the clip floor
    got, ref = _run(lm, oracle_mod, stft, W)
    _compare(got, ref)
    for b in range(B):
        assert np.isclose(got[b].min(), got[b].max() - 2.0, atol=1e-5)


@pytest.mark.parametrize("fpb", ["1", "2", "4", "8"])
def test_frames_per_thread_override(lm, oracle_mod, fpb, monkeypatch):
    """LOGMEL_FPB (A/B only) forces the tile height; the launch plan reports
    it and every clip still matches the oracle."""
    monkeypatch.setenv("LOGMEL_FPB", fpb)
    shape = (5, 777, 201, 80)
    info = lm.describe_log_mel_from_stft(*shape)
    assert info["frames_per_tile"] == (16 * 32 // 80) * int(fpb)
    stft, W = workloads.stft_inputs(*shape, seed=300 + int(fpb))
    _compare(*_run(lm, oracle_mod, stft, W))
