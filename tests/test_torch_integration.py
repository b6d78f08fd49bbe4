"""torch integration: custom ops, their fake (shape) implementations, the
inference-only guard, torch.compile(fullgraph=True) and CUDA-graph capture."""
import numpy as np
import pytest
import torch

import workloads


@pytest.fixture(scope="module")
def lm():
    import __graft_entry__
    __graft_entry__.build()
    import log_mel_spectrogram_gb300
    return log_mel_spectrogram_gb300


def test_fake_impls_give_shapes_without_a_gpu(lm):
    # Meta tensors dispatch to the registered fake implementations.
    stft = torch.empty(3, 301, 201, dtype=torch.complex64, device="meta")
    W = torch.empty(80, 201, device="meta")
    out = lm.log_mel_from_stft_op(stft, W)
    assert out.shape == (3, 301, 80) and out.dtype == torch.float32 and out.device.type == "meta"
    wave = torch.empty(2, 5, 480000, device="meta")
    mel = lm.mel_spectrogram_op(wave, 16000, 400, 0, 160, 0.0, 8000.0, 0, 128, 2.0, False, True, "reflect", "",
                                "htk", True, False)
    assert mel.shape == (2, 5, 128, 3001) and mel.dtype == torch.float32
    mel16 = lm.mel_spectrogram_op(torch.empty(4, 220500, device="meta", dtype=torch.int16), 22050, 1024, 0, 256,
                                  0.0, 0.0, 0, 128, 2.0, False, True, "reflect", "", "slaney", False, True)
    assert mel16.shape == (4, 128, 862) and mel16.dtype == torch.float16


def test_grad_inputs_are_rejected(lm):
    # The check comes before any device work, so it runs without a GPU.
    stft = torch.zeros(1, 2, 3, dtype=torch.complex64, requires_grad=True)
    W = torch.zeros(2, 3)
    with pytest.raises(RuntimeError, match="inference-only"):
        lm.log_mel_from_stft(stft, W)
    with pytest.raises(RuntimeError, match="inference-only"):
        lm.MelSpectrogram()(torch.zeros(1, 1000, requires_grad=True))


@pytest.mark.gpu
def test_custom_op_refuses_grad(lm):
    stft, W = workloads.stft_inputs(1, 10, 201, 80, seed=1, device="cuda")
    s = stft.clone().requires_grad_(True)
    with pytest.raises(RuntimeError, match="inference-only"):
        lm.log_mel_from_stft_op(s, W)
    with torch.no_grad():
        assert lm.log_mel_from_stft_op(s, W).shape == (1, 10, 80)


@pytest.mark.gpu
def test_custom_op_matches_and_compiles(lm):
    stft, W = workloads.stft_inputs(3, 301, 201, 128, seed=41, device="cuda")
    ref = lm.log_mel_from_stft(stft, W)
    torch.library.opcheck(lm.log_mel_from_stft_op, (stft, W), test_utils=("test_schema", "test_faketensor"))

    def f(s, w):
        return lm.log_mel_from_stft_op(s, w) * 1.0

    g = torch.compile(f, fullgraph=True)
    out = g(stft, W)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)

    x = workloads.wave_sines(2, 16000, 16000, seed=42, device="cuda")
    args = (16000, 400, 0, 160, 0.0, 8000.0, 0, 128, 2.0, False, True, "reflect", "", "htk", True, False)
    ref_w = lm.mel_spectrogram_op(x, *args)
    gw = torch.compile(lambda w: lm.mel_spectrogram_op(w, *args), fullgraph=True)
    assert torch.equal(gw(x), ref_w)


@pytest.mark.gpu
def test_cuda_graph_capture_small_batch(lm, oracle_mod):
    # The latency-bound small case (1 clip x 300 frames) captured once and
    # replayed on new inputs copied in place: each replay matches the oracle
    # within the f32 gate, and the eager call bit for bit.
    stft, W = workloads.stft_inputs(1, 300, 201, 80, seed=43, device="cuda")
    out = torch.empty(1, 300, 80, device="cuda")
    ws = torch.empty(lm.log_mel_from_stft_workspace_size(1, 300, 201, 80), dtype=torch.uint8, device="cuda")
    lm.log_mel_from_stft(stft, W, out=out, workspace=ws)  # warm-up outside capture (module load, attributes)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            lm.log_mel_from_stft(stft, W, out=out, workspace=ws)
    for seed in (44, 45):
        new, _ = workloads.stft_inputs(1, 300, 201, 80, seed=seed, device="cuda")
        stft.copy_(new)
        g.replay()
        torch.cuda.synchronize()
        ref = oracle_mod.log_mel_from_stft(new.cpu().numpy(), W.cpu().numpy()).astype(np.float64)
        got = out.cpu().numpy().astype(np.float64)
        assert np.all(np.abs(got - ref) <= 1e-4 + 1e-4 * np.abs(ref))
        assert torch.equal(out, lm.log_mel_from_stft(new, W))
