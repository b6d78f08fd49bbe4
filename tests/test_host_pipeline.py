"""GPU tests of the host-buffer entry points (lm_log_mel_from_stft_host,
lm_mel_spectrogram_host).

Clips are independent, so the chunked pipeline must reproduce the device
entry points bit for bit, whatever the chunk size, the ragged last chunk or
the reuse of the staging slots; one case is also held against the oracle.
"""
import threading

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


def _device_result(lm, stft, W, packed):
    dev = torch.device("cuda")
    out = lm.log_mel_from_stft(stft.to(dev), W.to(dev), packed=packed)
    return out.cpu()


@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
@pytest.mark.parametrize("packed", [None, False], ids=["packed", "dense"])
@pytest.mark.parametrize("chunk", [0, 1, 3], ids=lambda c: f"chunk{c}")
def test_stft_host_equals_device_path(lm, pinned, packed, chunk):
    # B = 7 with 3-clip chunks: chunks of 3, 3, 1 and a reused slot; F = 301
    # leaves a ragged tile in every clip.
    stft, W = workloads.stft_inputs(7, 301, 201, 80, seed=71)
    if pinned:
        stft = stft.pin_memory()
    Wd = W.cuda()
    got = lm.log_mel_from_stft_host(stft, Wd, packed=packed, chunk_clips=chunk)
    assert got.device.type == "cpu" and got.is_pinned() == pinned
    ref = _device_result(lm, stft, W, packed)
    assert torch.equal(got, ref)


def test_stft_host_many_chunks_against_oracle(lm, oracle_mod):
    # default chunking at the Whisper clip shape: min(32 MB / 4.8 MB per
    # clip, ceil(14 / 3)) = 5 clips per chunk, so 14 clips run as 5 + 5 + 4
    # through three slots
    stft, W = workloads.stft_inputs(14, 3000, 201, 128, seed=72)
    stft = stft.pin_memory()
    Wd = W.cuda()
    ws = torch.empty(lm.log_mel_from_stft_host_workspace_size(14, 3000, 201, 128), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty((14, 3000, 128), dtype=torch.float32).pin_memory()
    got = lm.log_mel_from_stft_host(stft, Wd, out=out, workspace=ws)
    assert got is out
    assert lm.workspace_error(ws) == 0
    assert torch.equal(got, _device_result(lm, stft, W, None))
    # two clips, from the first and the last chunk, against the oracle
    for b in (4, 13):
        ref = oracle_mod.log_mel_from_stft(stft[b:b + 1].numpy(), W.numpy())[0]
        err = np.abs(got[b].numpy().astype(np.float64) - ref)
        assert (err <= 1e-4 + 1e-4 * np.abs(ref)).all(), err.max()


def test_stft_host_is_stream_ordered(lm):
    # synchronize=False: the result is complete once the stream passes the
    # call; work enqueued before it on the same stream is seen by the copies
    stft, W = workloads.stft_inputs(5, 200, 201, 80, seed=73)
    stft = stft.pin_memory()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        Wd = torch.zeros_like(W, device="cuda")
        Wd.copy_(W.cuda(), non_blocking=True)
        got = lm.log_mel_from_stft_host(stft, Wd, chunk_clips=2, synchronize=False)
    s.synchronize()
    assert torch.equal(got, _device_result(lm, stft, W, None))


def test_stft_host_concurrent_callers(lm):
    # two host threads, each with its own stream and workspace, share the
    # library's pool of copy streams without mixing their events
    inputs = [workloads.stft_inputs(6, 250, 201, 80, seed=80 + i) for i in range(2)]
    inputs = [(s.pin_memory(), W) for s, W in inputs]
    results = [None, None]
    errors = []

    def work(i):
        try:
            torch.cuda.set_device(0)
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for _ in range(3):
                    results[i] = lm.log_mel_from_stft_host(inputs[i][0], inputs[i][1].cuda(), chunk_clips=1)
        except Exception as e:  # reported on the main thread
            errors.append(e)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i in range(2):
        assert torch.equal(results[i], _device_result(lm, inputs[i][0], inputs[i][1], None))


@pytest.mark.filterwarnings("ignore:The CUDA Graph is empty:UserWarning")  # the refusal enqueues nothing
def test_stft_host_refuses_graph_capture(lm):
    stft, W = workloads.stft_inputs(2, 50, 201, 80, seed=74)
    Wd = W.cuda()
    ws = torch.empty(lm.log_mel_from_stft_host_workspace_size(2, 50, 201, 80), dtype=torch.uint8, device="cuda")
    out = torch.empty((2, 50, 80), dtype=torch.float32)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.graph(g, stream=s):
        with pytest.raises(lm.LogmelError) as info:
            lm.log_mel_from_stft_host(stft, Wd, out=out, workspace=ws, packed=False, synchronize=False)
    assert info.value.status == 2


@pytest.mark.parametrize("case", ["whisper_f32_log", "pcm16_f16"])
@pytest.mark.parametrize("chunk", [0, 2])
def test_mel_host_equals_device_path(lm, case, chunk):
    if case == "whisper_f32_log":
        wave = workloads.wave_sines(5, 48000, 16000, seed=75)
        m = lm.MelSpectrogram(sample_rate=16000, n_fft=400, hop_length=160, n_mels=128, f_max=8000.0,
                              log_mel=True)
    else:
        wave = workloads.wave_pcm16(5, 22050, seed=76)
        m = lm.MelSpectrogram(sample_rate=22050, n_fft=1024, hop_length=256, n_mels=128, mel_scale="slaney",
                              norm="slaney", dtype=torch.float16)
    wave = wave.pin_memory()
    got = m.host(wave, chunk_clips=chunk)
    ref = m(wave.cuda()).cpu()
    torch.cuda.synchronize()
    assert got.dtype == ref.dtype and got.shape == ref.shape
    assert torch.equal(got, ref)
    m.close()
