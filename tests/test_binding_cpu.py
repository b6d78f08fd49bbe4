"""The Python binding's argument checks, which reject bad calls before any
CUDA call is made, so they run on a machine without a GPU."""
import pytest
import torch


@pytest.fixture(scope="module")
def lm():
    from log_mel_spectrogram_gb300 import build
    build.build()
    import log_mel_spectrogram_gb300
    return log_mel_spectrogram_gb300


def test_device_entry_points_refuse_host_tensors(lm):
    stft = torch.zeros(1, 4, 201, dtype=torch.complex64)
    W = torch.zeros(80, 201)
    with pytest.raises(ValueError, match="CUDA tensor"):
        lm.log_mel_from_stft(stft, W)
    with pytest.raises(ValueError, match="CUDA tensor"):
        lm.pack_mel_filters(W)
    m = lm.MelSpectrogram(n_fft=400, hop_length=160, n_mels=80)
    with pytest.raises(ValueError, match="CUDA tensor"):
        m(torch.zeros(1, 1000))


def test_host_entry_points_check_their_arguments(lm):
    stft = torch.zeros(2, 4, 201, dtype=torch.complex64)
    W = torch.zeros(80, 201)
    # the filters stay on the device
    with pytest.raises(ValueError, match="CUDA tensor"):
        lm.log_mel_from_stft_host(stft, W)
    # the batch must be a contiguous CPU tensor
    with pytest.raises(ValueError, match="contiguous"):
        lm.log_mel_from_stft_host(stft.transpose(0, 1), W)
    m = lm.MelSpectrogram(n_fft=400, hop_length=160, n_mels=80)
    with pytest.raises(ValueError, match="float32 or int16"):
        m.host(torch.zeros(1, 1000, dtype=torch.float64))
    with pytest.raises(ValueError, match="contiguous"):
        m.host(torch.zeros(1000, 2).t())


def test_inference_only(lm):
    W = torch.zeros(80, 201, requires_grad=True)
    stft = torch.zeros(1, 4, 201, dtype=torch.complex64)
    with pytest.raises(RuntimeError, match="inference-only"):
        lm.log_mel_from_stft(stft, W)
    with pytest.raises(RuntimeError, match="inference-only"):
        lm.log_mel_from_stft_host(stft, W)
    with torch.no_grad():  # allowed under no_grad; then the device check fires
        with pytest.raises(ValueError, match="CUDA tensor"):
            lm.log_mel_from_stft(stft, W)


def test_output_dtype_choice(lm):
    with pytest.raises(ValueError, match="float32 or torch.float16"):
        lm.MelSpectrogram(dtype=torch.float64)


def test_host_workspace_size_matches_the_c_abi(lm):
    import ctypes
    from log_mel_spectrogram_gb300 import _native
    n = ctypes.c_size_t()
    assert _native.lib().lm_log_mel_from_stft_host_workspace_size(14, 3000, 201, 128, 0, ctypes.byref(n)) == 0
    assert lm.log_mel_from_stft_host_workspace_size(14, 3000, 201, 128) == n.value
    # five clips per chunk (min(32 MB / 4.8 MB, ceil(14 / 3))): three slots of five
    in_clip, out_clip = 3000 * 201 * 8, 3000 * 128 * 4
    assert 3 * 5 * (in_clip + out_clip) <= n.value < 3 * 6 * (in_clip + out_clip)
    with pytest.raises(lm.LogmelError):
        lm.log_mel_from_stft_host_workspace_size(2, 10, 201, 600)
