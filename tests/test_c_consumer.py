"""The C ABI from plain C: include/logmel.h compiles as C99 and as C++ with
warnings as errors (no GPU), and tests/c_abi_consumer.c -- a C program that
links liblogmel.so and the CUDA runtime and nothing else -- computes results
that match the oracle (GPU)."""
import pathlib
import shutil
import subprocess

import numpy as np
import pytest

import workloads

ROOT = pathlib.Path(__file__).resolve().parents[1]
SRC = ROOT / "tests" / "c_abi_consumer.c"
CUDA = pathlib.Path(shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc").resolve().parents[1]


def _cc(lang: str) -> list:
    if lang == "c":
        return ["gcc", "-std=c99", "-x", "c"]
    return ["g++", "-std=c++11", "-x", "c++"]


@pytest.mark.parametrize("lang", ["c", "c++"])
def test_header_compiles_standalone(lang, tmp_path):
    probe = tmp_path / "probe.c"
    probe.write_text('#include "logmel.h"\nint main(void) { return (int)LM_OK + (int)sizeof(lm_mel_params) * 0; }\n')
    cmd = _cc(lang) + ["-Wall", "-Wextra", "-Werror", "-pedantic", "-fsyntax-only", f"-I{ROOT / 'include'}",
                       str(probe)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_consumer_program_compiles():
    cmd = _cc("c") + ["-Wall", "-Wextra", "-Werror", "-fsyntax-only", f"-I{ROOT / 'include'}",
                      f"-I{CUDA / 'include'}", str(SRC)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


@pytest.mark.gpu
def test_consumer_program_matches_oracle(tmp_path, oracle_mod):
    import __graft_entry__
    __graft_entry__.build()
    from log_mel_spectrogram_gb300 import build

    exe = tmp_path / "c_abi_consumer"
    lib_dir = build.LIB.parent
    cmd = ["gcc", "-std=c99", "-O2", f"-I{ROOT / 'include'}", f"-I{CUDA / 'include'}", str(SRC), "-o", str(exe),
           f"-L{lib_dir}", "-llogmel", f"-L{CUDA / 'lib64'}", "-lcudart", f"-Wl,-rpath,{lib_dir}",
           f"-Wl,-rpath,{CUDA / 'lib64'}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr

    B, F, NF, NM, WB, WT = 5, 157, 201, 80, 2, 16000
    stft, W = workloads.stft_inputs(B, F, NF, NM, seed=91)
    wave = workloads.wave_sines(WB, WT, 16000, seed=92)
    stft.numpy().tofile(tmp_path / "stft.bin")
    W.numpy().astype(np.float32).tofile(tmp_path / "filters.bin")
    wave.numpy().astype(np.float32).tofile(tmp_path / "wave.bin")
    (tmp_path / "shape.txt").write_text(f"{B} {F} {NF} {NM} {WB} {WT}\n")
    r = subprocess.run([str(exe), str(tmp_path)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr

    got = np.fromfile(tmp_path / "out_device.bin", dtype=np.float32).reshape(B, F, NM)
    host = np.fromfile(tmp_path / "out_host.bin", dtype=np.float32).reshape(B, F, NM)
    assert np.array_equal(got, host)
    ref = oracle_mod.log_mel_from_stft(stft.numpy(), W.numpy())
    err = np.abs(got.astype(np.float64) - ref)
    assert (err <= 1e-4 + 1e-4 * np.abs(ref)).all(), err.max()

    mel = np.fromfile(tmp_path / "mel.bin", dtype=np.float32)
    n_frames = 1 + WT // 160
    mel = mel.reshape(WB, 80, n_frames)
    ref = oracle_mod.mel_spectrogram(wave.numpy(), sample_rate=16000, n_fft=400, hop_length=160, n_mels=80,
                                     f_max=8000.0, log_mel=True)
    err = np.abs(mel.astype(np.float64) - ref)
    assert (err <= 1e-4 + 1e-4 * np.abs(ref)).all(), err.max()
