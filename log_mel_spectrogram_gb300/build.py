"""Builds liblogmel.so, the library's C-ABI shared object, in-tree.

Each ``csrc/*.cu`` file is compiled by nvcc for sm_103a in parallel, then
linked into ``log_mel_spectrogram_gb300/_build/liblogmel.so``.  The build is
skipped when the library is newer than every source and header.

``build(checked=True)`` makes the bounds-checked debug variant
``_build/checked/liblogmel_checked.so`` (-DLOGMEL_CHECKED): the same sources
with every computed global-memory index tested against its buffer.
"""
from __future__ import annotations

import concurrent.futures
import os
import pathlib
import shutil
import subprocess

PKG = pathlib.Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
OUT_DIR = PKG / "_build"
LIB = OUT_DIR / "liblogmel.so"
CHECKED_DIR = OUT_DIR / "checked"
CHECKED_LIB = CHECKED_DIR / "liblogmel_checked.so"

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "--expt-relaxed-constexpr",
              f"-I{INCLUDE}", f"-I{CSRC}"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build liblogmel.so")
    return cand


def sources() -> list[pathlib.Path]:
    return sorted(CSRC.glob("*.cu"))


def _stale(lib: pathlib.Path = LIB) -> bool:
    if not lib.exists():
        return True
    t = lib.stat().st_mtime
    deps = sources() + list(CSRC.glob("*.cuh")) + list(CSRC.glob("*.h")) + list(INCLUDE.glob("*.h"))
    deps.append(pathlib.Path(__file__))
    return any(d.stat().st_mtime > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False,
          checked: bool = False) -> pathlib.Path:
    """Compile and link liblogmel.so (or, with checked=True, the bounds-checked
    variant); returns its path."""
    lib, out_dir = (CHECKED_LIB, CHECKED_DIR) if checked else (LIB, OUT_DIR)
    if not force and not _stale(lib):
        return lib
    out_dir.mkdir(parents=True, exist_ok=True)
    nvcc = _nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_verbose else []
    if checked:
        extra.append("-DLOGMEL_CHECKED")

    def compile_one(src: pathlib.Path) -> pathlib.Path:
        obj = out_dir / (src.stem + ".o")
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra, "-c", str(src), "-o", str(obj)]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src.name}:\n{r.stdout}\n{r.stderr}")
        if (verbose or ptxas_verbose) and r.stderr:
            print(r.stderr, flush=True)
        return obj

    with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, len(sources()))) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = out_dir / f"{lib.stem}.{os.getpid()}.so"
    cmd = [nvcc, *ARCH, "-shared", "-o", str(tmp), *map(str, objs)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys
    build(force="--force" in sys.argv, verbose=True, ptxas_verbose="--ptxas" in sys.argv)
    print(LIB)
