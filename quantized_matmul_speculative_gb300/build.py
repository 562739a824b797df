"""Build libqmm.so (all CUDA kernels and the C ABI) for sm_103a with nvcc.

Each (bits, group size) instantiation of the tensor-core kernels is its own
translation unit; they compile in parallel.  Objects go to ``_build/`` and the
library lands next to this file.  A rebuild happens only when a source or
header is newer than the library.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
BUILD = ROOT / "_build"
LIBRARY = PKG / "libqmm.so"

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              f"-I{INCLUDE}", f"-I{CSRC}"]

MMA_INSTANCES = [(4, 32), (4, 64), (4, 128), (2, 32), (2, 64), (2, 128), (8, 32), (8, 64), (8, 128)]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not Path(path).exists():
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libqmm")
    return path


def units():
    """(source, object, extra flags) for every translation unit."""
    out = [(CSRC / "qmm_api.cu", BUILD / "qmm_api.o", [])]
    for bits, gs in MMA_INSTANCES:
        out.append((CSRC / "qmm_mma_inst.cu", BUILD / f"qmm_mma_b{bits}_g{gs}.o",
                    [f"-DQMM_BITS={bits}", f"-DQMM_GS={gs}"]))
    return out


def _inputs():
    files = list(CSRC.glob("*.cu")) + list(CSRC.glob("*.cuh")) + list(CSRC.glob("*.h")) + list(CSRC.glob("*.inc"))
    files += list(INCLUDE.glob("*.h")) + [Path(__file__)]
    return files


def up_to_date() -> bool:
    if not LIBRARY.exists():
        return False
    lib_t = LIBRARY.stat().st_mtime
    return all(f.stat().st_mtime <= lib_t for f in _inputs())


def build(force: bool = False, verbose: bool = False, jobs: int | None = None) -> Path:
    if not force and up_to_date():
        return LIBRARY
    BUILD.mkdir(exist_ok=True)
    cc = nvcc()

    def compile_one(unit):
        src, obj, extra = unit
        cmd = [cc, *ARCH, *NVCC_FLAGS, *extra, "-c", str(src), "-o", str(obj)]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed for {obj.name}:\n{res.stderr}")
        return obj, res.stderr

    jobs = jobs or min(len(units()), os.cpu_count() or 4)
    with ThreadPoolExecutor(max_workers=jobs) as ex:
        results = list(ex.map(compile_one, units()))
    if verbose:
        for obj, log in results:
            print(f"== {obj.name}\n{log}", file=sys.stderr)
    tmp = LIBRARY.with_name(f"libqmm.{os.getpid()}.tmp.so")
    cmd = [cc, *ARCH, "-shared", "-o", str(tmp), *[str(o) for o, _ in results]]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stderr}")
    os.replace(tmp, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
