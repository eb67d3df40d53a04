"""Build libtaco.so in-tree with nvcc for sm_103a.

``python -m grads_taco_compress_gb300.build_lib`` or ``build()`` compiles every
``csrc/*.cu`` translation unit in parallel and links the shared library into
``grads_taco_compress_gb300/lib/``.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import pathlib
import shutil
import subprocess

PKG = pathlib.Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
OUT_DIR = PKG / "lib"
BUILD_DIR = PKG / "_build"
LIB = OUT_DIR / "libtaco.so"

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
          "-I", str(ROOT / "include"), "-I", str(CSRC)]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build libtaco")
    return cand


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"command failed ({r.returncode}): {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return r.stdout + r.stderr


def build(verbose: bool = False, extra_flags: list[str] | None = None) -> pathlib.Path:
    """Compile and link; returns the library path."""
    nvcc = _nvcc()
    BUILD_DIR.mkdir(exist_ok=True)
    OUT_DIR.mkdir(exist_ok=True)
    sources = sorted(CSRC.glob("*.cu"))
    flags = CFLAGS + (extra_flags or [])
    if verbose:
        flags = flags + ["-Xptxas", "-v"]

    def compile_one(src: pathlib.Path):
        obj = BUILD_DIR / (src.stem + ".o")
        return _run([nvcc, *ARCH, *flags, "-c", str(src), "-o", str(obj)])

    with cf.ThreadPoolExecutor(max_workers=min(8, len(sources))) as ex:
        logs = list(ex.map(compile_one, sources))
    objs = [str(BUILD_DIR / (s.stem + ".o")) for s in sources]
    tmp = OUT_DIR / "libtaco.so.tmp"
    _run([nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", str(tmp), *objs,
          "-Xlinker", "-rpath,/usr/local/cuda/lib64"])
    os.replace(tmp, LIB)
    if verbose:
        print("".join(logs))
    return LIB


if __name__ == "__main__":
    import sys
    print(build(verbose="-v" in sys.argv))
