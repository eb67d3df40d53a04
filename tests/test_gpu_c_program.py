"""A plain C11 program against include/taco.h and libtaco.so, on the GPU.

The program (tests/c_roundtrip.c) copies a bf16 tensor in with cudaMemcpy,
calls taco_compress and taco_decompress_reduce, copies the shard and the
bf16 output back and writes them to files; it also checks that each bad
argument is rejected with its status and writes nothing. The outputs are
compared with the oracle here.
"""

from __future__ import annotations

import os
import shutil
import subprocess
from pathlib import Path

import numpy as np
import pytest

import parity
from grads_taco_compress_gb300 import binding as tb
from grads_taco_compress_gb300 import workloads as W
from oracle import taco_oracle as O

pytestmark = pytest.mark.gpu

ROOT = Path(__file__).resolve().parent.parent
CUDA = Path(os.environ.get("CUDA_HOME", "/usr/local/cuda"))


@pytest.fixture(scope="module")
def program(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not installed")
    tb.library()                                           # raises if libtaco is not built
    lib = tb.LIB_PATH
    exe = tmp_path_factory.mktemp("c") / "c_roundtrip"
    cmd = ["gcc", "-std=c11", "-Wall", "-Werror", "-pedantic", "-I", str(ROOT / "include"),
           "-I", str(CUDA / "include"), str(ROOT / "tests" / "c_roundtrip.c"), "-o", str(exe),
           str(lib), f"-Wl,-rpath,{lib.parent}", "-L", str(CUDA / "lib64"), "-lcudart",
           f"-Wl,-rpath,{CUDA / 'lib64'}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


@pytest.mark.parametrize("name,rows", [("tiny-512x1024", 96), ("gpt2-1.5b-act", 40), ("gpt3-6.7b-grad", 24)])
def test_c_program_round_trip(program, tmp_path, name, rows):
    w = W.WORKLOADS[name]
    x = W.make_shard(w, 0, N=rows)
    (tmp_path / "x.bin").write_bytes(x.tobytes())
    prefix = tmp_path / "res"
    r = subprocess.run([str(program), str(tmp_path / "x.bin"), str(rows), str(w.h), str(w.block), str(prefix)],
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stderr
    codes = np.fromfile(f"{prefix}.codes", dtype=np.uint8).reshape(rows, w.h)
    scales = np.fromfile(f"{prefix}.scales", dtype=np.float32).reshape(rows, w.K, 2)
    out = np.fromfile(f"{prefix}.out", dtype=np.uint16).reshape(rows, w.h)
    oc, oa, os_, _ = O.compress(x, w.block)
    parity.compare_codes(codes, oc)
    parity.compare_scales(scales[..., 0], oa, "alpha")
    parity.compare_scales(scales[..., 1], os_, "s")
    want = O.decompress_reduce(oc[None], oa[None], os_[None], w.block)
    parity.compare_recon(O.bf16_bits_to_f64(out), O.bf16_bits_to_f64(want))
