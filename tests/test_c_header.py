"""include/taco.h is a C header: a C11 file that includes it and takes the
address of every declared entry point compiles with gcc and links against
libtaco.so (every declaration has a definition with C linkage). The library
is built first where it is missing (nvcc cross-compiles without a GPU).
tests/test_gpu_c_program.py runs such a program on a GPU."""

import re
import shutil
import subprocess
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent
HEADER = ROOT / "include" / "taco.h"
LIB = ROOT / "grads_taco_compress_gb300" / "lib" / "libtaco.so"


def _declared():
    text = re.sub(r"/\*.*?\*/", "", HEADER.read_text(), flags=re.S)
    return sorted(set(re.findall(r"\b(taco_[a-z0-9_]+)\s*\(", text)))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc not installed")
def test_header_compiles_as_c_and_links(tmp_path):
    names = _declared()
    assert len(names) >= 20
    src = tmp_path / "uses_taco.c"
    body = "\n".join(f"  (void (*)(void))&{n}," for n in names)
    src.write_text(
        '#include "taco.h"\n#include <stddef.h>\n'
        f"void (*taco_entry_points[])(void) = {{\n{body}\n}};\n"
        "int main(void) { return taco_abi_version() > 0 ? 0 : 1; }\n")
    obj = tmp_path / "uses_taco.o"
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-pedantic", "-I", str(ROOT / "include"),
                    "-c", str(src), "-o", str(obj)], check=True, capture_output=True, text=True)
    if not LIB.exists():
        from grads_taco_compress_gb300 import build_lib
        build_lib.build()
    exe = tmp_path / "uses_taco"
    r = subprocess.run(["gcc", str(obj), "-o", str(exe), str(LIB), f"-Wl,-rpath,{LIB.parent}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
