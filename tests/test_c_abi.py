"""The C ABI from plain C: include/fa.h compiles as strict C99, and a C program
(tests/c_abi/c_abi_example.c) links libfa.so, runs a forward and a backward and
checks them against the fp64 oracle's C entry points."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")
EXAMPLE = os.path.join(ROOT, "tests", "c_abi", "c_abi_example.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")

pytestmark = pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")


def test_header_is_strict_c99(tmp_path):
    src = tmp_path / "h.c"
    src.write_text('#include "fa.h"\nint main(void) { return fa_status_string(FA_OK) == 0; }\n')
    subprocess.run(["gcc", "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror", "-fsyntax-only",
                    "-I", INCLUDE, str(src)], check=True)


def test_c_example_compiles():
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-fsyntax-only", "-I", INCLUDE,
                    "-I", os.path.join(CUDA, "include"), EXAMPLE], check=True)


@pytest.mark.gpu
def test_c_example_runs(tmp_path):
    import oracle
    from tiled_attention_03_gb300.build import LIB, build_library
    build_library()
    olib = oracle.build()
    exe = tmp_path / "c_abi_example"
    libdirs = [os.path.dirname(LIB), os.path.dirname(olib), os.path.join(CUDA, "lib64")]
    cmd = ["gcc", "-std=c99", "-O2", EXAMPLE, "-I", INCLUDE, "-I", os.path.join(CUDA, "include")]
    for d in libdirs:
        cmd += ["-L", d, f"-Wl,-rpath,{d}"]
    cmd += ["-lfa", "-loracle", "-lcudart", "-lm", "-o", str(exe)]
    subprocess.run(cmd, check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c_abi_example: ok" in r.stdout
