"""The C ABI used from C: include/gemm_f32.h compiles as strict C99 and C++,
and an example program (tests/c_api/abi_example.c) built against
libgemm_f32.so computes exact integer products in every mode."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")
EXAMPLE = os.path.join(ROOT, "tests", "c_api", "abi_example.c")
CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _cc():
    cc = shutil.which("gcc") or shutil.which("cc")
    if not cc:
        pytest.skip("no C compiler")
    return cc


def test_header_compiles_as_c99_and_cxx(tmp_path):
    src = tmp_path / "h.c"
    src.write_text('#include "gemm_f32.h"\n'
                   'int (*entry)(const float*, const float*, float*, int, int, int, gemm_f32_stream_t) = gemm_f32;\n'
                   'int main(void) { return entry == 0 ? GEMM_F32_EINVAL : GEMM_F32_OK; }\n')
    subprocess.run([_cc(), "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", INCLUDE,
                    "-I", os.path.join(CUDA_HOME, "include"), "-c", str(src), "-o",
                    str(tmp_path / "h.o")], check=True)
    cxx = shutil.which("g++")
    if cxx:
        srcx = tmp_path / "h.cc"
        srcx.write_text(src.read_text())
        subprocess.run([cxx, "-std=c++17", "-Wall", "-Wextra", "-Werror", "-I", INCLUDE, "-c",
                        str(srcx), "-o", str(tmp_path / "hx.o")], check=True)


def test_example_compiles_as_c99(tmp_path):
    subprocess.run([_cc(), "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", INCLUDE, "-I",
                    os.path.join(CUDA_HOME, "include"), "-c", EXAMPLE, "-o",
                    str(tmp_path / "ex.o")], check=True)


@pytest.mark.gpu
def test_example_runs_against_the_library(tmp_path):
    from accelerator_row_major_gb300 import build as build_mod
    build_mod.build()
    lib_dir = os.path.dirname(build_mod.LIB)
    exe = tmp_path / "abi_example"
    subprocess.run([_cc(), "-std=c99", "-O2", "-I", INCLUDE, "-I", os.path.join(CUDA_HOME, "include"),
                    EXAMPLE, "-o", str(exe), "-L", lib_dir, "-lgemm_f32",
                    "-L", os.path.join(CUDA_HOME, "lib64"), "-lcudart",
                    "-Wl,-rpath," + lib_dir + ":" + os.path.join(CUDA_HOME, "lib64")], check=True)
    out = subprocess.run([str(exe), "300", "200", "260"], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr
    lines = out.stdout.split()
    assert lines.count("ok") == 4, out.stdout
    assert "tc_gemm_kernel" in out.stdout and "ffma_gemm_kernel" in out.stdout
