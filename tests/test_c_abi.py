"""The C ABI from a plain C99 program (tests/c_abi_smoke.c): it includes only
the public header and links only the library, with no CUDA toolkit of its
own.  Host-only calls on the CPU; a GEMM on host buffers on a GPU."""
import os
import shutil
import subprocess

import pytest
import torch

import dense_gemm_epilogue_persistent_gb300 as G

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
PKG = os.path.dirname(G.LIB_PATH)


@pytest.fixture(scope="module")
def program(tmp_path_factory):
    cc = shutil.which("gcc") or shutil.which("cc")
    if not cc:
        pytest.skip("no C compiler")
    if not os.path.exists(G.LIB_PATH):
        pytest.skip("library not built")
    exe = str(tmp_path_factory.mktemp("c_abi") / "c_abi_smoke")
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-O1",
                    "-I", os.path.join(ROOT, "include"), os.path.join(HERE, "c_abi_smoke.c"),
                    "-L", PKG, "-lgemm_gb300", "-Wl,-rpath," + PKG, "-o", exe], check=True)
    return exe


def test_c_program_host_only_calls(program):
    r = subprocess.run([program, "check"], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "check: OK" in r.stdout


@pytest.mark.gpu
def test_c_program_runs_a_gemm_on_host_buffers(program):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    r = subprocess.run([program, "run"], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "bit-exact" in r.stdout
