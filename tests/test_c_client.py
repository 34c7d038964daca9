"""The library is usable from plain C: include/attn.h compiles as C11 and a
C program links libattn.so (CPU test); on a GB300 the program's closed-form
checks pass (K = 0: prefix means, LSE = ln(i + 1), dQ = 0, dV suffix sums)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_client", "attn_c_client.c")
PKG = os.path.join(ROOT, "exact_tiled_attention_22_gb300")


def build_client(tmp_path):
    from exact_tiled_attention_22_gb300 import build
    build.build()
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    exe = os.path.join(str(tmp_path), "attn_c_client")
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-Werror", SRC, "-o", exe,
           f"-I{ROOT}/include", f"-I{cuda}/include", f"-L{PKG}", "-lattn",
           f"-L{cuda}/lib64", "-lcudart", "-lm", f"-Wl,-rpath,{PKG}",
           f"-Wl,-rpath,{cuda}/lib64"]
    subprocess.run(cmd, check=True)
    return exe


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_c_client_compiles_and_links(tmp_path):
    assert os.path.exists(build_client(tmp_path))


@pytest.mark.gpu
def test_c_client_closed_forms(tmp_path):
    exe = build_client(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    print(r.stdout, r.stderr)
    assert r.returncode == 0, r.stdout + r.stderr
