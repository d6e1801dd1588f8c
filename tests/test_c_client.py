"""The C ABI from plain C (tests/host/c_client.c): a C11 program that includes
include/repops.h, links librepops.so and the CUDA runtime, and calls the
GEMM (row-major and transposed B), the contributor sort, the mean + SGD and
the Merkle commitment with device memory from cudaMalloc -- no Python or
PyTorch in the caller.  On the CPU it must compile and link; on a GPU it must
print "ok" and a Merkle root equal to the oracle's root of the expected C."""
import os
import shutil
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HERE = os.path.dirname(os.path.abspath(__file__))
CUDA = os.environ.get("CUDA_HOME") or "/usr/local/cuda"


def build_client(out_dir: str) -> str:
    from verifiable_repops_gemm_gb300 import build
    lib = build.build()
    cc = shutil.which("gcc") or shutil.which("cc")
    if not cc or not os.path.isdir(os.path.join(CUDA, "include")):
        pytest.skip("no C compiler or CUDA headers")
    exe = os.path.join(out_dir, "c_client")
    libdir = os.path.dirname(lib)
    cudalib = next((d for d in (os.path.join(CUDA, "lib64"), os.path.join(CUDA, "lib"))
                    if os.path.isdir(d)), os.path.join(CUDA, "lib64"))
    cmd = [cc, "-std=c11", "-O2", "-Wall", "-ffp-contract=off",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           os.path.join(HERE, "host", "c_client.c"), "-o", exe,
           "-L", libdir, "-lrepops", "-Wl,-rpath," + libdir,
           "-L", cudalib, "-lcudart", "-Wl,-rpath," + cudalib]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "warning" not in r.stderr, r.stderr
    return exe


def test_c_client_compiles_and_links(tmp_path):
    assert os.path.exists(build_client(str(tmp_path)))


@pytest.mark.gpu
def test_c_client_runs_bit_exact(rp, orc, tmp_path):
    exe = build_client(str(tmp_path))
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    words = r.stdout.split()
    assert words[0] == "ok", r.stdout
    # the same integer-valued operands as the C program: every sum exact
    M, N, K = 300, 200, 777
    i = np.arange(M)[:, None]
    k = np.arange(K)[None, :]
    A = ((i * 7 + k * 13 + 1) % 9 - 4).astype(np.int64)
    kk = np.arange(K)[:, None]
    j = np.arange(N)[None, :]
    B = ((kk * 7 + j * 13 + 2) % 9 - 4).astype(np.int64)
    C = (A @ B).astype(np.float32)
    assert words[1] == orc.merkle_root(C, 4096).hex()
