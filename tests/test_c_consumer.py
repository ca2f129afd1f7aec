"""The C ABI from C: tests/c_abi/consumer.c includes only the public header,
links libtpoverlap.so, the CPU oracle and the seeded input generator, and
checks AG+GEMM, GEMM+RS, GEMM+AR, the no-allocation entry point and argument
errors against the oracle.  Without a GPU the program is only compiled and
linked (the header is valid C and every symbol it uses resolves); on a GPU it
runs."""

import glob
import os
import subprocess

import pytest

from tensor_comm_gemm_gb300 import build as tb

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")
SOURCES = [os.path.join(HERE, "c_abi", "consumer.c"), os.path.join(ROOT, "oracle", "oracle.c"),
           os.path.join(ROOT, "tensor_comm_gemm_gb300", "gen", "tpo_synth.c")]


def cuda_lib_dirs():
    """Directories holding libcudart (lib64, or the toolkit's per-target lib)."""
    dirs = [os.path.join(CUDA, "lib64")] + glob.glob(os.path.join(CUDA, "targets", "*", "lib"))
    return [d for d in dirs if os.path.exists(os.path.join(d, "libcudart.so"))]


def build_consumer(out_dir: str) -> str:
    tb.build()
    pkg = os.path.dirname(tb.LIB)
    exe = os.path.join(out_dir, "consumer")
    libdirs = cuda_lib_dirs()
    cmd = (["gcc", "-O2", "-std=gnu11", "-Wall", "-Werror", "-ffp-contract=off", "-pthread"] + SOURCES +
           ["-I" + tb.INCLUDE, "-I" + os.path.join(CUDA, "include"), "-L" + pkg, "-ltpoverlap"] +
           ["-L" + d for d in libdirs] + ["-lcudart", "-lm", "-Wl,-rpath," + pkg] +
           ["-Wl,-rpath," + d for d in libdirs] + ["-o", exe])
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return exe


def test_consumer_compiles_and_links(tmp_path):
    assert os.access(build_consumer(str(tmp_path)), os.X_OK)


@pytest.mark.gpu
def test_consumer_runs_against_the_oracle(tmp_path, cuda_ok):
    exe = build_consumer(str(tmp_path))
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "all C ABI checks passed" in r.stdout
    assert r.stdout.count("relative Frobenius error") == 3
