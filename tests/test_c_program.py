"""libdsa from a plain C program: tests/c/decode_step.c runs one exact decode step through
the C ABI (indexer scores, top-k, the allocation-free sparse MLA) on device memory it
allocates itself and checks it against the fp64 oracle linked beside it.  Compiling and
linking it needs no GPU; running it does."""
import os
import subprocess

import pytest

import oracle
from sparse_attention_29_b300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _build_program(tmp_path):
    libbuild.build()
    oracle.build()
    exe = str(tmp_path / "decode_step")
    libdir = os.path.join(ROOT, "sparse_attention_29_b300")
    orcdir = os.path.join(ROOT, "oracle")
    cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-Werror", "-o", exe,
           os.path.join(ROOT, "tests", "c", "decode_step.c"),
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           "-L", libdir, "-ldsa", "-L", orcdir, "-lorc_dsa",
           "-L", os.path.join(CUDA, "lib64"), "-lcudart", "-lm",
           f"-Wl,-rpath,{libdir}:{orcdir}:{os.path.join(CUDA, 'lib64')}"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return exe


def test_c_program_compiles_and_links(tmp_path):
    assert os.path.exists(_build_program(tmp_path))


@pytest.mark.gpu
def test_c_program_decode_step_matches_oracle(tmp_path):
    exe = _build_program(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("ok")
