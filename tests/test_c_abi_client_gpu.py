"""The C ABI from plain C: tests/c_abi_client.c, built with gcc against
libdattn.so and the oracle, runs a decode through both workspace flavours and
checks it against the oracle with no Python binding and no torch involved."""
from __future__ import annotations

import os
import subprocess

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_client_decodes_through_the_abi(tmp_path):
    from oracle import build as oracle_build
    from token_decode_attention_gb300 import build as lib_build
    lib = lib_build.build()
    olib = oracle_build.build()
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    exe = str(tmp_path / "c_abi_client")
    cmd = ["gcc", "-O2", "-std=c11", os.path.join(ROOT, "tests", "c_abi_client.c"), "-o", exe,
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
           lib, olib, "-L", os.path.join(cuda, "lib64"), "-lcudart", "-lm", "-fopenmp",
           "-Wl,-rpath," + os.path.dirname(lib) + ":" + os.path.dirname(olib) + ":" +
           os.path.join(cuda, "lib64")]
    subprocess.run(cmd, check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip() == "ok"
