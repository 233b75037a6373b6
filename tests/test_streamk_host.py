"""Host logic of the stream-K partitioning, checked on the CPU: compiles
tests/streamk_check.cpp against the library's own streamk.h with g++ and runs
the brute-force checks (ranges tile the flattened positions, owners, unique
piece slots, first/last owners per unit)."""
from __future__ import annotations

import os
import subprocess

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_streamk_partition_arithmetic(tmp_path):
    exe = tmp_path / "streamk_check"
    subprocess.run(["g++", "-O2", "-std=c++17",
                    f"-I{os.path.join(ROOT, 'token_decode_attention_gb300', 'csrc')}",
                    os.path.join(ROOT, "tests", "streamk_check.cpp"), "-o", str(exe)],
                   check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    assert "passed" in r.stdout
