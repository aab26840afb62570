"""CPU test of the per-context address cache used by decode_attn_run_static: compiled with the
host compiler from the library's own header and run (no CUDA needed)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_scratch_address_cache_keys_on_the_context(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    exe = tmp_path / "scratch_cache"
    subprocess.run([cxx, "-std=c++17", "-O1", "-Wall", "-Werror",
                    "-I" + os.path.join(ROOT, "decode_attention_attn_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "c_scratch_cache.cpp"), "-o", str(exe)],
                   check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
