"""fa_check_device's reporting logic, on the CPU: the device error words it reads
back (the stream workspace's, and the fixed scratch of fa_bwd_noalloc) map to one
fa_status, and a timeout recorded by either entry point is reported as
FA_ERR_TIMEOUT.  The header that holds this logic is plain C++, compiled here with
g++ into a small check program (tests/c/error_words_check.cpp)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_error_words_map_to_status(tmp_path):
    if shutil.which("g++") is None:
        pytest.skip("g++ not available")
    exe = tmp_path / "error_words_check"
    cmd = ["g++", "-std=c++17", "-O1", "-Wall", "-Werror",
           os.path.join(ROOT, "tests", "c", "error_words_check.cpp"),
           "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(ROOT, "flashattention_backward_preprocess_gb300", "csrc"),
           "-o", str(exe)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
