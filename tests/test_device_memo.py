"""The per-device, thread-safe memo behind the library's kernel-attribute
setup (cudaFuncSetAttribute acts on the current device only, so "already set"
must be recorded per GPU).  The memo is plain C++; this compiles a host check
against the library's own header and runs it, no GPU needed."""
import os
import subprocess

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "selective_state_space_122_b300", "csrc")


def test_device_memo_bookkeeping(tmp_path):
    exe = tmp_path / "device_memo_check"
    src = os.path.join(ROOT, "tests", "device_memo_check.cpp")
    subprocess.run(["g++", "-std=c++17", "-O1", "-pthread", "-I", CSRC, "-o", str(exe), src], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "passed" in r.stdout
