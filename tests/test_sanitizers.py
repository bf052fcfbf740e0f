"""Host code under AddressSanitizer and UndefinedBehaviorSanitizer (CPU only).

The oracle (oracle/cp_oracle.cpp) and libcp's host-side geometry checks
(cp_geometry.h, the plain C++ that validates every C ABI call's geometry and
sizes the host path's scratch) are compiled with g++ -fsanitize=address,undefined
-fno-sanitize-recover=all into small driver programs that exercise them; any
out-of-bounds access, overflow or other undefined behaviour aborts the driver.
"""
import shutil
import subprocess
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent
SAN = ["-fsanitize=address,undefined", "-fno-sanitize-recover=all", "-fno-omit-frame-pointer",
       "-g", "-O1", "-std=c++17", "-pthread"]

pytestmark = pytest.mark.skipif(shutil.which("g++") is None, reason="needs g++")


def _build_and_run(tmp_path, name, sources, includes=()):
    exe = tmp_path / name
    cmd = ["g++", *SAN, *[f"-I{i}" for i in includes], "-o", str(exe), *map(str, sources)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0 and "asan" in (r.stderr or "").lower():
        pytest.skip("the toolchain has no sanitizer runtime: " + r.stderr.splitlines()[-1])
    assert r.returncode == 0, r.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=600,
                         env={"ASAN_OPTIONS": "detect_leaks=1:abort_on_error=1",
                              "UBSAN_OPTIONS": "print_stacktrace=1:halt_on_error=1"})
    assert run.returncode == 0, run.stdout + run.stderr
    return run.stdout


def test_oracle_under_sanitizers(tmp_path):
    out = _build_and_run(tmp_path, "oracle_san",
                         [ROOT / "tests" / "sanitize" / "oracle_main.cpp",
                          ROOT / "oracle" / "cp_oracle.cpp"])
    assert "oracle ok" in out


def test_host_checks_under_sanitizers(tmp_path):
    out = _build_and_run(tmp_path, "host_checks_san",
                         [ROOT / "tests" / "sanitize" / "host_checks_main.cpp"],
                         includes=[ROOT / "trellis_row_decode_gb300" / "csrc"])
    assert "host checks ok" in out
