"""CPU check of the kernels' window geometry (swa::Span in swa_kernels.h, used by every kernel's
block walk and masking decision) against brute force over the visibility rule.

tests/span_check.cpp includes the library's own header, so the code under test is exactly what the
kernels compile. It is built here with the host compiler and run over Lq, Lk and windows around
the tile edges, causal and two-sided. Mutation checks: copies of the header with a planted mistake
must be rejected.
"""
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "sliding_window_flash_gb300", "csrc")
CUDA_INC = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")


def _build(tmp_path, header_dir):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None or not os.path.exists(os.path.join(CUDA_INC, "cuda_runtime.h")):
        pytest.skip("needs a host C++ compiler and the CUDA headers")
    exe = str(tmp_path / "span_check")
    subprocess.run([cxx, "-std=c++17", "-O2", f"-I{header_dir}", f"-I{CUDA_INC}",
                    os.path.join(ROOT, "tests", "span_check.cpp"), "-o", exe],
                   check=True, capture_output=True, text=True)
    return subprocess.run([exe], capture_output=True, text=True, timeout=120)


def test_span_matches_brute_force(tmp_path):
    r = _build(tmp_path, CSRC)
    assert r.returncode == 0, r.stdout + r.stderr
    assert re.match(r"ok \d+", r.stdout)


@pytest.mark.parametrize("old,new", [
    ("const int hi = q_last + off - dmin;", "const int hi = q_last + off - dmax;"),
    ("const int lo = k0 + dmin - off;", "const int lo = k0 + dmax - off;"),
    ("k0 + kBlockN <= Lk && q0 + kBlockM <= Lq", "k0 + kBlockN <= Lk"),
])
def test_span_check_rejects_planted_mistakes(tmp_path, old, new):
    src = open(os.path.join(CSRC, "swa_kernels.h")).read()
    assert src.count(old) == 1, old
    hdr = tmp_path / "hdr"
    hdr.mkdir()
    (hdr / "swa_kernels.h").write_text(src.replace(old, new))
    r = _build(tmp_path, str(hdr))
    assert r.returncode == 1 and r.stdout.startswith("mismatch"), r.stdout


def test_fastdiv_matches_division(tmp_path):
    """swa::FastDiv, which the persistent kernels use to split their tile index, against the
    built-in division and remainder (tests/fastdiv_check.cpp)."""
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None or not os.path.exists(os.path.join(CUDA_INC, "cuda_runtime.h")):
        pytest.skip("needs a host C++ compiler and the CUDA headers")
    exe = str(tmp_path / "fastdiv_check")
    subprocess.run([cxx, "-std=c++17", "-O2", f"-I{CSRC}", f"-I{CUDA_INC}",
                    os.path.join(ROOT, "tests", "fastdiv_check.cpp"), "-o", exe],
                   check=True, capture_output=True, text=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert re.match(r"ok \d+", r.stdout)
