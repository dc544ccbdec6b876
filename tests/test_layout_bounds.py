"""The tcgen05 decode kernel's shared-memory and TMEM index arithmetic,
compiled for the host and checked exhaustively (tests/layout_bounds.cpp
over csrc/decode_tc_layout.h, the functions the kernel itself calls): every
store pattern inside its region, aligned, and covering it exactly once."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "nvfp4_sparse_mla_gb300", "csrc")


def test_decode_layout_in_bounds(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    exe = str(tmp_path / "layout_bounds")
    subprocess.run([cxx, "-std=c++17", "-O1", "-Wall", "-Werror", "-I", CSRC,
                    os.path.join(ROOT, "tests", "layout_bounds.cpp"), "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "ok: 0 failures" in r.stdout


def test_layout_check_catches_a_planted_mistake(tmp_path):
    """The check is not vacuous: the same driver over a copy of the header
    whose P^T rows lose their swizzle (every row writes the same 16-byte
    column) reports failures."""
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    hdr = os.path.join(CSRC, "decode_tc_layout.h")
    src = open(hdr).read()
    good = "NVMLA_HD int pt_off(int r, int piece) { return kOffP + static_cast<int>(swz(r, piece)); }"
    assert good in src
    bad = "NVMLA_HD int pt_off(int r, int piece) { return kOffP + static_cast<int>(swz(r, 0)) + 0 * piece; }"
    d = tmp_path / "hdr"
    d.mkdir()
    (d / "decode_tc_layout.h").write_text(src.replace(good, bad))
    shutil.copy(os.path.join(CSRC, "format.h"), d / "format.h")
    exe = str(tmp_path / "layout_bounds_bad")
    subprocess.run([cxx, "-std=c++17", "-O1", "-I", str(d), os.path.join(ROOT, "tests", "layout_bounds.cpp"),
                    "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 1 and "P^T" in r.stdout, r.stdout
