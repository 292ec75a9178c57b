"""The C-ABI from plain C99 (no Python, no PyTorch): compile the example host program
against include/flux3.h and libflux3.so with gcc and run it (host-side paths only, no GPU)."""
import os
import shutil
import subprocess

import pytest

from flow_matching_image_flux3_b300 import build as fbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "flow_matching_image_flux3_b300")


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")
def test_c_host_program(tmp_path):
    fbuild.build()
    exe = str(tmp_path / "c_host")
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           os.path.join(PKG, "examples", "c_host.c"), "-L", PKG, "-lflux3", f"-Wl,-rpath,{PKG}", "-o", exe]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    out = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stdout + out.stderr
    assert "all checks passed" in out.stdout
