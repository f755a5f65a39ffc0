"""The C ABI used from plain C (no GPU): tests/c_abi/abi_from_c.c compiles as
C99 with warnings as errors against include/la.h, links against the in-tree
library and runs its host-only checks (layout of la_dims, status strings,
argument validation, empty problems, workspace sizes)."""
import os
import shutil
import subprocess

import pytest

from linear_attention_head_gb300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_abi", "abi_from_c.c")


def test_c_program_uses_the_abi(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    libbuild.build()
    libdir = os.path.dirname(libbuild.LIB)
    exe = str(tmp_path / "abi_from_c")
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                    "-I", os.path.join(ROOT, "include"), SRC, "-L", libdir, "-llagb300",
                    "-Wl,-rpath," + libdir, "-o", exe], check=True, capture_output=True, text=True)
    run = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, run.stderr
    assert "all C ABI checks passed" in run.stdout
