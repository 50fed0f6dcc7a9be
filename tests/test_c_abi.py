"""The boundary from a plain C client: include/ea.h must compile as strict C99
and libea.so must link into a C program whose host-side calls behave as the
header states (no GPU needed)."""
import os
import shutil
import subprocess

import pytest

from sparse_head_attention_gb300 import build as ea_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_client_compiles_links_and_runs(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    lib = ea_build.build()
    exe = tmp_path / "c_abi_check"
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
           "-I" + os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c_abi_check.c"),
           "-L" + os.path.dirname(lib), "-Wl,-rpath," + os.path.dirname(lib), "-lea", "-lm",
           "-o", str(exe)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "all checks passed" in r.stdout
