"""The boundary from plain C: tests/c_client/check_abi.c includes only include/moe.h,
is compiled with gcc and linked against the in-tree libmoe.so, and runs the host-side
entry points (sizing, validation, the TP slice rule) on a machine without a GPU."""
import os
import shutil
import subprocess

import pytest

from conftest import ROOT


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc not available")
def test_c_client_links_and_validates(tmp_path):
    import expert_token_dispatch_gemm_b300 as moe
    lib_dir = os.path.dirname(moe.binding._LIB_PATH)
    exe = tmp_path / "check_abi"
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c_client", "check_abi.c"), "-L", lib_dir,
                    "-lmoe", f"-Wl,-rpath,{lib_dir}", "-o", str(exe)], check=True,
                   capture_output=True, text=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "0 failure(s)" in r.stdout
