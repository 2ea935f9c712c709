"""The C ABI from C (CPU only): tests/c/abi_host_check.c includes the public
header as C11, links libconvbnsilu.so, and calls the entry points that touch no
GPU -- output sizes, plans with and without overrides, argument checks, status
strings.  Catches C++ leaking into the header and ABI mismatches that a ctypes
binding would not notice (struct layouts are compiled from the header here).
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib_path():
    from conv2d_batchnorm_silu_gb300 import _build
    return _build.build()


def test_header_compiles_as_c_and_host_entries_answer(lib_path, tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = tmp_path / "abi_host_check"
    lib_dir = os.path.dirname(lib_path)
    cmd = [cc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic",
           "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c", "abi_host_check.c"),
           "-L", lib_dir, "-lconvbnsilu", f"-Wl,-rpath,{lib_dir}", "-o", str(exe)]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, run.stderr
    assert "c abi ok" in run.stdout
