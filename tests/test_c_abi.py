"""The C ABI from C: a C99 program built against include/pagedkv.h and linked
with libpagedkv.so drives the host entry points (block pool, copy-on-write,
block tables, SplitFuse composer, workspace sizing, status strings) and checks
them against hand-worked values.  No GPU is touched."""

import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_c_program_drives_the_host_abi(tmp_path, lib):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    libdir = os.path.dirname(lib.LIB_PATH)
    exe = str(tmp_path / "c_abi_host")
    build = subprocess.run(
        [gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
         "-I", os.path.join(ROOT, "include"), os.path.join(HERE, "c_abi_host.c"),
         "-o", exe, "-L", libdir, "-lpagedkv", f"-Wl,-rpath,{libdir}"],
        capture_output=True, text=True)
    assert build.returncode == 0, build.stderr
    run = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, run.stdout + run.stderr
    assert run.stdout.strip().splitlines()[-1] == "ok"
