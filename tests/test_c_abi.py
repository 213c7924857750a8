"""include/gla.h compiles as plain C (gcc, -std=c99 -Wall -Werror) and a C program links
against libgla.so and gets the documented statuses back. The program makes only calls that
validation rejects, so it launches nothing (see tests/c_abi_check.c)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_program_against_the_abi(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    from chunkwise_recurrent_prefill_gb300 import build_ext
    build_ext.build()
    libdir = os.path.join(ROOT, "chunkwise_recurrent_prefill_gb300", "_build")
    exe = str(tmp_path / "c_abi_check")
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror",
                    "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c_abi_check.c"),
                    "-L", libdir, "-lgla", f"-Wl,-rpath,{libdir}", "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert "c_abi_check ok" in r.stdout
