"""The C ABI from a plain C program: include/wo.h compiles as C (gcc -std=c11,
no C++), the program links against libwo.so, and the host-only entry points
(sizes, status names, the launch plan, the act-order group sort, argument
checks) behave as documented with no GPU."""
import os
import shutil
import subprocess

import pytest

from weight_only_quantized_fpa_gb300 import build as wo_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_plain_c_program_uses_the_abi(tmp_path):
    lib = wo_build.build()
    exe = tmp_path / "abi_host_calls"
    src = os.path.join(ROOT, "tests", "c", "abi_host_calls.c")
    libdir = os.path.dirname(lib)
    cc = subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                         src, "-o", str(exe), "-L", libdir, "-lwo", f"-Wl,-rpath,{libdir}"],
                        capture_output=True, text=True)
    assert cc.returncode == 0, cc.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("all ok")
