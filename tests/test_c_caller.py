"""The boundary from plain C: tests/c/abi_caller.c includes include/nest.h as a C11
translation unit (warnings as errors), links libnest.so and checks sizes, status names
and argument validation.  No GPU is needed: every call there is host-only or is refused
before any device work."""
import os
import shutil
import subprocess

import pytest

from nested_bit_quantized_gb300 import build as nb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_plain_c_caller(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    nb.build()
    libdir = os.path.dirname(nb.LIB)
    exe = str(tmp_path / "abi_caller")
    subprocess.run([cc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c", "abi_caller.c"), "-L", libdir, "-lnest",
                    "-Wl,-rpath," + libdir, "-o", exe], check=True)
    out = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stderr
    assert out.stdout.strip() == "ok"
