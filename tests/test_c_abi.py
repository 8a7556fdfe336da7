"""The C ABI from plain C: ``tests/c_abi_check.c`` is compiled as C99 against
``include/tq.h`` (so the header must be valid C), linked against libtq.so and
run. It calls host-side entry points only, so no GPU is needed."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_plain_c_caller(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    from turboquant_paged_kv_gb300 import build
    lib = build.build()
    exe = tmp_path / "c_abi_check"
    subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c_abi_check.c"), "-o", str(exe), lib,
                    "-Wl,-rpath," + os.path.dirname(lib), "-lm"], check=True)
    out = subprocess.run([str(exe)], stdout=subprocess.PIPE, text=True)
    assert out.returncode == 0, out.stdout
    assert out.stdout.strip().endswith("ALL OK")
    assert "slot 134 tile 2144 block 17152" in out.stdout
