"""The C ABI from plain C (CPU only): tests/c_abi/consumer.c must compile as
strict C99 against include/wtconv.h, link libwtconv.so, and see every
refusal it expects (argument validation runs on the host, so no GPU is
needed)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "memory_bound_cnn_wtconv2d_gb300")


def test_plain_c_consumer_compiles_links_and_runs(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    from memory_bound_cnn_wtconv2d_gb300 import build
    build.build()
    exe = str(tmp_path / "consumer")
    subprocess.run([cc, "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c_abi", "consumer.c"), "-L", PKG, "-lwtconv",
                    "-Wl,-rpath," + PKG, "-o", exe], check=True, capture_output=True, text=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr
