"""The C ABI from plain C: a C99 program compiled against include/h3attn.h
alone links libh3attn.so and checks the host-side validation answers (no
GPU is touched: every call is refused, or is empty, before any launch)."""
import os
import shutil
import subprocess

import pytest

import video_dit_dense_gb300 as h3

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_plain_c_caller_links_and_sees_the_validation():
    gcc = shutil.which("gcc") or shutil.which("cc")
    if gcc is None:
        pytest.skip("no C compiler")
    h3.build()
    libdir = os.path.dirname(h3.LIB_PATH)
    out_dir = os.path.join(ROOT, "tests", "c", "_build")
    os.makedirs(out_dir, exist_ok=True)
    exe = os.path.join(out_dir, "abi_check")
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c", "abi_check.c"), "-L", libdir, "-lh3attn",
                    f"-Wl,-rpath,{libdir}", "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "abi_check: ok" in r.stdout
