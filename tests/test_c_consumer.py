"""The C ABI from C: compile tests/c_consumer.c with gcc against the public
header and link it to the built library; run it (host checks only, no GPU)."""

import os
import shutil
import subprocess

import pytest

from flashattention_paged_kv_fwd_b300 import binding
from flashattention_paged_kv_fwd_b300 import build as pa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")
def test_c_program_uses_the_library(tmp_path):
    pa_build.build()
    libdir = os.path.dirname(binding.library_path())
    exe = tmp_path / "c_consumer"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-o", str(exe),
                    os.path.join(ROOT, "tests", "c_consumer.c"),
                    "-I", os.path.join(ROOT, "include"), "-L", libdir, "-lpagedattn",
                    "-Wl,-rpath," + libdir],
                   check=True, capture_output=True, text=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c consumer ok" in r.stdout
