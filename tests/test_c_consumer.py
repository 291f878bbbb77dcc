"""The C ABI from C: tests/c/consumer.c, a C99 program that includes only
include/treeverify.h, is compiled with the host C compiler, linked against
libtreeverify.so and run.  It exercises only calls that need no GPU, so the
header is shown to be plain C and the library usable without Python."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_program_builds_links_and_runs(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    from speculative_decoding_tree_masked_gb300 import _build, _lib
    if not os.path.exists(_lib.LIB_PATH):
        _build.build()
    libdir = os.path.dirname(_lib.LIB_PATH)
    exe = tmp_path / "consumer"
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c",
                                                                       "consumer.c"),
                    "-o", str(exe), "-L", libdir, "-ltreeverify", "-Wl,-rpath," + libdir],
                   check=True, capture_output=True, text=True)
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, run.stderr
    assert run.stdout.strip() == "ok"
