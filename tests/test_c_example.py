"""The C example include/gdn_spec_example.c (one decode step through the ABI)
compiles against include/gdn_spec.h with warnings as errors (host only, no
link, no GPU), so the documented call sequence stays in step with the ABI."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_example_compiles(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    inc = os.path.join(ROOT, "include")
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-c", "-I", inc,
                        os.path.join(inc, "gdn_spec_example.c"), "-o", str(tmp_path / "example.o")],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
