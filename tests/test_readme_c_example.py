"""The C example in README.md compiles against include/gdn_spec.h (host only,
no link, no GPU), so the documented call sequence stays in step with the ABI."""
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_readme_c_example_compiles(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    text = open(os.path.join(ROOT, "README.md")).read()
    code = re.search(r"```c\n(.*?)```", text, re.S).group(1)
    src = tmp_path / "example.c"
    src.write_text(
        "#include <stdio.h>\n#include <stdint.h>\n#include \"gdn_spec.h\"\n"
        "int step(int32_t slots, float *ckpt, void *rawv, void *rawk, float *ring_g,\n"
        "         float *ring_beta, int32_t *write_pos, int32_t *cache_base, int32_t *is_flush,\n"
        "         uint32_t *status, const int32_t *slot_idx, int32_t B, const void *q,\n"
        "         const void *k, const void *v, const void *a, const void *b,\n"
        "         const float *A_log, const float *dt_bias, void *out,\n"
        "         const int32_t *accept_len, void *stream) {\n" + code + "    return rc;\n}\n")
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-c", "-I", os.path.join(ROOT, "include"),
                        str(src), "-o", str(tmp_path / "example.o")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
