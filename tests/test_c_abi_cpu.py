"""The C ABI from plain C: include/fi.h compiles as strict C99 and a C
program linked against libfi.so plans a batch, reads its summary and gets
the documented status codes back (host-side paths only; no kernel runs)."""
import os
import shutil
import subprocess

import pytest

from ._gpu import ensure_built

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIB_DIR = os.path.join(ROOT, "paged_kv_attention_27_gb300", "lib")


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")
def test_c_program_plans_through_the_abi(tmp_path):
    ensure_built()
    exe = str(tmp_path / "plan_from_c")
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c_abi", "plan_from_c.c"),
                    "-L", LIB_DIR, "-lfi", f"-Wl,-rpath,{LIB_DIR}", "-o", exe],
                   check=True, capture_output=True, text=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    got = dict(zip(*[iter(r.stdout.split())] * 2))
    # 1 + 17 + 64 + 100 keys; one chunk per (request, kv head) at these lengths
    assert got == {"total_kv_tokens": "182", "items": "8", "windowed_kv_tokens": "182",
                   "windowed_items": "8", "ws_ok": "1"}
