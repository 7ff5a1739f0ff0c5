"""The C ABI from plain C: tests/c/abi_from_c.c is compiled as C11 with
warnings as errors against include/pagedattn.h, linked with the library and
run (it needs no GPU)."""
import os
import subprocess

from paged_gqa_decode_02_gb300 import build as pbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_header_and_library_work_from_plain_c(tmp_path):
    lib = pbuild.build()
    exe = tmp_path / "abi_from_c"
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c", "abi_from_c.c"),
                    "-o", str(exe), lib, "-Wl,-rpath," + os.path.dirname(lib)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("0 failure(s)") and "FAIL" not in r.stdout
