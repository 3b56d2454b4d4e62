"""The header is plain C: a C99 program (tests/abi_consumer.c) compiles against it with
-pedantic -Werror, links against the library and sees the documented host-side statuses
(CPU only; no call reaches a kernel)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIBDIR = os.path.join(ROOT, "mla_flash_attention_gb300")


@pytest.fixture(scope="module")
def built_lib():
    if not os.path.exists(os.path.join(LIBDIR, "libmla_gb300.so")):
        from mla_flash_attention_gb300 import build

        build.build()
    return LIBDIR


def test_c99_consumer_compiles_links_and_sees_the_documented_statuses(built_lib, tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = str(tmp_path / "abi_consumer")
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                    "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "abi_consumer.c"),
                    "-L", built_lib, "-lmla_gb300", "-Wl,-rpath," + built_lib, "-o", exe],
                   check=True, capture_output=True, text=True)
    r = subprocess.run([exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
