"""The library used from plain C99 (no C++ compiler, no Python, no GPU):
include/zerogr.h compiles under -std=c99 -pedantic, and a program linked
against libzerogr.so builds a host-resident index of the worked-example
catalogue and reads its statistics through the C ABI."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "generative_recommendation_constrained_gb300")


@pytest.fixture(scope="module")
def lib():
    import importlib.util
    spec = importlib.util.spec_from_file_location("_zg_build", os.path.join(PKG, "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.build()


def test_plain_c_program(lib, tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if not cc:
        pytest.skip("no C compiler")
    exe = str(tmp_path / "abi_host")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                        os.path.join(ROOT, "tests", "c", "abi_host.c"), "-I", os.path.join(ROOT, "include"),
                        "-L", PKG, "-lzerogr", f"-Wl,-rpath,{PKG}", "-o", exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stdout + out.stderr
    lines = dict(l.split(" ", 1) for l in out.stdout.strip().splitlines())
    assert "sm_103a" in lines["version"]
    f = lines["unique"].split()
    stats = dict(zip(["unique"] + f[1::2], [f[0]] + f[2::2]))
    # five distinct items; step 3 rows are the four distinct 2-prefixes, five
    # entries, and the prefix 3-5 has the two children 1 and 4
    assert stats == {"unique": "5", "rows3": "4", "nnz3": "5", "maxfan3": "2", "bytes3": stats["bytes3"]}
    assert int(stats["bytes3"]) >= 16 + 4 * 5 + 2 * 5
    assert lines["bad"] == "token status 1 message set"
