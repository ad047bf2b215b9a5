"""The boundary is a C ABI: a plain C program (`tests/c_client.c`) that
includes only `include/credit.h` compiles with gcc, links `libcredit.so`
and gets the documented answers from entry points that need no GPU."""
import os
import shutil
import subprocess

import pytest

from dsmem_thread_block_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_plain_c_client_links_and_runs(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    lib = B.build()
    libdir = os.path.dirname(lib)
    exe = tmp_path / "c_client"
    cuda_inc = "/usr/local/cuda/include"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-I", cuda_inc, os.path.join(ROOT, "tests", "c_client.c"), "-L", libdir,
                    "-lcredit", f"-Wl,-rpath,{libdir}", "-o", str(exe)], check=True)
    env = dict(os.environ)
    env["LD_LIBRARY_PATH"] = os.pathsep.join(
        p for p in ("/usr/local/cuda/lib64", env.get("LD_LIBRARY_PATH", "")) if p)
    r = subprocess.run([str(exe)], capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode == 0, (r.stdout, r.stderr)
    version, bad = r.stdout.split()
    assert bad == "0" and version.count(".") == 2
