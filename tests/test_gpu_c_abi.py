"""The boundary from plain C: tests/c_abi/ep_example.c links libep.so and the
CUDA runtime only (no PyTorch), runs layout (both kernel forms), dispatch and
combine on a hand-worked 8-token case, and checks every result against the
values worked out in its source."""
from __future__ import annotations

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu


def test_plain_c_program(ep, tmp_path):
    from combine_get_dispatch_04_gb300 import build
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = str(tmp_path / "ep_example")
    lib_dir = os.path.dirname(build.LIB)
    subprocess.run([cc, "-std=c11", "-O1", "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(cuda, "include"), os.path.join(ROOT, "tests", "c_abi",
                                                                     "ep_example.c"),
                    "-o", exe, "-L", lib_dir, "-lep", "-L", os.path.join(cuda, "lib64"),
                    "-lcudart", "-Wl,-rpath," + lib_dir, "-Wl,-rpath," + os.path.join(cuda, "lib64")],
                   check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "ok"
