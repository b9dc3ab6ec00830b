"""libengram from plain C: tests/c/engram_c_abi.c, built with the host C compiler against
include/engram.h and the in-tree libengram.so, runs a tiny case through engram_forward and through
the four stage calls (bit-identical), checks the id buckets, the gate's masked tokens and
engram_sync_status (0, then -3 after a raw id outside the token map)."""
import os
import shutil
import subprocess

import pytest

from engram_gram_hash_02_gb300 import binding as B
from engram_gram_hash_02_gb300 import build as BUILD

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_c_caller_forward_equals_stage_calls(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no host C compiler")
    B.lib()                                           # fails loudly if the library is not built
    libdir = os.path.dirname(os.path.abspath(B.LIB_PATH))
    cuda = os.path.dirname(os.path.dirname(os.path.realpath(BUILD.nvcc())))
    exe = str(tmp_path / "engram_c_abi")
    subprocess.run([cc, "-std=c99", "-O2", "-Wall", "-I", BUILD.INCLUDE, "-I", os.path.join(cuda, "include"),
                    os.path.join(HERE, "c", "engram_c_abi.c"), "-L", libdir, "-lengram",
                    "-L", os.path.join(cuda, "lib64"), "-lcudart", f"-Wl,-rpath,{libdir}",
                    f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}", "-o", exe], check=True)
    out = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stdout + out.stderr
    assert out.stdout.strip() == "ok"
