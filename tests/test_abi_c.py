"""The boundary from a plain C client: include/moe.h compiles as C11 and as
C++17 with warnings as errors, and tests/abi_c/moe_abi_check.c, linked
against libmoe.so, passes its host-only checks (no GPU)."""
import os
import shutil
import subprocess

import pytest

from persistent_megakernel_sm_gb300 import build as cuda_build
from persistent_megakernel_sm_gb300.binding import LIB_PATH

HERE = os.path.dirname(os.path.abspath(__file__))
REPO = os.path.dirname(HERE)
INCLUDE = os.path.join(REPO, "include")
SRC = os.path.join(HERE, "abi_c", "moe_abi_check.c")

pytestmark = pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")


def test_header_compiles_as_c_and_cxx(tmp_path):
    tu = tmp_path / "tu.c"
    tu.write_text('#include "moe.h"\nint moe_header_only_tu(void) { return MOE_OK; }\n')
    for cmd in (["gcc", "-std=c11", "-Wall", "-Wextra", "-pedantic", "-Werror"],
                ["g++", "-std=c++17", "-Wall", "-Wextra", "-pedantic", "-Werror", "-x", "c++"]):
        if shutil.which(cmd[0]) is None:
            continue
        r = subprocess.run(cmd + ["-I", INCLUDE, "-c", str(tu), "-o", str(tmp_path / "tu.o")],
                           capture_output=True, text=True)
        assert r.returncode == 0, r.stderr


def test_c_client_host_checks(tmp_path):
    cuda_build.build()
    exe = tmp_path / "moe_abi_check"
    lib_dir = os.path.dirname(LIB_PATH)
    r = subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-pedantic", "-Werror",
                        "-I", INCLUDE, SRC, "-o", str(exe), "-L", lib_dir, "-lmoe",
                        f"-Wl,-rpath,{lib_dir}", "-lpthread"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    # no device is needed: every call made here returns before any CUDA call
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([str(exe)], capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("0 failures"), r.stdout
