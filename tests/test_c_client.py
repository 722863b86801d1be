"""The C ABI from plain C: tests/c_abi_client.c includes only include/vit_attn.h, builds
with gcc -std=c99 -pedantic -Wall -Wextra -Werror, links against libvitattn.so and runs
the calls that need no GPU. Catches a header that only compiles as C++, a declaration
that does not link, and host validation that differs between C and Python callers."""
import os
import shutil
import subprocess

import pytest

import vision_encoder_varlen_gb300 as vit
from vision_encoder_varlen_gb300 import _build

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_plain_c_client(tmp_path):
    gcc = shutil.which("gcc")
    if not gcc:
        pytest.skip("gcc is missing")
    lib = _build.build()
    libdir = os.path.dirname(lib)
    exe = str(tmp_path / "c_abi_client")
    r = subprocess.run([gcc, "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror",
                        "-I", os.path.join(ROOT, "include"), os.path.join(HERE, "c_abi_client.c"),
                        "-L", libdir, "-lvitattn", f"-Wl,-rpath,{libdir}", "-o", exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    got = dict(line.split("=", 1) for line in r.stdout.splitlines())
    assert got["version"] == vit.version()
    assert got["status_bad_head_dim"] == vit.status_string(-2)
    assert int(got["ws_16x80"]) == vit.workspace_size(1024, 16, 1, 80) > 0
    assert int(got["ws_bad_d"]) == 0
    assert int(got["attn_bad_d"]) == -2                 # VIT_ERR_BAD_HEAD_DIM
    assert int(got["attn_neg_max_seqlen"]) == -14       # VIT_ERR_BAD_ARGUMENT
    assert int(got["prologue_bad_mode"]) == -14
    assert int(got["fused_empty_table"]) == -14
    assert int(got["read_status_null"]) == -1           # VIT_ERR_NULL_POINTER
