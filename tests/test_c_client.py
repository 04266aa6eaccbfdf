"""The boundary from plain C: a C99 program that includes only include/w4.h
and links libw4gb300.so, the way a C caller would ("Fused int4 and int8
dequantize-matmul in C", section 4: the interface is a C header).  It runs
the calls that need no device -- version, status strings, workspace sizes --
and argument checks that return before any launch, and checks that y is left
untouched.  The header must also compile as C++ (extern "C")."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")

PROGRAM = r"""
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "w4.h"

int main(void) {
    float y[2] = {7.0f, 7.0f};
    if (w4_version() < 100) return 1;
    if (strncmp(w4_status_string(W4_ESHAPE), "W4_ESHAPE", 9) != 0) return 2;
    /* decode needs no scratch; prefill needs the f16 image of the codes; absurd shapes: SIZE_MAX */
    if (w4_workspace_bytes(W4_OP_LINEAR_Q4, 1, 2048, 2048, 0) != 0) return 3;
    if (w4_workspace_bytes(W4_OP_LINEAR_Q4, 2048, 2048, 2048, 0) != (size_t)2048 * 2048 * 2) return 4;
    if (w4_workspace_bytes(W4_OP_LINEAR_Q4, (int64_t)1 << 31, 1, 1, 0) != SIZE_MAX) return 5;
    /* the error order: a negative dimension, then the shape, then empty dims, then pointers */
    if (w4_linear_q4(NULL, NULL, NULL, NULL, y, -1, 2, 4, W4_LAYOUT_ROWMAJOR, NULL, 0, 0, NULL) != W4_EINVAL)
        return 6;
    if (w4_linear_w4a16_group(NULL, NULL, NULL, y, 1, 2, 4, 3, W4_LAYOUT_ROWMAJOR, NULL, 0, 0, NULL) != W4_ESHAPE)
        return 7;
    if (w4_linear_q4(NULL, NULL, NULL, NULL, y, 0, 2, 4, W4_LAYOUT_ROWMAJOR, NULL, 0, 0, NULL) != W4_OK) return 8;
    if (w4_linear_q4(NULL, NULL, NULL, NULL, y, 1, 2, 4, W4_LAYOUT_ROWMAJOR, NULL, 0, 0, NULL) != W4_EINVAL)
        return 9;
    if (w4_linear_q4(NULL, NULL, NULL, NULL, y, 1, 2, 4, 7, NULL, 0, 0, NULL) != W4_EINVAL) return 10;
    if (y[0] != 7.0f || y[1] != 7.0f) return 11;
    puts("c-abi ok");
    return 0;
}
"""


@pytest.fixture(scope="module")
def libdir():
    from w4a16_int4_quantized_gb300 import build
    return os.path.dirname(build.build())


def test_header_compiles_as_cxx():
    cxx = shutil.which("g++") or pytest.skip("no C++ compiler")
    r = subprocess.run([cxx, "-std=c++17", "-Wall", "-Werror", "-fsyntax-only", "-x", "c++", "-I", INCLUDE, "-"],
                       input='#include "w4.h"\n', capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_c99_client_links_and_runs(libdir, tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc") or pytest.skip("no C compiler")
    src = tmp_path / "client.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "client"
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", INCLUDE, str(src),
                        "-L", libdir, "-lw4gb300", f"-Wl,-rpath,{libdir}", "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0 and run.stdout.strip() == "c-abi ok", (run.returncode, run.stdout, run.stderr)
