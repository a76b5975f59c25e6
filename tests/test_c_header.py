"""The boundary from plain C: a C99 program that includes only
include/rope_chain.h compiles with warnings as errors, links against
librope_chain.so, and gets the version and the host-side rejections (no
GPU needed: malformed calls are refused before any CUDA call)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "rope_chain.h"

int main(void) {
    if (rc_version() <= 0) return 10;
    /* D must be 8192: refused on the host, nothing launched */
    rc_status s = rc_context_norms(NULL, 4, 4096, NULL, NULL, 1, 1e-6f, NULL, 0);
    if (s != RC_ERR_UNSUPPORTED) return 11;
    if (strlen(rc_last_error()) == 0) return 12;
    /* a NULL operand */
    s = rc_kv_project(NULL, NULL, RC_W_KN, NULL, 1, 4, 8192, 1024, NULL, 0, 0);
    if (s != RC_ERR_INVALID_ARG) return 13;
    printf("ok %d\n", rc_version());
    return 0;
}
"""


def test_header_compiles_and_links_as_c(tmp_path):
    from rope_chain_gb300 import _build
    lib = _build.build()
    cuda_home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    inc = os.path.join(cuda_home, "include")
    if not os.path.exists(os.path.join(inc, "cuda_runtime_api.h")):
        pytest.skip("no CUDA headers")
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no gcc")
    src = tmp_path / "use.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "use"
    libdir = os.path.dirname(lib)
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-I", inc, str(src), "-o", str(exe), "-L", libdir, "-lrope_chain",
                    f"-Wl,-rpath,{libdir}"], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    assert r.stdout.startswith("ok ")
