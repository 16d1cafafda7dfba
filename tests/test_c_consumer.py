"""A plain C99 program compiles against include/ssd.h, links libssd.so and
calls the ABI (calls that launch nothing: sizing, status names, and an
argument error that returns before any launch)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "mamba_ssd_chunked_scan_gb300")

SRC = r"""
#include <stdio.h>
#include "ssd.h"
int main(void) {
    ssd_params_t p = {8, 2048, 80, 64, 128, 1, 128, 0, 0, SSD_BF16};
    ssd_params_t bad = p;
    bad.chunk = 256;
    printf("%s %zu %zu %s\n", ssd_status_string(SSD_OK), ssd_fwd_workspace_size(&p),
           ssd_fwd_workspace_size(&bad),
           ssd_status_string(ssd_fwd(&bad, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0)));
    return 0;
}
"""


def test_c99_program_uses_the_abi(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    from mamba_ssd_chunked_scan_gb300 import build
    build.build()
    c = tmp_path / "consumer.c"
    c.write_text(SRC)
    exe = tmp_path / "consumer"
    subprocess.check_call(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(c),
                           "-L", PKG, "-lssd", f"-Wl,-rpath,{PKG}", "-o", str(exe)])
    out = subprocess.check_output([str(exe)], text=True).split()
    # 256 bytes (the status header) without a GPU; with one, the leftover-unit plan's piece states too
    assert out[0] == "SSD_OK" and int(out[1]) >= 256 and out[2:] == ["0", "SSD_ERR_UNSUPPORTED"]
