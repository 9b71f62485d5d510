"""The boundary used from plain C: a C11 program includes include/nvfp4rac.h, links the built
library and calls it -- the layout helpers, the tail-path setting, and an argument error that the
library reports before any CUDA call -- so the header is valid C and the ABI needs no C++ or
Python on the caller's side.  CPU only (no device call)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "nvfp4rac.h"

int main(void)
{
    if (nvq_sf_cols(272) != 20 || nvq_fp8_sf_cols(2080) != 68) return 1;
    if (nvq_sf_bytes(129, 8) != 256 * 8) return 2;
    if (nvq_sf_offset(33, 5, 20) != (0 * 5 + 1) * 512 + 1 * 16 + 1 * 4 + 1) return 3;
    if (nvq_set_tail_path(NVQ_TAIL_ROWS) != NVQ_OK || nvq_set_tail_path(9) != NVQ_ERR_ARG) return 4;
    if (nvq_set_tail_path(NVQ_TAIL_AUTO) != NVQ_OK) return 5;
    /* K = 48 is not a multiple of 32: refused on the host, before any CUDA call */
    nvq_status s = fp8_quantize((const void*)0x100000, 64, 48, 64, 1, (uint8_t*)0x100000, 64,
                                (uint8_t*)0x100000, 8, NULL);
    if (s != NVQ_ERR_SHAPE || strncmp(nvq_last_error(), "fp8_quantize", 12) != 0) return 6;
    printf("ok\n");
    return 0;
}
"""


def test_c_program_uses_the_abi(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    from nvfp4_w4a4_quantized_quantize_gb300 import _lib
    lib = _lib.LIB_PATH
    src = tmp_path / "use_abi.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "use_abi"
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src), lib,
                    "-Wl,-rpath," + os.path.dirname(lib), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0 and out.stdout.strip() == "ok", (out.returncode, out.stdout, out.stderr)
