"""The C ABI from plain C: a C11 program compiled with gcc against
include/mm_moe.h and linked to libmm_moe.so calls the host-side entry points
(no GPU work): version, status strings, workspace queries and argument
rejections.  It shows the header is valid C and the library usable without
Python."""
import os
import shutil
import subprocess

import pytest

import routing_permute_mxfp8_gb300 as mm
from routing_permute_mxfp8_gb300 import build as mmbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "mm_moe.h"

int main(void) {
  int bad = 0;
  size_t n = 0;
  if (mm_version() <= 0) bad |= 1;
  if (strlen(mm_status_string(MM_OK)) == 0) bad |= 2;
  /* the DeepSeek-V3-shaped prefill workspace, and a rejected shape (H % 128) */
  if (mm_mega_moe_workspace_size(8192, 7168, 8, 256, 2048, 0, MM_WSCALE_ROWS, &n) != MM_OK || n == 0) bad |= 4;
  if (mm_mega_moe_workspace_size(64, 200, 2, 8, 128, 0, MM_WSCALE_ROWS, &n) == MM_OK) bad |= 8;
  if (mm_moe_init_routing_workspace_size(16384, 8, 256, &n) != MM_OK || n < (size_t)16384 * 8 * 4) bad |= 16;
  if (mm_moe_token_permute_out_rows(8, -3) != 5) bad |= 32;
  /* ep_world_size 2 is rejected before anything is enqueued */
  if (mm_mega_moe((void*)16, NULL, (void*)16, (void*)16, MM_DT_FLOAT32, (void*)16, (void*)16, (void*)16,
                  (void*)16, MM_DT_FP8_E4M3FN, MM_WSCALE_ROWS, NULL, NULL, NULL, NULL, MM_DT_FP8_E4M3FN, 0,
                  64, 256, 2, 8, 2, 128, 0, 4, MM_DT_FP8_E4M3FN, 0, 0, "swiglu", NULL, 0, (void*)16, NULL, NULL,
                  NULL, NULL, NULL, NULL, NULL, 0, NULL, NULL) != MM_ERR_UNSUPPORTED)
    bad |= 64;
  printf("%d\n", bad);
  return bad;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_c_program_uses_the_abi(tmp_path):
    if not os.path.exists(mm.lib_path()):
        mmbuild.build()
    lib = mm.lib_path()
    src = tmp_path / "use_abi.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "use_abi"
    libdir = os.path.dirname(lib)
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-I", INCLUDE, str(src), "-o", str(exe), lib,
                    f"-Wl,-rpath,{libdir}"], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, (r.stdout, r.stderr)
