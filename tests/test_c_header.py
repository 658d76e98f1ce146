"""The C ABI from plain C: include/pa.h compiles as C11 (no C++ in the declarations),
a C program links libpa.so and calls the entry points that need no GPU."""

import os
import subprocess

import pytest

from paged_kv_decode_metadata_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "pa.h"

int main(void) {
  /* sizes and heuristics are host arithmetic: no device is touched */
  size_t ws = pa_workspace_bytes(32, 32, 128, 5);
  if (ws != 2 * (size_t)(32 * 32 * 5 * 4) + (size_t)32 * 32 * 5 * 128 * 4) return 1;
  if (pa_choose_splits(32, 8, 128, 64, PA_KV_BF16, 152) != 5) return 2;
  if (pa_choose_splits(64, 8, 256, 64, PA_KV_INT8, 152) != 8) return 3;
  if (pa_window_pages(4096, 1, 64, 256) != 65) return 4;
  if (strcmp(pa_status_string(PA_ERR_UNSUPPORTED), "unsupported shape") != 0) return 5;
  /* host validation returns before any launch */
  if (pa_reduce(NULL, NULL, NULL, 1, 32, 128, 4, NULL, NULL, NULL, 1) != PA_ERR_INVALID) return 6;
  if (pa_decode_step_static_scratch(NULL, NULL, NULL, 0, 0, NULL, 0, 0, 16, NULL, NULL, NULL,
                                    16, NULL, 16, NULL, NULL, NULL, NULL, NULL, PA_KV_BF16, 0,
                                    32, 8, 128, 64, 100, 4, 0.1f, NULL, NULL, NULL, 1) != PA_OK)
    return 7;
  printf("ok\n");
  return 0;
}
"""


def test_header_compiles_as_c_and_library_links(tmp_path):
    lib = build.build()
    src = tmp_path / "use_pa.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "use_pa"
    cmd = ["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
           lib, "-o", str(exe), f"-Wl,-rpath,{os.path.dirname(lib)}", "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip() == "ok", (r.returncode, r.stdout, r.stderr)
