"""The boundary from C: a C99 program compiled against include/moe.h (strict,
pedantic, warnings as errors) links libmoe.so and calls the host-side entry
points -- version and status strings, workspace sizes and layout, and a
forward and a multi-step host forward with NULL arguments, which must be
rejected before any CUDA call."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "precision_moe_grouped_gb300")

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "moe.h"

int main(void) {
  moe_shape s;
  moe_ws_layout L;
  size_t bytes;
  int32_t rc;
  s.num_tokens = 4096; s.num_experts = 256; s.top_k = 8; s.hidden = 7168; s.inter = 2048;
  bytes = moe_workspace_size(&s, MOE_W4A8_MXFP4_FP8);
  if (bytes == 0) { printf("size 0\n"); return 1; }
  rc = moe_workspace_layout(&s, MOE_W4A8_MXFP4_FP8, &L);
  if (rc != MOE_OK || (size_t)L.total != bytes) { printf("layout %d\n", (int)rc); return 2; }
  if (strlen(moe_version()) == 0) return 3;
  if (strcmp(moe_status_string(MOE_ERR_INVALID_ARG), "invalid argument") != 0) return 4;
  rc = moe_forward(&s, MOE_W4A8_MXFP4_FP8, NULL, NULL, NULL, NULL, NULL, NULL, NULL,
                   NULL, 0, NULL);
  if (rc != MOE_ERR_INVALID_ARG) { printf("forward %d\n", (int)rc); return 5; }
  if (moe_steps_workspace_size(&s, MOE_W4A8_MXFP4_FP8) <= bytes) return 7;
  rc = moe_forward_host_steps(&s, MOE_W4A8_MXFP4_FP8, 2, NULL, NULL, NULL, NULL, NULL, NULL,
                              NULL, NULL, 0, NULL, NULL);
  if (rc != MOE_ERR_INVALID_ARG) { printf("steps %d\n", (int)rc); return 8; }
  s.num_experts = 0;
  if (moe_workspace_size(&s, MOE_W4A8_MXFP4_FP8) != 0) return 6;
  printf("ok %lu\n", (unsigned long)bytes);
  return 0;
}
"""


def test_header_compiles_as_c99_and_links(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    lib = os.path.join(PKG, "libmoe.so")
    if cc is None:
        pytest.skip("no C compiler")
    if not os.path.exists(lib):
        pytest.skip("libmoe.so not built")
    src = tmp_path / "abi.c"
    exe = tmp_path / "abi"
    src.write_text(PROGRAM)
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                    "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                    "-L", PKG, "-lmoe", "-Wl,-rpath," + PKG], check=True)
    cuda_lib = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "lib64")
    env = dict(os.environ)
    env["LD_LIBRARY_PATH"] = ":".join(p for p in (PKG, cuda_lib, env.get("LD_LIBRARY_PATH", ""))
                                      if p)
    r = subprocess.run([str(exe)], capture_output=True, text=True, env=env, timeout=60)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    assert r.stdout.startswith("ok ")
