"""The boundary is a C ABI: a plain C99 program (no C++, no torch) compiles
against include/moe.h, links libmoe.so and calls the host-only entry points
(workspace sizes, launch counts, plan flags, error strings, argument checks).
Runs on the CPU: none of these calls launches a kernel."""
import os
import shutil
import subprocess

import pytest

from sparse_mixture_experts_65_b300 import _native as N

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_SRC = r"""
#include <stdio.h>
#include <string.h>
#include "moe.h"

static int fail(const char* what) { printf("FAIL %s\n", what); return 1; }

int main(void) {
  moe_config c;
  memset(&c, 0, sizeof c);
  c.T = 4096; c.d = 7168; c.E = 256; c.k = 8; c.f = 2048;
  c.n_shared = 1; c.f_shared = 2048;
  c.dtype = MOE_BF16; c.act = MOE_ACT_SWIGLU; c.gate = MOE_GATE_SIGMOID_RENORM;
  c.capacity_factor = 0.0; c.alpha = 1e-4f;
  size_t ws = 0;
  if (moe_workspace_size(&c, &ws) != MOE_OK || ws == 0) return fail("workspace size");
  int32_t n = 0;
  if (moe_launch_count(&c, &n) != MOE_OK || n != 4) return fail("launch count");
  uint32_t flags = 0;
  if (moe_plan_flags(&c, &flags) != MOE_OK || !(flags & MOE_PLAN_ROUTE_CLUSTER))
    return fail("plan flags");
  /* e4m3 weights need a layer without a shared expert */
  if (moe_workspace_size_fp8(&c, &ws) != MOE_ERR_UNSUPPORTED) return fail("fp8 shared");
  c.n_shared = 0; c.f_shared = 0;
  if (moe_workspace_size_fp8(&c, &ws) != MOE_OK) return fail("fp8 workspace");
  if (moe_plan_flags_fp8(&c, &flags) != MOE_OK) return fail("fp8 plan flags");
  /* argument checks before any device work */
  if (moe_workspace_size(NULL, &ws) != MOE_ERR_ARG) return fail("null config");
  c.k = 0;
  if (moe_workspace_size(&c, &ws) == MOE_OK) return fail("k = 0 accepted");
  if (moe_set_tuning(MOE_TUNE_COUNT, 0) != MOE_ERR_ARG) return fail("tuning knob range");
  const char* s = moe_error_string(MOE_ERR_UNSUPPORTED);
  if (!s || !*s) return fail("error string");
  printf("OK %s\n", s);
  return 0;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_plain_c_program_uses_the_library(tmp_path):
    N.lib()   # the built library must be present (a clear error otherwise)
    src = tmp_path / "abi.c"
    src.write_text(C_SRC)
    exe = tmp_path / "abi"
    lib_dir = os.path.dirname(N.LIB_PATH)
    cmd = ["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
           str(src), "-o", str(exe), "-L", lib_dir, "-lmoe", f"-Wl,-rpath,{lib_dir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("OK ")
