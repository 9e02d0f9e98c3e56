"""The public header is plain C: a C11 program that includes it compiles with every warning
as an error, links against the library and calls entry points that touch no GPU (version,
status strings, sizes, host-side argument validation)."""
import os
import shutil
import subprocess

import pytest

from nvfp4_routed_moe_sort_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "nvfp4_routed_moe_sort_gb300")

PROGRAM = r"""
#include "moe_nvfp4.h"
#include <stdio.h>

int main(void) {
  if (moe_abi_version() != MOE_NVFP4_ABI_VERSION) return 1;
  const char* ok = moe_status_string(MOE_OK);
  if (ok == NULL || ok[0] == '\0') return 2;
  /* 300 tokens, top-2, 8 local experts: 600 slots + 127 padding rows per expert, to 128 */
  if (moe_plan_capacity(300, 2, 8) != 1664) return 3;
  /* missing buffers are rejected on the host, before any GPU work */
  moe_status_t st = moe_plan(NULL, MOE_IDS_INT32, 4, 2, 4, 0, 4, NULL, NULL, NULL, NULL, NULL, 0, NULL, NULL);
  if (st == MOE_OK) return 4;
  printf("%s\n", moe_status_string(st));
  return 0;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")
def test_header_compiles_as_c_and_links(tmp_path):
    build()
    src = tmp_path / "use_header.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "use_header"
    cc = subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
                         str(src), "-L", PKG, "-lmoe_nvfp4", f"-Wl,-rpath,{PKG}", "-o", str(exe)],
                        capture_output=True, text=True)
    assert cc.returncode == 0, cc.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, (run.returncode, run.stdout, run.stderr)
    assert run.stdout.strip()  # the status string of the rejected call


TEST_PROGRAM = r"""
#include "moe_nvfp4_test.h"
#include <stdio.h>

int main(void) {
  moe_test_options_t o = moe_test_default_options();
  if (o.decode_hooks != 0 || o.withhold_release != 0 || o.wait_limit_ns != 2000000000ull) return 1;
  if (moe_abi_version() != MOE_NVFP4_ABI_VERSION) return 2;
  printf("ok\n");
  return 0;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")
def test_test_header_compiles_as_c_and_links_against_the_test_build(tmp_path):
    build()
    src = tmp_path / "use_test_header.c"
    src.write_text(TEST_PROGRAM)
    exe = tmp_path / "use_test_header"
    cc = subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
                         str(src), "-L", PKG, "-lmoe_nvfp4_test", f"-Wl,-rpath,{PKG}", "-o", str(exe)],
                        capture_output=True, text=True)
    assert cc.returncode == 0, cc.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, (run.returncode, run.stdout, run.stderr)
