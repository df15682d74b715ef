"""The C ABI from C: include/jetlong.h compiles as strict C99 and a C program
links against libjetlong.so and calls the host-side entry points (group
size, workspace sizes, argument validation) -- no GPU needed."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "bifocal_rope_extension_causal_b300")

C_PROGRAM = r"""
#include "jetlong.h"
#include <stdio.h>
#include <string.h>

int main(void) {
  int bad = 0;
  /* G = max(1, ceil(L / w_pretrained)) */
  if (jl_group_size(131072, 32768) != 4 || jl_group_size(32767, 32768) != 1 ||
      jl_group_size(32769, 32768) != 2 || jl_group_size(-1, 5) != -1) bad |= 1;
  /* workspace sizes are positive for valid shapes and 0 for invalid ones */
  if (jl_bifocal_prefill_workspace_size(1, 1024, 4, 2, 128, 512) == 0 ||
      jl_bifocal_prefill_workspace_size(0, 1024, 4, 2, 128, 512) != 0 ||
      jl_bifocal_decode_workspace_size(1, 32, 128, 131072) == 0 ||
      jl_bifocal_prefill_host_workspace_size(1, 1024, 4, 2, 128, 512) <=
          jl_bifocal_prefill_workspace_size(1, 1024, 4, 2, 128, 512)) bad |= 2;
  /* argument validation happens before any CUDA call */
  if (jl_bifocal_prefill(NULL, NULL, NULL, NULL, NULL, 1, 128, 2, 1, 128, 16, 64, 1e4, 0.f, NULL, NULL,
                         0, NULL) != JL_ERR_INVALID) bad |= 4;
  if (strlen(jl_last_error()) == 0) bad |= 8;
  printf("%d\n", bad);
  return bad;
}
"""


@pytest.fixture(scope="module")
def lib_path():
    from bifocal_rope_extension_causal_b300 import build
    build.build()
    return os.path.join(PKG, "libjetlong.so")


def test_header_compiles_as_c99(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = tmp_path / "h.c"
    src.write_text('#include "jetlong.h"\nint main(void) { return 0; }\n')
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                        "-I", os.path.join(ROOT, "include"), "-c", str(src), "-o", str(tmp_path / "h.o")],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_c_program_calls_the_library(tmp_path, lib_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = tmp_path / "prog.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "prog"
    r = subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), lib_path,
                        "-Wl,-rpath," + PKG, "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, f"C checks failed: bitmask {r.stdout.strip()} {r.stderr}"
