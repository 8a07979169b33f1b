"""The boundary is a C ABI: the public header compiles as C99 and C++17, and
a plain C program that includes it links libswz.so and calls host-only entry
points (no GPU needed) with the documented results."""
import os
import shutil
import subprocess

import pytest

from conftest import ROOT

C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "swz.h"

int main(void) {
  /* panel G = 4 on an 8 x 8 grid and XOR on 8 x 8 are permutations;
     Morton on 16 x 32 is not; an unknown order is rejected */
  if (swz_is_bijective(SWZ_PANEL, 8, 8, 4) != 1) return 1;
  if (swz_is_bijective(SWZ_XOR, 8, 8, 1) != 1) return 2;
  if (swz_is_bijective(SWZ_MORTON, 16, 32, 1) != 0) return 3;
  if (swz_is_bijective(9, 8, 8, 1) != SWZ_EINVAL) return 4;
  if (strlen(swz_strerror(SWZ_ENOTBIJECTIVE)) == 0) return 5;
  /* plans need no device for non-persistent launches */
  swz_gemm_opts o;
  memset(&o, 0, sizeof o);
  o.cta_pair = 1;
  int tm = 0, tn = 0, sm = 0, sn = 0, programs = 0;
  if (swz_gemm_plan(8192, 8192, 8192, 0, &o, &tm, &tn, &sm, &sn, &programs) != SWZ_OK) return 6;
  if (tm != 64 || tn != 32 || sm != 32 || sn != 32 || programs != 2048) return 7;
  /* argument checks come before any CUDA call */
  if (swz_gemm(NULL, NULL, NULL, 16, 16, 16, SWZ_ROW, 1, 0, NULL) != SWZ_EINVAL) return 8;
  printf("ok\n");
  return 0;
}
"""


@pytest.fixture(scope="module")
def lib_dir():
    from thread_block_smem_gb300 import build
    return os.path.dirname(build.build())


@pytest.mark.parametrize("std,lang", [("c99", "c"), ("c++17", "c++")])
def test_header_compiles(std, lang):
    cc = shutil.which("gcc") if lang == "c" else shutil.which("g++")
    if cc is None:
        pytest.skip("no host compiler")
    r = subprocess.run([cc, "-fsyntax-only", f"-std={std}", "-Wall", "-Wextra", "-x", lang,
                        os.path.join(ROOT, "include", "swz.h")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_c_program_links_and_calls(tmp_path, lib_dir):
    cc = shutil.which("gcc")
    if cc is None:
        pytest.skip("no host compiler")
    src = tmp_path / "caller.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "caller"
    r = subprocess.run([cc, "-std=c99", "-Wall", str(src), "-I", os.path.join(ROOT, "include"),
                        "-L", lib_dir, "-lswz", "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    env = dict(os.environ, LD_LIBRARY_PATH=lib_dir + os.pathsep + os.environ.get("LD_LIBRARY_PATH", ""))
    r = subprocess.run([str(exe)], capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", (r.returncode, r.stdout, r.stderr)
