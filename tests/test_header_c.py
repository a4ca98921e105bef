"""The boundary is a C ABI: the header compiles as plain C99 and a C program
links against libarnorm.so and calls it (host-only entry points, no GPU)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "ar_rmsnorm.h"

int main(void) {
  ar_plan_t plan;
  memset(&plan, 0, sizeof plan);
  if (ar_version() < 100) return 1;
  if (ar_select_mode(8, 8192, 6144) != AR_MODE_ONE_STAGE) return 2;
  if (ar_get_plan(8, 1024, 8192, AR_MODE_AUTO, 152, &plan) != AR_OK) return 3;
  if (plan.kernel != AR_KERNEL_STREAM || plan.launches != 1 || plan.prefetch != AR_PREFETCH_ROW)
    return 4;
  if (ar_get_plan(8, 1, 7168, AR_MODE_AUTO, 152, &plan) != AR_OK || plan.cluster != 8) return 5;
  /* argument errors come back as codes before any CUDA call */
  if (ar_rmsnorm(NULL, 0, NULL, NULL, 1e-6f, 4, 1024, NULL, NULL, AR_MODE_AUTO, NULL) != AR_ERR_ARG)
    return 6;
  if (ar_rmsnorm_two_stage_static(NULL, 2, NULL, NULL, 1e-6f, AR_STATIC_SCRATCH_ELEMS, 8, NULL,
                                  NULL, NULL) != AR_ERR_SCRATCH_LIMIT)
    return 7;
  if (strlen(ar_strerror(AR_ERR_ALIAS)) == 0) return 8;
  printf("ok %d %d %d\n", plan.cluster, plan.vpt, plan.threads);
  return 0;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_c_program_links_and_calls_the_library(arlib, tmp_path):
    src = tmp_path / "use_ar.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "use_ar"
    libdir = os.path.dirname(arlib.LIB_PATH)
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                        f"-I{os.path.join(ROOT, 'include')}", str(src), "-o", str(exe),
                        f"-L{libdir}", "-l:libarnorm.so", f"-Wl,-rpath,{libdir}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.startswith("ok"), (r.returncode, r.stdout, r.stderr)


@pytest.mark.skipif(shutil.which("g++") is None, reason="needs g++")
def test_header_compiles_as_cpp_and_links_with_c_linkage(arlib, tmp_path):
    """The same program as C++17 (extern "C" in the header): the symbols
    resolve unmangled."""
    src = tmp_path / "use_ar.cpp"
    src.write_text(C_PROGRAM.replace("memset(&plan, 0, sizeof plan);",
                                     "std::memset(&plan, 0, sizeof plan);")
                   .replace("#include <string.h>", "#include <cstring>"))
    exe = tmp_path / "use_ar_cpp"
    libdir = os.path.dirname(arlib.LIB_PATH)
    r = subprocess.run(["g++", "-std=c++17", "-Wall", "-Wextra", "-Werror", "-pedantic",
                        f"-I{os.path.join(ROOT, 'include')}", str(src), "-o", str(exe),
                        f"-L{libdir}", "-l:libarnorm.so", f"-Wl,-rpath,{libdir}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.startswith("ok"), (r.returncode, r.stdout, r.stderr)
