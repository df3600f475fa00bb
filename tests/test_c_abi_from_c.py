"""The boundary is a C ABI: include/bi.h compiles as strict C99, and a plain C
program links libbi.so and calls its host-side entry points (version, error
text, argument validation, size queries, the prefill schedule) with no Python
and no GPU involved."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "invariant_forward_policy_gb300")

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "bi.h"

int main(void) {
  int64_t cu[3] = {0, 6, 11}, sp[2] = {0, 10}, rec[4 * 8];
  int64_t n, i;
  bi_status st;
  printf("version %d\n", bi_version());
  /* a null pointer is refused before anything is launched */
  st = bi_rmsnorm(NULL, NULL, NULL, NULL, 4, 256, 1e-6f, BI_INVARIANT, NULL);
  printf("rmsnorm_null %d %s\n", (int)st, strlen(bi_last_error()) > 0 ? "msg" : "nomsg");
  printf("ssd_state_bytes %lld\n", (long long)bi_ssd_state_bytes(4, 2, 64, 128, 64));
  printf("gemm_tile_n %d\n", bi_gemm_tile_n(32000, 512, BI_EPI_NONE));
  n = bi_prefill_plan(cu, sp, NULL, 2, 4, 6, rec, 4);
  printf("plan %lld", (long long)n);
  for (i = 0; i < n && i < 4; ++i) printf(" (%lld %lld %lld)", (long long)rec[8 * i], (long long)rec[8 * i + 1],
                                         (long long)rec[8 * i + 3]);
  printf("\n");
  return 0;
}
"""


@pytest.fixture(scope="module")
def lib_path():
    path = os.path.join(PKG, "libbi.so")
    if not os.path.exists(path):
        from invariant_forward_policy_gb300 import build
        build.build()
    return path


def test_header_is_strict_c99():
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    r = subprocess.run([cc, "-fsyntax-only", "-x", "c", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                        os.path.join(ROOT, "include", "bi.h")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_plain_c_program_calls_the_library(tmp_path, lib_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "abi.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "abi"
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src), "-o",
                        str(exe), "-L", PKG, "-lbi", f"-Wl,-rpath,{PKG}"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120,
                       env=dict(os.environ, CUDA_VISIBLE_DEVICES=""))
    assert r.returncode == 0, r.stderr
    out = dict(line.split(" ", 1) for line in r.stdout.strip().splitlines())
    assert out["version"] == "100"
    assert out["rmsnorm_null"] == "1 msg"                                   # BI_ERR_INVALID_ARG with a message
    assert out["ssd_state_bytes"] == str(4 * (4 * 128 * 64 + 64 * 4 * 128 + 64 * 4 * 64 + 64 * 4))
    assert int(out["gemm_tile_n"]) in (16, 32, 64, 128, 256)
    assert out["plan"] == "4 (0 0 4) (1 1 4) (1 0 2) (2 1 1)"               # the schedule of the Python test
