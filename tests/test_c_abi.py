"""The boundary is plain C: include/turboquant.h compiles as C99 with every
warning an error, and a C program linked against libturboquant.so makes the
host-side calls (setup tables, plan sizes, status strings, argument errors
returned before any launch).  No GPU is touched."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")
LIBDIR = os.path.join(ROOT, "online_kv_cache_04_b300")

PROGRAM = r"""
#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "turboquant.h"

static int fail(const char* what) {
  fprintf(stderr, "FAIL: %s\n", what);
  return 1;
}

int main(void) {
  enum { D = 16 };
  double pi[D * D];
  if (tq_make_rotation(D, 0x71550001ull, pi) != TQ_OK) return fail("tq_make_rotation");
  /* Π Πᵀ = I */
  for (int i = 0; i < D; ++i)
    for (int j = 0; j < D; ++j) {
      double s = 0.0;
      for (int k = 0; k < D; ++k) s += pi[i * D + k] * pi[j * D + k];
      if (fabs(s - (i == j ? 1.0 : 0.0)) > 1e-12) return fail("rotation not orthogonal");
    }
  double c[4], b[3], mse = 0.0;
  if (tq_make_codebook(128, 2, c, b, &mse) != TQ_OK) return fail("tq_make_codebook");
  for (int i = 0; i < 4; ++i)
    if (c[i] != -c[3 - i]) return fail("codebook not symmetric");
  if (!(c[0] < c[1] && c[1] < c[2] && c[2] < c[3]) || b[1] != 0.0) return fail("codebook order");
  if (!(mse > 0.0 && 128.0 * mse < 0.25)) return fail("codebook mse");
  double* S = malloc(sizeof(double) * 32 * D);
  double* sr = malloc(sizeof(double) * 32 * D);
  if (!S || !sr || tq_make_qjl(32, D, 0x71550002ull, pi, S, sr) != TQ_OK) return fail("tq_make_qjl");
  free(S);
  free(sr);
  if (tq_plan_bytes(128, 128, 2) == 0 || tq_plan_bytes(100, 128, 2) != 0) return fail("tq_plan_bytes");
  if (tq_make_rotation(1, 0, pi) != TQ_ERR_ARG) return fail("rotation argument check");
  if (tq_quantize(NULL, NULL, TQ_BF16, 1, 128, NULL, 0, NULL) != TQ_ERR_ARG) return fail("quantize argument check");
  if (tq_append_kv(NULL, NULL, NULL, TQ_F32, 1, 1, NULL, NULL, NULL, 1, NULL) != TQ_ERR_ARG)
    return fail("append argument check");
  const char* s = tq_status_str(TQ_ERR_WORKSPACE);
  if (s == NULL || strlen(s) == 0) return fail("tq_status_str");
  printf("c abi ok\n");
  return 0;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_header_is_c99_and_host_calls_work_from_c(tmp_path):
    from online_kv_cache_04_b300 import _lib

    _lib.load()  # the library is built
    src = tmp_path / "abi.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "abi"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", INCLUDE, str(src), "-o",
                    str(exe), "-L", LIBDIR, "-lturboquant", f"-Wl,-rpath,{LIBDIR}", "-lm"], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stderr
    assert "c abi ok" in out.stdout
