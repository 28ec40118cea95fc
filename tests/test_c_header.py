"""The boundary from plain C (no GPU needed: nothing here launches work).

A C99 program that includes include/dion.h and include/muon.h is compiled with
gcc (warnings as errors) and linked against libdion.so.  It drives the host-only
calls of both headers with fake, never dereferenced device addresses (plan
creation, validation errors, workspace checks that precede any CUDA call) and
prints the size and field offsets of the two descriptor structs, which must be
those the ctypes binding declares.
"""
import ctypes
import os
import shutil
import subprocess

import pytest

from rank_orthonormalized_optimizer_03_b300 import build, dion

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "dion.h"
#include "muon.h"

#define CHECK(c) do { if (!(c)) { printf("FAILED %s (line %d): %s\n", #c, __LINE__, dion_last_error()); return 1; } } while (0)
#define FAKE(k) ((void*)(uintptr_t)(0x7f0000000000ull + (uint64_t)(k) * (1ull << 32)))

static dion_matrix_desc desc(int k, int64_t m, int64_t n, int64_t r, int32_t variant) {
  dion_matrix_desc d;
  memset(&d, 0, sizeof d);
  d.X = (float*)FAKE(4 * k); d.G = FAKE(4 * k + 1); d.R = (float*)FAKE(4 * k + 2); d.V = (float*)FAKE(4 * k + 3);
  d.m = m; d.n = n; d.r = r; d.ld_x = n; d.ld_g = n; d.ld_r = n;
  d.g_dtype = DION_DTYPE_BF16; d.variant = variant;
  d.eta = 0.02f; d.beta = 0.95f; d.scale = 0.0f; d.reserved = 0.0f;
  return d;
}

#define OFF(T, f) printf(#T " " #f " %zu\n", offsetof(T, f))

int main(void) {
  CHECK(dion_abi_version() == DION_ABI_VERSION);
  CHECK(dion_status_string(DION_ERR_WORKSPACE) != NULL && strlen(dion_status_string(DION_ERR_WORKSPACE)) > 0);

  dion_matrix_desc d[3];
  d[0] = desc(0, 3072, 3072, 192, DION_VARIANT_ORTH);
  d[1] = desc(1, 8192, 3072, 192, DION_VARIANT_DION);
  d[2] = desc(2, 1000, 264, 264, DION_VARIANT_ORTH);
  size_t ws = 0;
  dion_plan* plan = NULL;
  CHECK(dion_plan_create(d, 3, &ws, &plan) == DION_OK);
  CHECK(plan != NULL && ws > 0);
  CHECK(dion_plan_count(plan) == 3);
  CHECK(dion_plan_launches_per_step(plan) > 0);
  CHECK(dion_plan_set_hparams(plan, 1, 0.01f, 0.9f) == DION_OK);
  CHECK(dion_plan_set_hparams(plan, 3, 0.01f, 0.9f) == DION_ERR_INVALID_ARG);
  size_t off = 0; int64_t rows = 0, cols = 0, ld = 0;
  CHECK(dion_plan_buffer(plan, 2, 1, &off, &rows, &cols, &ld) == DION_OK);
  CHECK(rows == 1000 && cols == 264 && ld >= 264 && off + (size_t)(rows * ld * 4) <= ws);
  /* workspace checks come before any CUDA call */
  CHECK(dion_step_batched(plan, NULL, ws, NULL) == DION_ERR_WORKSPACE);
  CHECK(dion_step_batched(plan, FAKE(99), ws - 1, NULL) == DION_ERR_WORKSPACE);
  dion_plan_destroy(plan);
  dion_plan_destroy(NULL);

  /* rank above min(m, n), bad dtype, reserved field set: rejected with a message */
  dion_matrix_desc bad = desc(0, 64, 32, 33, DION_VARIANT_ORTH);
  plan = NULL;
  CHECK(dion_plan_create(&bad, 1, &ws, &plan) == DION_ERR_INVALID_ARG && plan == NULL);
  CHECK(strlen(dion_last_error()) > 0);
  bad = desc(0, 64, 32, 8, DION_VARIANT_ORTH); bad.g_dtype = 7;
  CHECK(dion_plan_create(&bad, 1, &ws, &plan) == DION_ERR_INVALID_ARG);
  bad = desc(0, 64, 32, 8, DION_VARIANT_ORTH); bad.reserved = 1.0f;
  CHECK(dion_plan_create(&bad, 1, &ws, &plan) == DION_ERR_INVALID_ARG);

  muon_matrix_desc md[2];
  memset(md, 0, sizeof md);
  for (int k = 0; k < 2; ++k) {
    md[k].X = (float*)FAKE(10 + 3 * k); md[k].G = FAKE(11 + 3 * k); md[k].B = (float*)FAKE(12 + 3 * k);
    md[k].m = 768 * (k + 1); md[k].n = 768; md[k].ld_x = md[k].ld_g = md[k].ld_b = 768;
    md[k].g_dtype = DION_DTYPE_F32; md[k].eta = 0.02f; md[k].mu = 0.95f;
  }
  muon_plan* mp = NULL;
  CHECK(muon_plan_create(md, 2, 5, MUON_NS_BF16, 1.0f, &ws, &mp) == DION_OK && mp != NULL && ws > 0);
  CHECK(muon_plan_launches_per_step(mp) > 0);
  CHECK(muon_step_batched(mp, NULL, ws, NULL) == DION_ERR_WORKSPACE);
  muon_plan_destroy(mp);
  muon_plan_destroy(NULL);

  printf("dion_matrix_desc size %zu\n", sizeof(dion_matrix_desc));
  OFF(dion_matrix_desc, X); OFF(dion_matrix_desc, G); OFF(dion_matrix_desc, R); OFF(dion_matrix_desc, V);
  OFF(dion_matrix_desc, m); OFF(dion_matrix_desc, n); OFF(dion_matrix_desc, r);
  OFF(dion_matrix_desc, ld_x); OFF(dion_matrix_desc, ld_g); OFF(dion_matrix_desc, ld_r);
  OFF(dion_matrix_desc, g_dtype); OFF(dion_matrix_desc, variant);
  OFF(dion_matrix_desc, eta); OFF(dion_matrix_desc, beta); OFF(dion_matrix_desc, scale);
  OFF(dion_matrix_desc, reserved);
  printf("muon_matrix_desc size %zu\n", sizeof(muon_matrix_desc));
  OFF(muon_matrix_desc, X); OFF(muon_matrix_desc, G); OFF(muon_matrix_desc, B);
  OFF(muon_matrix_desc, m); OFF(muon_matrix_desc, n);
  OFF(muon_matrix_desc, ld_x); OFF(muon_matrix_desc, ld_g); OFF(muon_matrix_desc, ld_b);
  OFF(muon_matrix_desc, g_dtype); OFF(muon_matrix_desc, eta); OFF(muon_matrix_desc, mu);
  OFF(muon_matrix_desc, scale);
  printf("ok\n");
  return 0;
}
"""


def test_headers_compile_as_c_and_match_the_binding(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    build.build()
    src = tmp_path / "abi.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "abi"
    res = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", dion.INCLUDE,
                          "-o", str(exe), str(src), dion.LIB_PATH, "-Wl,-rpath," + os.path.dirname(dion.LIB_PATH)],
                         capture_output=True, text=True)
    assert res.returncode == 0, res.stderr[-3000:]
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    out = run.stdout.splitlines()
    assert run.returncode == 0 and out and out[-1] == "ok", run.stdout + run.stderr

    layout = {}
    for ln in out[:-1]:
        parts = ln.split()
        if len(parts) == 3 and parts[1] == "size":
            layout[(parts[0], "__size__")] = int(parts[2])
        elif len(parts) == 3:
            layout[(parts[0], parts[1])] = int(parts[2])
    for cname, cls in (("dion_matrix_desc", dion.MatrixDesc), ("muon_matrix_desc", dion.MuonDesc)):
        assert layout[(cname, "__size__")] == ctypes.sizeof(cls), cname
        for field, _ in cls._fields_:
            assert layout[(cname, field)] == getattr(cls, field).offset, (cname, field)
