"""include/dsa.h is a C header: a plain C11 program compiles against it, links
libdsa.so and gets the documented answers from calls that need no GPU (the
status strings, the workspace sizes and argument errors, which every entry
point returns before it makes any CUDA call)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "dsa.h"

static int fails = 0;
#define CHECK(cond) do { if (!(cond)) { printf("FAIL line %d: %s\n", __LINE__, #cond); ++fails; } } while (0)

int main(void) {
  CHECK(strcmp(dsa_status_string(DSA_OK), "ok") == 0);
  CHECK(strcmp(dsa_status_string((dsa_status_t)99), "unknown status") == 0);
  CHECK(dsa_workspace_bytes(DSA_OP_INDEXER_TOPK, 4096, 4096, 2048) == (size_t)4096 * 4096 * 4);
  CHECK(dsa_workspace_bytes(DSA_OP_TOPK, 10, 10, 4) == 0);
  CHECK(dsa_workspace_bytes(DSA_OP_INDEXER_TOPK, -1, 5, 1) == (size_t)-1);
  void* a = (void*)0x10000;  /* fake, aligned, never dereferenced */
  int32_t* ai = (int32_t*)a;
  float* af = (float*)a;
  /* argument errors come back before any CUDA call */
  CHECK(dsa_indexer_logits(NULL, NULL, a, NULL, DSA_BF16, af, ai, ai, 8, 8, 64, 128, af, 8, 0,
                           NULL) == DSA_ERR_INVALID_ARG);
  CHECK(dsa_indexer_logits(a, NULL, a, NULL, DSA_BF16, af, ai, ai, 8, 8, 128, 128, af, 8, 0,
                           NULL) == DSA_ERR_UNSUPPORTED);
  CHECK(dsa_topk(af, 8, ai, ai, 4, 8, 0, ai, NULL, 0, NULL) == DSA_ERR_INVALID_ARG);
  CHECK(dsa_indexer_topk(a, NULL, a, NULL, DSA_E4M3, af, ai, ai, 8, 8, 64, 128, 2, ai, a, 1 << 20,
                         NULL) == DSA_ERR_INVALID_ARG);  /* e4m3 without key scales */
  CHECK(dsa_indexer_topk_host(a, NULL, a, NULL, DSA_BF16, af, ai, ai, 8, 8, 64, 128, 2, ai, NULL,
                              0, NULL) == DSA_ERR_INVALID_ARG);  /* no device buffer */
  CHECK(dsa_topk_merge(af, ai, 4, 16385, 8, ai, NULL) == DSA_ERR_UNSUPPORTED);
  printf(fails ? "failed\n" : "c abi ok\n");
  return fails ? 1 : 0;
}
"""


def test_plain_c_program_uses_the_header_and_library(tmp_path):
    from top_selection_dsa_gb300 import build
    lib = build.build()
    cc = shutil.which("gcc") or shutil.which("cc")
    if not cc:
        pytest.skip("no C compiler")
    src = tmp_path / "use_dsa.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "use_dsa"
    libdir = os.path.dirname(lib)
    r = subprocess.run([cc, "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                        str(src), "-o", str(exe), "-L", libdir, "-l:libdsa.so",
                        f"-Wl,-rpath,{libdir}"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c abi ok" in r.stdout
