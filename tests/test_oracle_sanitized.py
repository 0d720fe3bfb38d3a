"""The oracle's C code under AddressSanitizer and UndefinedBehaviorSanitizer.

A copy of oracle/dsa_oracle.c is built with -fsanitize=address,undefined and
loaded (through DSA_ORACLE_LIB) by a child Python process with the ASan
runtime preloaded; the child runs every oracle entry point on small inputs
that reach its edge cases (dirty and empty ranges, ties, NaN and -inf,
clamped and padded paged rows, scale boundaries, skipped slots).  Any
out-of-bounds access or undefined behaviour aborts the child with a report.
"""
import os
import shutil
import subprocess
import sys
import textwrap

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent(r"""
    import numpy as np
    import oracle
    from top_selection_dsa_gb300 import workloads as wl

    rng = np.random.default_rng(5)
    # prefill logits + top-k (bf16 and e4m3), rows with garbage around ranges
    p = wl.prefill(96, 80, 4, 64, 8, np.array([0, 5, -3, 70, 40] * 19 + [79], np.int32),
                   np.array([80, 5, 200, 75, 10] * 19 + [80], np.int32), seed=1, name="san")
    lg = oracle.logits(p.q, p.k, p.w, p.row_starts, p.row_ends)
    lg32 = lg.astype(np.float32)
    lg32[3, :] = 0.0
    lg32[4, ::2] = np.nan
    lg32[6, :] = -np.inf
    for k in (1, 8, 100):
        oracle.topk(lg32, p.row_starts, p.row_ends, k)
    oracle.sort_by_score(lg32, oracle.topk(lg32, p.row_starts, p.row_ends, 8))
    p8 = wl.prefill(64, 64, 4, 128, 8, seed=2, dtype=wl.E4M3, name="san8")
    oracle.logits(p8.q, p8.k, p8.w, p8.row_starts, p8.row_ends, dtype=p8.dtype,
                  k_scale=p8.k_scale, rows=np.array([0, 31, 63], np.int64))
    # paged: short, empty, over-capacity and exact-capacity contexts
    pd = wl.paged_decode(B=4, next_n=2, ctx_lo=16, ctx_hi=300, block_size=16, H=4, D=64, topk=8)
    cl = np.array([0, 1, 300, 10**6], np.int32)
    oracle.paged_row_ranges(cl, 2)
    oracle.logits_paged(pd.q, pd.w, pd.k_cache, pd.block_table, pd.context_lens, next_n=2)
    # the steps before the indexer
    for v in (0.0, 1e-40, 448.0, 449.0, -464.0, 1e30, float("nan")):
        oracle.f64_to_e4m3(np.array([v]))
    qb = wl.to_bf16_bits(rng.standard_normal((5, 3, 128)).astype(np.float32))
    qb[0] = 0
    oracle.q_quant_fold(qb, rng.standard_normal((5, 3)).astype(np.float32), 0.5, 4)
    kb = wl.to_bf16_bits(rng.standard_normal((6, 128)).astype(np.float32))
    slots = np.array([0, -1, 5, 63, 64, 10**9], np.int64)
    cache = np.zeros((4, 16, 128), np.uint8)
    scale = np.zeros((4, 16), np.float32)
    oracle.k_norm_insert(kb, np.ones(128, np.float32), np.zeros(128, np.float32), 1e-6, slots,
                         cache, scale)
    cand = rng.standard_normal((3, 16)).astype(np.float32)
    cols = rng.permutation(64)[:48].reshape(3, 16).astype(np.int32)
    cols[0, 3] = -1
    oracle.topk_merge(cand, cols, 8)
    print("sanitized oracle ok")
""")


def test_oracle_clean_under_asan_and_ubsan(tmp_path):
    gcc = shutil.which("gcc")
    if not gcc:
        pytest.skip("gcc not found")
    asan = subprocess.run([gcc, "-print-file-name=libasan.so"], capture_output=True,
                          text=True).stdout.strip()
    if not asan or not os.path.isabs(asan) or not os.path.exists(asan):
        pytest.skip("ASan runtime not available")
    lib = str(tmp_path / "libdsa_oracle_san.so")
    src = os.path.join(ROOT, "oracle", "dsa_oracle.c")
    r = subprocess.run([gcc, "-std=c11", "-O1", "-g", "-fno-omit-frame-pointer",
                        "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
                        "-fsanitize=address,undefined", "-fno-sanitize-recover=undefined",
                        "-o", lib, src, "-lm"], capture_output=True, text=True)
    if r.returncode:
        pytest.skip("sanitizer build failed: " + r.stderr[-300:])
    env = dict(os.environ, DSA_ORACLE_LIB=lib, LD_PRELOAD=asan,
               ASAN_OPTIONS="detect_leaks=0:abort_on_error=1",
               UBSAN_OPTIONS="print_stacktrace=1:halt_on_error=1",
               OMP_NUM_THREADS="2", PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=600)
    report = (r.stdout + r.stderr)[-3000:]
    assert r.returncode == 0, report
    assert "sanitized oracle ok" in r.stdout, report
    assert "runtime error" not in r.stderr, report
    assert "AddressSanitizer" not in r.stderr, report
