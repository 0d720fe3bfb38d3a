"""The C-ABI library builds, loads and validates arguments on the host (no GPU).

Only argument-validation paths are exercised: every call here is rejected
before the library makes any CUDA call, so no device is needed.  Pointers are
fake addresses that are never dereferenced.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def api():
    from top_selection_dsa_gb300 import build
    build.build()
    from top_selection_dsa_gb300 import api as _api
    return _api


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "dsa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dsa_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for name in ("dsa_indexer_logits", "dsa_topk", "dsa_indexer_topk",
                 "dsa_indexer_topk_paged", "dsa_workspace_bytes", "dsa_status_string",
                 "dsa_get_last_device_error"):
        assert name in syms


def test_library_exports_every_declared_symbol(api):
    lib = ctypes.CDLL(api.LIB_PATH)
    for name in declared_symbols():
        assert hasattr(lib, name), name
    assert set(declared_symbols()) == set(api.EXPORTS)


def test_status_strings(api):
    for s in range(5):
        assert api.status_string(s)
    assert api.status_string(99) == "unknown status"


def test_workspace_bytes(api):
    wb = api.lib.dsa_workspace_bytes
    assert wb(api.DSA_OP_INDEXER_LOGITS, 10, 10, 4) == 0
    assert wb(api.DSA_OP_TOPK, 10, 10, 4) == 0
    assert wb(api.DSA_OP_INDEXER_TOPK, 4096, 4096, 2048) == 4096 * 4096 * 4
    assert wb(api.DSA_OP_INDEXER_TOPK, 3, 5, 1) == 256        # rows padded to 16 B, total to 256
    # few long rows: per-row scratch of the split top-k (2048-bin histogram,
    # 16 state words, 3 words for each of up to 256 4096-key units, 16384
    # candidate keys), rounded up to 64 words; it follows the logits in the
    # composed calls
    def split(rows, S):
        words = 2048 + 16 + 3 * 256 + 16384
        return rows * (-(-words // 64) * 64) * 4
    assert wb(api.DSA_OP_TOPK, 16, 131072, 2048) == split(16, 131072)   # fewer than 32 rows
    assert wb(api.DSA_OP_TOPK, 128, 131072, 2048) == 0        # 32-512 rows: a CTA per row
    assert wb(api.DSA_OP_TOPK, 128, 300000, 2048) == split(128, 300000)  # rows past 262144
    assert wb(api.DSA_OP_TOPK, 4096, 131072, 2048) == 0       # many rows: no scratch
    assert wb(api.DSA_OP_TOPK, 128, 16384, 2048) == 0         # short rows: no scratch
    assert wb(api.DSA_OP_INDEXER_TOPK_PAGED, 128, 131072, 2048) == 128 * 131072 * 4
    assert wb(api.DSA_OP_INDEXER_TOPK_PAGED, 16, 131072, 2048) == \
        16 * 131072 * 4 + split(16, 131072)
    assert wb(api.DSA_OP_INDEXER_TOPK, 0, 100, 1) == 0
    bad = ctypes.c_size_t(-1).value
    assert wb(api.DSA_OP_INDEXER_TOPK, -1, 5, 1) == bad
    assert wb(17, 1, 1, 1) == bad


A = ctypes.c_void_p(0x10000)       # fake, 16-byte aligned, never dereferenced
MIS = ctypes.c_void_p(0x10004)     # fake, misaligned for TMA
NUL = None


def logits_call(api, q=A, k=A, ks=NUL, dtype=0, w=A, rs=A, re=A, T=8, S=8, H=64, D=128,
                out=A, ld=8, flags=0):
    return api.lib.dsa_indexer_logits(q, NUL, k, ks, dtype, w, rs, re, T, S, H, D, out, ld,
                                      flags, NUL)


def test_indexer_logits_validation(api):
    E, U = api.DSA_ERR_INVALID_ARG, api.DSA_ERR_UNSUPPORTED
    assert logits_call(api, q=NUL) == E
    assert logits_call(api, k=NUL) == E
    assert logits_call(api, w=NUL) == E
    assert logits_call(api, rs=NUL) == E
    assert logits_call(api, out=NUL) == E
    assert logits_call(api, T=-1) == E
    assert logits_call(api, ld=7) == E                       # ld < S
    assert logits_call(api, q=MIS) == E                      # TMA needs 16-byte alignment
    assert logits_call(api, k=MIS) == E
    assert logits_call(api, flags=2) == E
    assert logits_call(api, dtype=5) == E
    assert logits_call(api, H=3) == U
    assert logits_call(api, H=128) == U                      # > 64 index heads
    assert logits_call(api, D=96) == U
    assert logits_call(api, dtype=1, ks=A, D=64) == U        # e4m3 needs D = 128
    assert logits_call(api, dtype=1, ks=NUL) == E            # e4m3 needs key scales
    assert logits_call(api, dtype=0, ks=A) == E              # bf16 takes none


def test_topk_validation(api):
    E = api.DSA_ERR_INVALID_ARG
    f = api.lib.dsa_topk
    need = api.lib.dsa_workspace_bytes(api.DSA_OP_TOPK, 4, 100000, 8)
    assert need > 0
    assert f(A, 100000, A, A, 4, 100000, 8, A, NUL, 0, NUL) == E       # split path needs scratch
    assert f(A, 100000, A, A, 4, 100000, 8, A, A, need - 1, NUL) == E
    assert f(A, 100000, A, A, 4, 100000, 8, A, MIS, need, NUL) == E
    assert f(NUL, 8, A, A, 4, 8, 2, A, NUL, 0, NUL) == E
    assert f(A, 8, A, A, 4, 8, 0, A, NUL, 0, NUL) == E       # k < 1
    assert f(A, 4, A, A, 4, 8, 2, A, NUL, 0, NUL) == E       # ld < S
    assert f(A, 8, A, A, 4, 8, 2, NUL, NUL, 0, NUL) == E
    assert f(A, 8, NUL, A, 4, 8, 2, A, NUL, 0, NUL) == E


def test_indexer_topk_validation(api):
    E = api.DSA_ERR_INVALID_ARG
    f = api.lib.dsa_indexer_topk
    need = api.lib.dsa_workspace_bytes(api.DSA_OP_INDEXER_TOPK, 8, 8, 2)
    assert f(A, NUL, A, NUL, 0, A, A, A, 8, 8, 64, 128, 2, A, NUL, need, NUL) == E  # no ws
    assert f(A, NUL, A, NUL, 0, A, A, A, 8, 8, 64, 128, 2, A, A, need - 1, NUL) == E
    assert f(A, NUL, A, NUL, 0, A, A, A, 8, 8, 64, 128, 2, A, MIS, need, NUL) == E
    assert f(A, NUL, A, NUL, 0, A, A, A, 8, 8, 64, 128, 0, A, A, need, NUL) == E
    assert f(A, NUL, A, NUL, 0, A, A, A, 8, 8, 3, 128, 2, A, A, need, NUL) == \
        api.DSA_ERR_UNSUPPORTED


def paged_call(api, q=A, w=A, kc=A, ks=NUL, nblk=10, dtype=0, bt=A, maxb=4, cl=A, B=2,
               next_n=2, bs=64, H=64, D=128, out=A, ld=256):
    return api.lib.dsa_indexer_logits_paged(q, NUL, w, kc, ks, nblk, dtype, bt, maxb, cl, B,
                                            next_n, bs, H, D, out, ld, NUL)


def test_paged_validation(api):
    E, U = api.DSA_ERR_INVALID_ARG, api.DSA_ERR_UNSUPPORTED
    assert paged_call(api, bt=NUL) == E
    assert paged_call(api, cl=NUL) == E
    assert paged_call(api, kc=MIS) == E
    assert paged_call(api, nblk=0) == E
    assert paged_call(api, next_n=0) == E
    assert paged_call(api, ld=255) == E                       # ld < max_blocks * block_size
    assert paged_call(api, bs=48) == U                        # not a power of two
    assert paged_call(api, bs=256) == U
    assert paged_call(api, next_n=5) == U                     # 5 * 64 > 256 MMA columns
    assert paged_call(api, H=4) == U
    assert paged_call(api, dtype=1) == E                      # e4m3 without key scales
    f = api.lib.dsa_indexer_topk_paged
    need = api.lib.dsa_workspace_bytes(api.DSA_OP_INDEXER_TOPK_PAGED, 4, 256, 8)
    assert f(A, NUL, A, A, NUL, 10, 0, A, 4, A, 2, 2, 64, 64, 128, 8, A, NUL, need, NUL) == E
    assert f(A, NUL, A, A, NUL, 10, 0, A, 4, A, 2, 2, 64, 64, 128, 0, A, A, need, NUL) == E


def test_binding_refuses_cpu_tensors(api):
    import torch
    q = torch.zeros(4, 64, 128, dtype=torch.bfloat16)
    k = torch.zeros(4, 128, dtype=torch.bfloat16)
    w = torch.zeros(4, 64)
    r = torch.zeros(4, dtype=torch.int32)
    with pytest.raises(ValueError):
        api.indexer_logits(q, k, w, r, r)


def test_topk_sort_by_score_validation(api):
    E, U = api.DSA_ERR_INVALID_ARG, api.DSA_ERR_UNSUPPORTED
    f = api.lib.dsa_topk_sort_by_score
    assert f(NUL, 8, A, 4, 2, NUL) == E
    assert f(A, 8, NUL, 4, 2, NUL) == E
    assert f(A, 8, A, -1, 2, NUL) == E
    assert f(A, 8, A, 4, 0, NUL) == E
    assert f(A, 0, A, 4, 2, NUL) == E
    assert f(ctypes.c_void_p(0x10002), 8, A, 4, 2, NUL) == E     # logits not 4-byte aligned
    assert f(A, 8, A, 4, 8193, NUL) == U                         # k above the sort's limit
    assert f(A, 8, A, 0, 2, NUL) == api.DSA_OK                   # nothing to do, nothing launched


def test_prologue_validation(api):
    E, U = api.DSA_ERR_INVALID_ARG, api.DSA_ERR_UNSUPPORTED
    f = api.lib.dsa_q_quant_fold_weights
    assert f(NUL, A, 1.0, 4, 64, 128, 64, A, A, NUL) == E
    assert f(A, A, 1.0, 4, 64, 128, 32, A, A, NUL) == E          # padded_heads < H
    assert f(MIS, A, 1.0, 4, 64, 128, 64, A, A, NUL) == E        # q not 16-byte aligned
    assert f(A, A, 1.0, 4, 64, 64, 64, A, A, NUL) == U           # D != 128
    assert f(A, A, 1.0, 4, 16, 128, 128, A, A, NUL) == U         # more than 64 heads
    g = api.lib.dsa_k_norm_quant_insert
    B16, E8 = api.DSA_BF16, api.DSA_E4M3
    assert g(NUL, A, A, 1e-6, A, 4, 128, B16, A, NUL, 8, 64, NUL) == E
    assert g(A, A, A, 1e-6, A, 4, 128, E8, A, NUL, 8, 64, NUL) == E    # e4m3 needs scales
    assert g(A, A, A, 1e-6, A, 4, 128, B16, A, A, 8, 64, NUL) == E     # bf16 takes none
    assert g(A, A, A, -1.0, A, 4, 128, B16, A, NUL, 8, 64, NUL) == E   # eps < 0
    assert g(A, A, A, 1e-6, A, 4, 128, B16, A, NUL, 0, 64, NUL) == E   # no blocks
    assert g(A, A, A, 1e-6, A, 4, 64, B16, A, NUL, 8, 64, NUL) == U    # D != 128


def test_topk_merge_validation(api):
    E, U = api.DSA_ERR_INVALID_ARG, api.DSA_ERR_UNSUPPORTED
    f = api.lib.dsa_topk_merge
    assert f(NUL, A, 4, 16, 8, A, NUL) == E
    assert f(A, A, 4, 0, 8, A, NUL) == E
    assert f(A, A, 4, 16, 0, A, NUL) == E
    assert f(A, A, -1, 16, 8, A, NUL) == E
    assert f(A, A, 4, 16385, 8, A, NUL) == U
    assert f(A, A, 4, 16, 16385, A, NUL) == U


def test_topk_merge_ranks_validation(api):
    E, U = api.DSA_ERR_INVALID_ARG, api.DSA_ERR_UNSUPPORTED
    f = api.lib.dsa_topk_merge_ranks                        # (s, c, W, T, kr, k, out, stream)
    assert f(NUL, A, 2, 4, 16, 8, A, NUL) == E
    assert f(A, A, 0, 4, 16, 8, A, NUL) == E                 # no rank
    assert f(A, A, 2, -1, 16, 8, A, NUL) == E
    assert f(A, A, 2, 4, 0, 8, A, NUL) == E
    assert f(A, A, 2, 4, 16, 0, A, NUL) == E
    assert f(A, A, 2, 4, 16, 8, ctypes.c_void_p(0x10002), NUL) == E   # out not 4-byte aligned
    assert f(A, A, 2, 4, 8193, 8, A, NUL) == U               # W * kr > 16384
    assert f(A, A, 2, 4, 16, 16385, A, NUL) == U


def test_topk_dcp_candidates_validation(api):
    E, U = api.DSA_ERR_INVALID_ARG, api.DSA_ERR_UNSUPPORTED
    f = api.lib.dsa_topk_dcp_candidates
    # (logits, ld, rs, re, T, S, k, rank, world, interleave, scores, cols, ws, ws_bytes, stream)
    assert f(NUL, 8, A, A, 4, 8, 2, 0, 2, 64, A, A, NUL, 0, NUL) == E
    assert f(A, 8, A, A, 4, 8, 2, 2, 2, 64, A, A, NUL, 0, NUL) == E    # rank >= world
    assert f(A, 8, A, A, 4, 8, 2, -1, 2, 64, A, A, NUL, 0, NUL) == E
    assert f(A, 8, A, A, 4, 8, 2, 0, 0, 64, A, A, NUL, 0, NUL) == E    # world < 1
    assert f(A, 8, A, A, 4, 8, 2, 0, 2, 0, A, A, NUL, 0, NUL) == E     # interleave < 1
    assert f(A, 8, A, A, 4, 8, 0, 0, 2, 64, A, A, NUL, 0, NUL) == E    # k < 1
    assert f(A, 4, A, A, 4, 8, 2, 0, 2, 64, A, A, NUL, 0, NUL) == E    # ld < S
    assert f(A, 8, A, A, 4, 8, 2, 0, 2, 64, NUL, A, NUL, 0, NUL) == E
    assert f(A, 8, A, A, 4, 8, 2, 0, 2, 64, A, ctypes.c_void_p(0x10002), NUL, 0, NUL) == E
    need = api.lib.dsa_workspace_bytes(api.DSA_OP_TOPK, 4, 100000, 8)
    assert f(A, 100000, A, A, 4, 100000, 8, 0, 2, 64, A, A, NUL, 0, NUL) == E   # needs scratch
    # global positions past INT32_MAX
    assert f(A, 100000, A, A, 4, 100000, 8, 0, 1 << 16, 64, A, A, A, need, NUL) == U


def test_indexer_topk_host_validation(api):
    E, U = api.DSA_ERR_INVALID_ARG, api.DSA_ERR_UNSUPPORTED
    nb = api.lib.dsa_indexer_topk_host_bytes
    need = nb(4096, 4096, 64, 128, 2048, api.DSA_BF16)
    # inputs (q, k, weights, ranges, indices) plus one chunk's logits: up to 8
    # chunks of at least 512 rows
    inputs = 4096 * 64 * 128 * 2 + 4096 * 128 * 2 + 4096 * 64 * 4 * 2 + 2 * 4096 * 4 + \
        4096 * 2048 * 4
    assert inputs < need <= inputs + 512 * 4096 * 4 + 10 * 256
    assert nb(-1, 8, 64, 128, 2, api.DSA_BF16) == ctypes.c_size_t(-1).value
    assert nb(8, 8, 64, 128, 2, 7) == ctypes.c_size_t(-1).value
    f = api.lib.dsa_indexer_topk_host
    n = nb(8, 8, 64, 128, 2, api.DSA_BF16)
    assert f(A, NUL, A, NUL, 0, A, A, A, 8, 8, 64, 128, 2, A, NUL, n, NUL) == E    # no buffer
    assert f(A, NUL, A, NUL, 0, A, A, A, 8, 8, 64, 128, 2, A, A, n - 1, NUL) == E  # too small
    assert f(A, NUL, A, NUL, 0, A, A, A, 8, 8, 64, 128, 2, A, MIS, n, NUL) == E
    assert f(NUL, NUL, A, NUL, 0, A, A, A, 8, 8, 64, 128, 2, A, A, n, NUL) == E
    assert f(A, NUL, A, NUL, 0, A, A, A, 8, 8, 64, 128, 2, NUL, A, n, NUL) == E
    assert f(A, NUL, A, NUL, 0, A, A, A, 8, 8, 64, 128, 0, A, A, n, NUL) == E
    assert f(A, NUL, A, NUL, 0, A, A, A, 8, 8, 3, 128, 2, A, A, n, NUL) == U
    assert f(A, NUL, A, NUL, 1, A, A, A, 8, 8, 64, 128, 2, A, A, n, NUL) == E     # e4m3, no scales
    assert f(A, NUL, A, NUL, 0, A, A, A, 0, 8, 64, 128, 2, A, A, n, NUL) == api.DSA_OK  # no rows
    assert f(NUL, NUL, A, NUL, 0, NUL, NUL, NUL, 0, 8, 64, 128, 2, NUL, A, n, NUL) == api.DSA_OK
    assert f(A, NUL, NUL, NUL, 0, A, A, A, 8, 8, 64, 128, 2, A, A, n, NUL) == E   # keys, no k


def host_chunks(T, unit=64):
    """Row chunks of dsa_indexer_topk_host with no device: up to 12 chunks of
    a multiple of 64 rows, at least 512 rows each where T allows, the
    remainder first; with three or more, the first and the last cut down to
    one unit (the rest of each a chunk of its own)."""
    if T <= 0:
        return []
    nch = min(12, -(-T // 512))
    chunk = max(1, -(-(-(-T // nch)) // unit) * unit)
    first = T - (T - 1) // chunk * chunk
    nfull = (T - first) // chunk
    cut = nfull >= 2
    bounds = [0] + ([unit] if cut and first > unit else []) + [first]
    for c in range(1, nfull + 1):
        if cut and c == nfull and chunk > unit:
            bounds.append(T - unit)
        bounds.append(first + c * chunk)
    return [b - a for a, b in zip(bounds, bounds[1:])]


def test_host_chunks_cover_the_rows():
    for T in (1, 63, 64, 511, 512, 700, 1536, 4096, 4700, 32768, 100000):
        sizes = host_chunks(T)
        assert sum(sizes) == T and min(sizes) > 0 and len(sizes) <= 14
        if len(sizes) >= 4:
            assert sizes[0] == 64 and sizes[-1] == 64
    assert host_chunks(32768) == [64, 2496 - 64] + [2752] * 10 + [2752 - 64, 64]
    assert host_chunks(32768, unit=608) == [608, 2368 - 608] + [3040] * 9 + [3040 - 608, 608]


def test_indexer_topk_host_bytes_layout(api):
    # The device buffer holds every input and the indices, then one row
    # chunk's workspace, sized for the largest need over the chunks (a short
    # chunk of long rows can take the split top-k).
    ws = lambda rows, S, k: api.lib.dsa_workspace_bytes(api.DSA_OP_INDEXER_TOPK, rows, S, k)  # noqa: E731
    up = lambda x: -(-x // 256) * 256  # noqa: E731

    def expect(T, S, H, D, k, dtype):
        esz = 1 if dtype == api.DSA_E4M3 else 2
        need = max([ws(1, S, k)] + [ws(r, S, k) for r in host_chunks(T)])
        regions = [S * D * esz, S * 4 if dtype == api.DSA_E4M3 else 0, T * H * D * esz, T * H * 4,
                   T * H * 4, T * 4, T * 4, T * k * 4, need]
        return sum(up(r) for r in regions)

    nb = api.lib.dsa_indexer_topk_host_bytes
    for T, S, H, D, k, dt in [(4096, 4096, 64, 128, 2048, api.DSA_BF16),
                              (4700, 40000, 8, 64, 2048, api.DSA_BF16),
                              (700, 700, 8, 64, 64, api.DSA_BF16),
                              (1536, 1536, 64, 128, 512, api.DSA_E4M3),
                              (1, 5, 1, 64, 1, api.DSA_BF16),
                              (0, 64, 8, 64, 16, api.DSA_BF16)]:
        assert nb(T, S, H, D, k, dt) == expect(T, S, H, D, k, dt), (T, S)
    # 4700 rows: chunks of 64, 28, 8 x 512, 448 and 64 rows, which the
    # top-k takes with one 1024-thread CTA per row (32-512 rows, columns >
    # 16384), except the 28-row chunk: split scratch
    assert host_chunks(4700) == [64, 28] + [512] * 8 + [448, 64]
    assert api.lib.dsa_workspace_bytes(api.DSA_OP_TOPK, 64, 40000, 2048) == 0
    assert api.lib.dsa_workspace_bytes(api.DSA_OP_TOPK, 512, 40000, 2048) == 0
    assert api.lib.dsa_workspace_bytes(api.DSA_OP_TOPK, 28, 40000, 2048) > 0


def mx_call(api, q=A, qsf=A, k=A, ksf=A, w=A, rs=A, re=A, T=8, S=8, H=64, D=128, lg=A, ld=8,
            flags=0):
    return api.lib.dsa_indexer_logits_mxfp4(q, qsf, k, ksf, w, rs, re, T, S, H, D, lg, ld, flags,
                                            None)


def test_mxfp4_argument_errors(api):
    assert mx_call(api, q=NUL) == api.DSA_ERR_INVALID_ARG
    assert mx_call(api, qsf=NUL) == api.DSA_ERR_INVALID_ARG
    assert mx_call(api, ksf=NUL) == api.DSA_ERR_INVALID_ARG
    assert mx_call(api, q=MIS) == api.DSA_ERR_INVALID_ARG          # TMA needs 16 B
    assert mx_call(api, qsf=ctypes.c_void_p(0x10002)) == api.DSA_ERR_INVALID_ARG
    assert mx_call(api, H=32) == api.DSA_ERR_UNSUPPORTED             # 64 heads only
    assert mx_call(api, D=64) == api.DSA_ERR_UNSUPPORTED             # D = 128 only
    assert mx_call(api, ld=7) == api.DSA_ERR_INVALID_ARG             # ld < S
    assert mx_call(api, flags=4) == api.DSA_ERR_INVALID_ARG
    assert mx_call(api, T=-1) == api.DSA_ERR_INVALID_ARG
    assert mx_call(api, T=0) == api.DSA_OK                           # nothing to do, no launch
    f = api.lib.dsa_indexer_topk_mxfp4
    assert f(A, A, A, A, A, A, A, 8, 8, 64, 128, 0, A, A, 4096, None) == api.DSA_ERR_INVALID_ARG
    assert f(A, A, A, A, A, A, A, 8, 8, 64, 128, 4, NUL, A, 4096, None) == api.DSA_ERR_INVALID_ARG
    assert f(A, A, A, A, A, A, A, 8, 8, 64, 128, 4, A, NUL, 0, None) == api.DSA_ERR_INVALID_ARG
