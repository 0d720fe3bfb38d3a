"""CPU oracle for the DSA lightning-indexer path -- test infrastructure only.

Only the test-suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library
(``top_selection_dsa_gb300``) never imports it, and it never imports the
product library: the two share no code.  The only module both sides use is the
seeded input generator ``top_selection_dsa_gb300.workloads``, which holds none
of the method's arithmetic.

The arithmetic lives in ``dsa_oracle.c`` (plain C, fp64, straight from the
definitions; see its header for the sources and readings).  This module builds
it with gcc on first use and wraps it for numpy arrays.

Functions:
    logits(...)          dense prefill logits, fp64          (indexer score)
    logits_paged(...)    paged-decode logits, fp64           (indexer score)
    logits_mxfp4(...)    prefill logits of MXFP4 q/k (E2M1 + E8M0 block scales)
    paged_row_ranges()   the row ranges of paged decode
    topk(...)            masked per-row top-k of given fp32 logits
                         (torch_dsa_topk, vime PR #502, third review comment)
    sort_by_score(...)   a top-k index buffer in descending score order
    topk_merge(...)      per-rank (score, column) candidates -> the global top-k
    f64_to_e4m3()        E4M3 encoder (nearest, ties to even, saturating)
    q_quant_fold(...)    query quantisation + weight fold (before the indexer)
    k_norm_insert(...)   key LayerNorm + quantisation + paged insert
    k_layer_norm(...)    the key LayerNorm alone, fp64, before the bf16 cast
    bf16_to_f64 / e4m3_to_f64 / e2m1_to_f64 / e8m0_to_f64   element decoders
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dsa_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libdsa_oracle.so")
_lock = threading.Lock()
_lib = None

BF16 = 0
E4M3 = 1


def build(force: bool = False) -> str:
    """Compile dsa_oracle.c into a shared library (gcc, OpenMP)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC",
           "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        # DSA_ORACLE_LIB: a separately built copy of the same source (the
        # sanitizer test loads one built with -fsanitize=address,undefined).
        lib = ctypes.CDLL(os.environ.get("DSA_ORACLE_LIB") or build())
        P = ctypes.c_void_p
        i64 = ctypes.c_int64
        i32 = ctypes.c_int
        lib.dsa_oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.dsa_oracle_bf16_to_f64.restype = ctypes.c_double
        lib.dsa_oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        lib.dsa_oracle_e4m3_to_f64.restype = ctypes.c_double
        lib.dsa_oracle_logits.argtypes = [P, P, P, P, i32, P, P, P, i64, i64,
                                          i32, i32, P, i64, P, i32]
        lib.dsa_oracle_logits.restype = i32
        lib.dsa_oracle_paged_row_ranges.argtypes = [P, i32, i32, P, P]
        lib.dsa_oracle_paged_row_ranges.restype = i32
        lib.dsa_oracle_logits_paged.argtypes = [P, P, P, P, i32, P, P, i64, P,
                                                i32, i32, i32, i32, i32, P, i64,
                                                i64, P, i32]
        lib.dsa_oracle_logits_paged.restype = i32
        lib.dsa_oracle_topk.argtypes = [P, i64, P, P, i64, i64, i32, P, i32]
        lib.dsa_oracle_topk.restype = i32
        lib.dsa_oracle_f64_to_e4m3.argtypes = [ctypes.c_double]
        lib.dsa_oracle_f64_to_e4m3.restype = ctypes.c_uint8
        lib.dsa_oracle_q_quant_fold.argtypes = [P, P, ctypes.c_float, i32, i32, i32, i32, P, P]
        lib.dsa_oracle_q_quant_fold.restype = i32
        lib.dsa_oracle_k_norm_insert.argtypes = [P, P, P, ctypes.c_float, P, i32, i32, i32, i64,
                                                 P, P]
        lib.dsa_oracle_k_norm_insert.restype = i32
        lib.dsa_oracle_k_layer_norm.argtypes = [P, P, P, ctypes.c_float, i32, i32, P]
        lib.dsa_oracle_e2m1_to_f64.argtypes = [ctypes.c_uint8]
        lib.dsa_oracle_e2m1_to_f64.restype = ctypes.c_double
        lib.dsa_oracle_e8m0_to_f64.argtypes = [ctypes.c_uint8]
        lib.dsa_oracle_e8m0_to_f64.restype = ctypes.c_double
        lib.dsa_oracle_logits_mxfp4.argtypes = [P, P, P, P, P, P, P, i64, i64, i32, i32, P, i64,
                                                P, i32]
        lib.dsa_oracle_logits_mxfp4.restype = i32
        lib.dsa_oracle_k_layer_norm.restype = i32
        lib.dsa_oracle_max_threads.argtypes = []
        lib.dsa_oracle_max_threads.restype = i32
        _lib = lib
        return lib


def max_threads() -> int:
    return int(_load().dsa_oracle_max_threads())


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def _elems(x, dtype):
    """Element storage for the C side: bf16 as uint16 bits, e4m3 as uint8."""
    if dtype == BF16:
        return np.ascontiguousarray(x).view(np.uint16)
    if dtype == E4M3:
        return np.ascontiguousarray(x).view(np.uint8)
    raise ValueError(f"unknown dtype {dtype}")


def bf16_to_f64(bits) -> np.ndarray:
    lib = _load()
    b = np.asarray(bits, dtype=np.uint16).ravel()
    return np.array([lib.dsa_oracle_bf16_to_f64(int(v)) for v in b])


def e4m3_to_f64(codes) -> np.ndarray:
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8).ravel()
    return np.array([lib.dsa_oracle_e4m3_to_f64(int(v)) for v in c])


def logits(q, k, w, row_starts, row_ends, *, dtype=BF16, q_scale=None,
           k_scale=None, rows=None, nthreads=0) -> np.ndarray:
    """fp64 index logits [len(rows) or T, S]; -inf outside each row's range.

    q: [T, H, D] (uint16 bf16 bits or uint8 e4m3 codes), k: [S, D],
    w: [T, H] fp32, row_starts/row_ends: [T] int32.
    """
    qe = _elems(q, dtype)
    ke = _elems(k, dtype)
    T, H, D = qe.shape
    S = ke.shape[0]
    assert ke.shape[1] == D
    wf = _c(w, np.float32)
    assert wf.shape == (T, H)
    rs = _c(row_starts, np.int32)
    re_ = _c(row_ends, np.int32)
    qs = _c(q_scale, np.float32)
    ks = _c(k_scale, np.float32)
    rr = _c(rows, np.int64)
    n = T if rr is None else rr.shape[0]
    out = np.empty((n, S), dtype=np.float64)
    rc = _load().dsa_oracle_logits(_ptr(qe), _ptr(qs), _ptr(ke), _ptr(ks), dtype,
                                   _ptr(wf), _ptr(rs), _ptr(re_), T, S, H, D,
                                   _ptr(rr), n, _ptr(out), nthreads)
    if rc != 0:
        raise ValueError("oracle logits: bad arguments")
    return out


def e2m1_to_f64(codes) -> np.ndarray:
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8).ravel()
    return np.array([lib.dsa_oracle_e2m1_to_f64(int(v)) for v in c])


def e8m0_to_f64(codes) -> np.ndarray:
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8).ravel()
    return np.array([lib.dsa_oracle_e8m0_to_f64(int(v)) for v in c])


def logits_mxfp4(q, q_sf, k, k_sf, w, row_starts, row_ends, *, rows=None,
                 nthreads=0) -> np.ndarray:
    """fp64 index logits [len(rows) or T, S] of MXFP4 operands.

    q: [T, H, D/2] packed E2M1 (uint8, the low nibble is the even element),
    q_sf: [T, H, D/32] E8M0 codes, k: [S, D/2], k_sf: [S, D/32], w: [T, H].
    """
    qe = np.ascontiguousarray(q, dtype=np.uint8)
    ke = np.ascontiguousarray(k, dtype=np.uint8)
    T, H, D2 = qe.shape
    D = 2 * D2
    S = ke.shape[0]
    assert ke.shape[1] == D2
    qs = np.ascontiguousarray(q_sf, dtype=np.uint8)
    ks = np.ascontiguousarray(k_sf, dtype=np.uint8)
    assert qs.shape == (T, H, D // 32) and ks.shape == (S, D // 32)
    wf = _c(w, np.float32)
    rs = _c(row_starts, np.int32)
    re_ = _c(row_ends, np.int32)
    rr = _c(rows, np.int64)
    n = T if rr is None else rr.shape[0]
    out = np.empty((n, S), dtype=np.float64)
    rc = _load().dsa_oracle_logits_mxfp4(_ptr(qe), _ptr(qs), _ptr(ke), _ptr(ks), _ptr(wf),
                                         _ptr(rs), _ptr(re_), T, S, H, D, _ptr(rr), n,
                                         _ptr(out), nthreads)
    if rc != 0:
        raise ValueError("oracle logits_mxfp4: bad arguments")
    return out


def paged_row_ranges(context_lens, next_n):
    cl = _c(context_lens, np.int32)
    B = cl.shape[0]
    rs = np.empty(B * next_n, dtype=np.int32)
    re_ = np.empty(B * next_n, dtype=np.int32)
    rc = _load().dsa_oracle_paged_row_ranges(_ptr(cl), B, next_n, _ptr(rs), _ptr(re_))
    if rc != 0:
        raise ValueError("oracle paged_row_ranges: bad arguments")
    return rs, re_


def logits_paged(q, w, k_cache, block_table, context_lens, *, next_n,
                 dtype=BF16, q_scale=None, k_scale=None, ld=None, rows=None,
                 nthreads=0) -> np.ndarray:
    """fp64 paged-decode logits [len(rows) or B*next_n, ld] over logical keys.

    q: [B*next_n, H, D], w: [B*next_n, H], k_cache: [num_blocks, block, D],
    block_table: [B, max_blocks] int32, context_lens: [B] int32.
    """
    qe = _elems(q, dtype)
    kc = _elems(k_cache, dtype)
    R, H, D = qe.shape
    _, block_size, D2 = kc.shape
    assert D2 == D
    bt = _c(block_table, np.int32)
    B, max_blocks = bt.shape
    assert R == B * next_n
    cl = _c(context_lens, np.int32)
    if ld is None:
        ld = int(cl.max()) if B else 0
    wf = _c(w, np.float32)
    qs = _c(q_scale, np.float32)
    ks = _c(k_scale, np.float32)
    rr = _c(rows, np.int64)
    n = R if rr is None else rr.shape[0]
    out = np.empty((n, ld), dtype=np.float64)
    rc = _load().dsa_oracle_logits_paged(
        _ptr(qe), _ptr(qs), _ptr(kc), _ptr(ks), dtype, _ptr(wf), _ptr(bt),
        max_blocks, _ptr(cl), B, next_n, block_size, H, D, _ptr(rr), n, ld,
        _ptr(out), nthreads)
    if rc != 0:
        raise ValueError("oracle logits_paged: bad arguments")
    return out


def topk(logits_f32, row_starts, row_ends, k, *, S=None, nthreads=0) -> np.ndarray:
    """Masked top-k [T, k] int32 of given fp32 logits [T, ld].

    Columns [0, S) are considered (S defaults to the row length).
    """
    lg = np.ascontiguousarray(logits_f32, dtype=np.float32)
    T, ld = lg.shape
    if S is None:
        S = ld
    rs = _c(row_starts, np.int32)
    re_ = _c(row_ends, np.int32)
    out = np.empty((T, k), dtype=np.int32)
    rc = _load().dsa_oracle_topk(_ptr(lg), ld, _ptr(rs), _ptr(re_), T, S, k,
                                 _ptr(out), nthreads)
    if rc != 0:
        raise ValueError("oracle topk: bad arguments")
    return out


def sort_by_score(logits_f32, topk_idx) -> np.ndarray:
    """Rows of a top-k index buffer [T, k] in descending order of their score.

    torch_dsa_topk (vime PR #502, third review comment) takes torch.topk,
    whose indices come in descending order of value; the library's canonical
    output is ascending column order instead, and this puts a row back into
    score order.  Reading where the page is silent: equal scores keep
    ascending column order (-0.0 equals +0.0), -inf and NaN scores (which
    no top-k selects) count as equal and lowest, and the -1 padding stays at
    the tail.  Plain numpy: one stable two-key sort per row.
    """
    lg = np.asarray(logits_f32, dtype=np.float32)
    idx = np.asarray(topk_idx, dtype=np.int32)
    out = np.full_like(idx, -1)
    for t in range(idx.shape[0]):
        cols = idx[t][idx[t] >= 0]
        v = lg[t, cols].astype(np.float64)
        v = np.where(np.isnan(v) | (v == -np.inf), -np.inf, v)
        v = np.where(v == 0.0, 0.0, v)                 # -0.0 -> +0.0
        order = np.lexsort((cols, -v))                  # score descending, then column ascending
        out[t, :cols.size] = cols[order]
    return out


def f64_to_e4m3(values) -> np.ndarray:
    """E4M3 codes of the given values (uint8): the nearest code, ties to even."""
    lib = _load()
    v = np.asarray(values, dtype=np.float64).ravel()
    return np.array([lib.dsa_oracle_f64_to_e4m3(float(x)) for x in v], dtype=np.uint8)


def q_quant_fold(q_bf16_bits, weights, weight_scale, padded_heads):
    """q [T,H,D] bf16 bits -> (e4m3 codes [T,Hp,D], folded weights [T,Hp])."""
    q = np.ascontiguousarray(q_bf16_bits).view(np.uint16)
    T, H, D = q.shape
    w = _c(weights, np.float32)
    q8 = np.empty((T, padded_heads, D), np.uint8)
    wo = np.empty((T, padded_heads), np.float32)
    rc = _load().dsa_oracle_q_quant_fold(_ptr(q), _ptr(w), float(weight_scale), T, H, D,
                                         padded_heads, _ptr(q8), _ptr(wo))
    if rc != 0:
        raise ValueError("oracle q_quant_fold: bad arguments")
    return q8, wo


def k_norm_insert(k_bf16_bits, ln_weight, ln_bias, eps, slots, cache, scale=None):
    """LayerNorm + cast to bf16 (+ e4m3 quantisation when scale is given) of
    k [T,D] bf16 bits into cache [num_blocks, block_size, D] (uint16 bf16
    bits, or uint8 e4m3 codes with scale [num_blocks*block_size]), in place."""
    k = np.ascontiguousarray(k_bf16_bits).view(np.uint16)
    T, D = k.shape
    g, b = _c(ln_weight, np.float32), _c(ln_bias, np.float32)
    sl = _c(slots, np.int64)
    assert cache.flags.c_contiguous and (scale is None or scale.flags.c_contiguous)
    dtype = 0 if scale is None else 1
    capacity = cache.shape[0] * cache.shape[1]
    rc = _load().dsa_oracle_k_norm_insert(_ptr(k), _ptr(g), _ptr(b), float(eps), _ptr(sl), T, D,
                                          dtype, capacity, _ptr(cache), _ptr(scale))
    if rc != 0:
        raise ValueError("oracle k_norm_insert: bad arguments")
    return cache, scale


def k_layer_norm(k_bf16_bits, ln_weight, ln_bias, eps) -> np.ndarray:
    """The key LayerNorm of k [T,D] bf16 bits in fp64, before the cast back
    to bf16 that k_norm_insert applies: [T,D] float64."""
    k = np.ascontiguousarray(k_bf16_bits).view(np.uint16)
    T, D = k.shape
    g, b = _c(ln_weight, np.float32), _c(ln_bias, np.float32)
    out = np.empty((T, D), np.float64)
    rc = _load().dsa_oracle_k_layer_norm(_ptr(k), _ptr(g), _ptr(b), float(eps), T, D, _ptr(out))
    if rc != 0:
        raise ValueError("oracle k_layer_norm: bad arguments")
    return out


def topk_merge(cand_scores, cand_cols, k) -> np.ndarray:
    """The k best of each row's (score, column) candidates [T, C]: valid ones
    (column >= 0, score neither -inf nor NaN) ordered by score descending, ties
    to the lower column (-0.0 equals +0.0); written in ascending column order,
    -1 padding.  The definition of the global top-k applied to the union of
    the ranks' candidates (decode context parallelism, vLLM page)."""
    sc = np.asarray(cand_scores, dtype=np.float32)
    cc = np.asarray(cand_cols, dtype=np.int64)
    out = np.full((sc.shape[0], k), -1, np.int32)
    for t in range(sc.shape[0]):
        v = sc[t].astype(np.float64)
        ok = (cc[t] >= 0) & ~np.isnan(v) & (v != -np.inf)
        cols, vals = cc[t][ok], np.where(v[ok] == 0.0, 0.0, v[ok])
        take = cols[np.lexsort((cols, -vals))][:k]
        out[t, :take.size] = np.sort(take)
    return out
