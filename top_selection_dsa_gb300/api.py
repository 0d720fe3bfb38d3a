"""Thin ctypes binding over libdsa.so (include/dsa.h).

Argument marshalling only: every function checks that its torch tensors are
CUDA (host tensors for indexer_topk_host), contiguous and of the documented
dtype, then passes raw pointers, sizes and the current CUDA stream of the
tensors' device to the C ABI, with that device current for the call.  All arithmetic runs in the
library's kernels.  Importing this module loads libdsa.so and raises if it has
not been built -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdsa.so")

# Mirrors of the enums in include/dsa.h.
DSA_OK, DSA_ERR_INVALID_ARG, DSA_ERR_UNSUPPORTED, DSA_ERR_CUDA, DSA_ERR_TIMEOUT = range(5)
DSA_BF16, DSA_E4M3 = 0, 1
(DSA_OP_INDEXER_LOGITS, DSA_OP_TOPK, DSA_OP_INDEXER_TOPK, DSA_OP_INDEXER_LOGITS_PAGED,
 DSA_OP_INDEXER_TOPK_PAGED) = range(5)
DSA_LOGITS_CLEAN = 1

# Every entry point of include/dsa.h.
EXPORTS = (
    "dsa_indexer_logits", "dsa_topk", "dsa_indexer_topk", "dsa_indexer_logits_paged",
    "dsa_indexer_topk_paged", "dsa_workspace_bytes", "dsa_status_string",
    "dsa_get_last_device_error", "dsa_selftest_wait_timeout", "dsa_indexer_topk_noalloc",
    "dsa_topk_sort_by_score", "dsa_q_quant_fold_weights", "dsa_k_norm_quant_insert",
    "dsa_topk_merge", "dsa_indexer_topk_host_bytes", "dsa_indexer_topk_host",
    "dsa_indexer_logits_mxfp4", "dsa_indexer_topk_mxfp4", "dsa_topk_merge_ranks",
    "dsa_topk_dcp_candidates",
)


class DSAError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is not built: run `python -m top_selection_dsa_gb300.build` "
            "(nvcc, sm_103a). There is no CPU fallback.")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, I64, U32, U64, SZ = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint32,
                               ctypes.c_uint64, ctypes.c_size_t)
    lib.dsa_indexer_logits.argtypes = [P, P, P, P, I, P, P, P, I, I, I, I, P, I64, U32, P]
    lib.dsa_topk.argtypes = [P, I64, P, P, I, I, I, P, P, SZ, P]
    lib.dsa_indexer_topk.argtypes = [P, P, P, P, I, P, P, P, I, I, I, I, I, P, P, SZ, P]
    lib.dsa_indexer_logits_paged.argtypes = [P, P, P, P, P, I, I, P, I, P, I, I, I, I, I, P,
                                             I64, P]
    lib.dsa_indexer_topk_paged.argtypes = [P, P, P, P, P, I, I, P, I, P, I, I, I, I, I, I, P,
                                           P, SZ, P]
    lib.dsa_workspace_bytes.argtypes = [I, I64, I64, I]
    lib.dsa_workspace_bytes.restype = SZ
    lib.dsa_status_string.argtypes = [I]
    lib.dsa_status_string.restype = ctypes.c_char_p
    lib.dsa_get_last_device_error.argtypes = []
    lib.dsa_selftest_wait_timeout.argtypes = [U64, P]
    lib.dsa_topk_sort_by_score.argtypes = [P, I64, P, I, I, P]
    F = ctypes.c_float
    lib.dsa_q_quant_fold_weights.argtypes = [P, P, F, I, I, I, I, P, P, P]
    lib.dsa_k_norm_quant_insert.argtypes = [P, P, P, F, P, I, I, I, P, P, I, I, P]
    lib.dsa_topk_merge.argtypes = [P, P, I, I, I, P, P]
    lib.dsa_topk_merge_ranks.argtypes = [P, P, I, I, I, I, P, P]
    lib.dsa_topk_dcp_candidates.argtypes = [P, I64, P, P, I, I, I, I, I, I, P, P, P, SZ, P]
    lib.dsa_indexer_topk_host_bytes.argtypes = [I, I, I, I, I, I]
    lib.dsa_indexer_topk_host_bytes.restype = SZ
    lib.dsa_indexer_topk_host.argtypes = [P, P, P, P, I, P, P, P, I, I, I, I, I, P, P, SZ, P]
    lib.dsa_indexer_logits_mxfp4.argtypes = [P, P, P, P, P, P, P, I, I, I, I, P, I64, U32, P]
    lib.dsa_indexer_topk_mxfp4.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, P, P, SZ, P]
    for name in ("dsa_indexer_logits_mxfp4", "dsa_indexer_topk_mxfp4"):
        getattr(lib, name).restype = I
    for name in ("dsa_indexer_logits", "dsa_topk", "dsa_indexer_topk",
                 "dsa_indexer_logits_paged", "dsa_indexer_topk_paged",
                 "dsa_get_last_device_error", "dsa_selftest_wait_timeout",
                 "dsa_topk_sort_by_score", "dsa_q_quant_fold_weights",
                 "dsa_k_norm_quant_insert", "dsa_topk_merge", "dsa_indexer_topk_host"):
        getattr(lib, name).restype = I
    return lib


lib = _load()


def status_string(status: int) -> str:
    return lib.dsa_status_string(int(status)).decode()


def _check(status: int, what: str):
    if status != DSA_OK:
        raise DSAError(status, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need(t, name, dtypes, device=None):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.dtype not in dtypes:
        raise ValueError(f"{name} must have dtype in {dtypes}, got {t.dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


_E4M3_TYPES = (torch.float8_e4m3fn, torch.uint8)


def _elem_dtype(q, k):
    if q.dtype == torch.bfloat16 and k.dtype == torch.bfloat16:
        return DSA_BF16
    if q.dtype in _E4M3_TYPES and k.dtype in _E4M3_TYPES:
        return DSA_E4M3
    raise ValueError(f"q/k must both be bf16 or both e4m3, got {q.dtype}/{k.dtype}")


def workspace_bytes(op: int, rows: int, cols: int, k: int) -> int:
    n = lib.dsa_workspace_bytes(op, rows, cols, k)
    if n == ctypes.c_size_t(-1).value:
        raise ValueError("dsa_workspace_bytes: bad arguments")
    return int(n)


def _workspace(nbytes, device, workspace):
    if nbytes == 0:
        return workspace
    if workspace is None:
        return torch.empty(nbytes, dtype=torch.uint8, device=device)
    if workspace.numel() * workspace.element_size() < nbytes:
        raise ValueError(f"workspace holds {workspace.numel() * workspace.element_size()} "
                         f"bytes, {nbytes} needed")
    return workspace


def indexer_logits(q, k, weights, row_starts, row_ends, *, q_scale=None, k_scale=None,
                   logits=None, clean=False):
    """fp32 index logits [T, ld] (ld = logits.shape[1] if given, else S)."""
    dt = _elem_dtype(q, k)
    T, H, D = q.shape
    S = k.shape[0]
    dev = q.device
    for t, n, d in ((q, "q", (q.dtype,)), (k, "k", (k.dtype,)), (weights, "weights", (torch.float32,)),
                    (row_starts, "row_starts", (torch.int32,)), (row_ends, "row_ends", (torch.int32,)),
                    (q_scale, "q_scale", (torch.float32,)), (k_scale, "k_scale", (torch.float32,))):
        _need(t, n, d, dev)
    if logits is None:
        logits = torch.empty((T, S), dtype=torch.float32, device=dev)
    _need(logits, "logits", (torch.float32,), dev)
    with torch.cuda.device(dev):
        st = lib.dsa_indexer_logits(_ptr(q), _ptr(q_scale), _ptr(k), _ptr(k_scale), dt,
                                    _ptr(weights), _ptr(row_starts), _ptr(row_ends), T, S, H, D,
                                    _ptr(logits), logits.shape[1] if logits.dim() == 2 else S,
                                    DSA_LOGITS_CLEAN if clean else 0, _stream(dev))
    _check(st, "dsa_indexer_logits")
    return logits


def topk(logits, row_starts, row_ends, k, *, S=None, out=None, workspace=None):
    """Masked top-k [T, k] int32 of fp32 logits [T, ld] over columns [0, S)."""
    T, ld = logits.shape
    S = ld if S is None else S
    dev = logits.device
    _need(logits, "logits", (torch.float32,), dev)
    _need(row_starts, "row_starts", (torch.int32,), dev)
    _need(row_ends, "row_ends", (torch.int32,), dev)
    if out is None:
        out = torch.empty((T, k), dtype=torch.int32, device=dev)
    _need(out, "out", (torch.int32,), dev)
    nbytes = workspace_bytes(DSA_OP_TOPK, T, S, k)
    ws = _workspace(nbytes, dev, workspace)
    with torch.cuda.device(dev):
        st = lib.dsa_topk(_ptr(logits), ld, _ptr(row_starts), _ptr(row_ends), T, S, k, _ptr(out),
                          _ptr(ws) if nbytes else None, nbytes, _stream(dev))
    _check(st, "dsa_topk")
    return out


def indexer_topk(q, k, weights, row_starts, row_ends, topk_k, *, q_scale=None, k_scale=None,
                 out=None, workspace=None):
    """Index logits + masked top-k in one library call: [T, topk_k] int32."""
    dt = _elem_dtype(q, k)
    T, H, D = q.shape
    S = k.shape[0]
    dev = q.device
    for t, n, d in ((q, "q", (q.dtype,)), (k, "k", (k.dtype,)), (weights, "weights", (torch.float32,)),
                    (row_starts, "row_starts", (torch.int32,)), (row_ends, "row_ends", (torch.int32,)),
                    (q_scale, "q_scale", (torch.float32,)), (k_scale, "k_scale", (torch.float32,))):
        _need(t, n, d, dev)
    if out is None:
        out = torch.empty((T, topk_k), dtype=torch.int32, device=dev)
    _need(out, "out", (torch.int32,), dev)
    nbytes = workspace_bytes(DSA_OP_INDEXER_TOPK, T, S, topk_k)
    ws = _workspace(nbytes, dev, workspace)
    with torch.cuda.device(dev):
        st = lib.dsa_indexer_topk(_ptr(q), _ptr(q_scale), _ptr(k), _ptr(k_scale), dt, _ptr(weights),
                                  _ptr(row_starts), _ptr(row_ends), T, S, H, D, topk_k, _ptr(out),
                                  _ptr(ws), nbytes, _stream(dev))
    _check(st, "dsa_indexer_topk")
    return out


def _mx_common(q, q_sf, k, k_sf, weights, row_starts, row_ends):
    dev = q.device
    for t, n, d in ((q, "q", (torch.uint8,)), (q_sf, "q_sf", (torch.uint8,)),
                    (k, "k", (torch.uint8,)), (k_sf, "k_sf", (torch.uint8,)),
                    (weights, "weights", (torch.float32,)),
                    (row_starts, "row_starts", (torch.int32,)),
                    (row_ends, "row_ends", (torch.int32,))):
        _need(t, n, d, dev)
    T, H, D2 = q.shape
    return dev, T, H, 2 * D2, k.shape[0]


def indexer_logits_mxfp4(q, q_sf, k, k_sf, weights, row_starts, row_ends, *, logits=None,
                         clean=False):
    """fp32 index logits [T, ld] of MXFP4 operands: q [T,H,D/2] and k [S,D/2]
    packed E2M1 (uint8), q_sf [T,H,D/32] and k_sf [S,D/32] E8M0 scale bytes."""
    dev, T, H, D, S = _mx_common(q, q_sf, k, k_sf, weights, row_starts, row_ends)
    if logits is None:
        logits = torch.empty((T, S), dtype=torch.float32, device=dev)
    _need(logits, "logits", (torch.float32,), dev)
    with torch.cuda.device(dev):
        st = lib.dsa_indexer_logits_mxfp4(_ptr(q), _ptr(q_sf), _ptr(k), _ptr(k_sf),
                                          _ptr(weights), _ptr(row_starts), _ptr(row_ends), T, S,
                                          H, D, _ptr(logits),
                                          logits.shape[1] if logits.dim() == 2 else S,
                                          DSA_LOGITS_CLEAN if clean else 0, _stream(dev))
    _check(st, "dsa_indexer_logits_mxfp4")
    return logits


def indexer_topk_mxfp4(q, q_sf, k, k_sf, weights, row_starts, row_ends, topk_k, *, out=None,
                       workspace=None):
    """MXFP4 index logits + masked top-k in one library call: [T, topk_k] int32."""
    dev, T, H, D, S = _mx_common(q, q_sf, k, k_sf, weights, row_starts, row_ends)
    if out is None:
        out = torch.empty((T, topk_k), dtype=torch.int32, device=dev)
    _need(out, "out", (torch.int32,), dev)
    nbytes = workspace_bytes(DSA_OP_INDEXER_TOPK, T, S, topk_k)
    ws = _workspace(nbytes, dev, workspace)
    with torch.cuda.device(dev):
        st = lib.dsa_indexer_topk_mxfp4(_ptr(q), _ptr(q_sf), _ptr(k), _ptr(k_sf), _ptr(weights),
                                        _ptr(row_starts), _ptr(row_ends), T, S, H, D, topk_k,
                                        _ptr(out), _ptr(ws), nbytes, _stream(dev))
    _check(st, "dsa_indexer_topk_mxfp4")
    return out


def _need_host(t, name, dtypes):
    if t is None:
        return
    if t.is_cuda:
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.dtype not in dtypes:
        raise ValueError(f"{name} must have dtype in {dtypes}, got {t.dtype}")


def indexer_topk_host_bytes(T, S, H, D, topk_k, dtype=DSA_BF16) -> int:
    n = lib.dsa_indexer_topk_host_bytes(T, S, H, D, topk_k, dtype)
    if n == ctypes.c_size_t(-1).value:
        raise ValueError("dsa_indexer_topk_host_bytes: bad arguments")
    return int(n)


def indexer_topk_host(q, k, weights, row_starts, row_ends, topk_k, *, q_scale=None,
                      k_scale=None, out=None, device_buffer=None, device=None):
    """indexer_topk on HOST tensors (pin them for overlap): [T, topk_k] int32 on the host.

    The library uploads the inputs in row chunks, scores and selects on the
    GPU, and downloads the indices, overlapping the three; the call returns
    after the current stream has finished.
    """
    dt = _elem_dtype(q, k)
    T, H, D = q.shape
    S = k.shape[0]
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else \
        torch.device(device)
    for t, n, d in ((q, "q", (q.dtype,)), (k, "k", (k.dtype,)), (weights, "weights", (torch.float32,)),
                    (row_starts, "row_starts", (torch.int32,)), (row_ends, "row_ends", (torch.int32,)),
                    (q_scale, "q_scale", (torch.float32,)), (k_scale, "k_scale", (torch.float32,))):
        _need_host(t, n, d)
    if out is None:
        out = torch.empty((T, topk_k), dtype=torch.int32, pin_memory=True)
    _need_host(out, "out", (torch.int32,))
    nbytes = indexer_topk_host_bytes(T, S, H, D, topk_k, dt)
    if device_buffer is None:
        device_buffer = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev)
    _need(device_buffer, "device_buffer", (torch.uint8,), dev)
    if device_buffer.numel() < nbytes:
        raise ValueError(f"device_buffer holds {device_buffer.numel()} bytes, {nbytes} needed")
    with torch.cuda.device(dev):
        st = lib.dsa_indexer_topk_host(_ptr(q), _ptr(q_scale), _ptr(k), _ptr(k_scale), dt,
                                       _ptr(weights), _ptr(row_starts), _ptr(row_ends), T, S, H, D,
                                       topk_k, _ptr(out), _ptr(device_buffer), nbytes, _stream(dev))
    _check(st, "dsa_indexer_topk_host")
    torch.cuda.current_stream(dev).synchronize()
    return out


def _paged_common(q, weights, k_cache, block_table, context_lens, q_scale, k_scale):
    dt = _elem_dtype(q, k_cache)
    dev = q.device
    for t, n, d in ((q, "q", (q.dtype,)), (k_cache, "k_cache", (k_cache.dtype,)),
                    (weights, "weights", (torch.float32,)),
                    (block_table, "block_table", (torch.int32,)),
                    (context_lens, "context_lens", (torch.int32,)),
                    (q_scale, "q_scale", (torch.float32,)), (k_scale, "k_scale", (torch.float32,))):
        _need(t, n, d, dev)
    return dt, dev


def indexer_logits_paged(q, weights, k_cache, block_table, context_lens, *, next_n,
                         q_scale=None, k_scale=None, logits=None):
    """Paged-decode logits [B*next_n, ld] over logical key positions."""
    dt, dev = _paged_common(q, weights, k_cache, block_table, context_lens, q_scale, k_scale)
    R, H, D = q.shape
    num_blocks, block_size, _ = k_cache.shape
    B, max_blocks = block_table.shape
    if logits is None:
        logits = torch.empty((R, max_blocks * block_size), dtype=torch.float32, device=dev)
    _need(logits, "logits", (torch.float32,), dev)
    with torch.cuda.device(dev):
        st = lib.dsa_indexer_logits_paged(_ptr(q), _ptr(q_scale), _ptr(weights), _ptr(k_cache),
                                          _ptr(k_scale), num_blocks, dt, _ptr(block_table),
                                          max_blocks, _ptr(context_lens), B, next_n, block_size, H,
                                          D, _ptr(logits), logits.shape[1], _stream(dev))
    _check(st, "dsa_indexer_logits_paged")
    return logits


def indexer_topk_paged(q, weights, k_cache, block_table, context_lens, topk_k, *, next_n,
                       q_scale=None, k_scale=None, out=None, workspace=None):
    """Paged-decode logits + masked top-k: [B*next_n, topk_k] logical positions."""
    dt, dev = _paged_common(q, weights, k_cache, block_table, context_lens, q_scale, k_scale)
    R, H, D = q.shape
    num_blocks, block_size, _ = k_cache.shape
    B, max_blocks = block_table.shape
    if out is None:
        out = torch.empty((R, topk_k), dtype=torch.int32, device=dev)
    _need(out, "out", (torch.int32,), dev)
    nbytes = workspace_bytes(DSA_OP_INDEXER_TOPK_PAGED, R, max_blocks * block_size, topk_k)
    ws = _workspace(nbytes, dev, workspace)
    with torch.cuda.device(dev):
        st = lib.dsa_indexer_topk_paged(_ptr(q), _ptr(q_scale), _ptr(weights), _ptr(k_cache),
                                        _ptr(k_scale), num_blocks, dt, _ptr(block_table),
                                        max_blocks, _ptr(context_lens), B, next_n, block_size, H,
                                        D, topk_k, _ptr(out), _ptr(ws), nbytes, _stream(dev))
    _check(st, "dsa_indexer_topk_paged")
    return out


def topk_sort_by_score(logits, topk_idx):
    """Rows of a top-k index buffer [T, k] reordered in place into descending
    score order (ties to the lower column, -1 padding at the tail)."""
    dev = topk_idx.device
    _need(logits, "logits", (torch.float32,), dev)
    _need(topk_idx, "topk_idx", (torch.int32,), dev)
    if logits.dim() != 2 or topk_idx.dim() != 2 or logits.shape[0] != topk_idx.shape[0]:
        raise ValueError("logits [T, ld] and topk_idx [T, k] expected")
    if logits.stride(1) != 1 or not topk_idx.is_contiguous():
        raise ValueError("row-major logits and a contiguous topk_idx expected")
    T, k = topk_idx.shape
    with torch.cuda.device(dev):
        st = lib.dsa_topk_sort_by_score(_ptr(logits), logits.stride(0), _ptr(topk_idx), T, k,
                                        _stream(dev))
    _check(st, "dsa_topk_sort_by_score")
    return topk_idx


def topk_merge(cand_scores, cand_cols, k, *, out=None):
    """[T, C] (score, global column) candidates -> the [T, k] global top-k,
    ascending columns, -1 padding (negative columns are empty slots)."""
    dev = cand_scores.device
    _need(cand_scores, "cand_scores", (torch.float32,), dev)
    _need(cand_cols, "cand_cols", (torch.int32,), dev)
    T, C = cand_scores.shape
    if tuple(cand_cols.shape) != (T, C):
        raise ValueError("cand_scores and cand_cols must have the same [T, C] shape")
    if out is None:
        out = torch.empty((T, k), dtype=torch.int32, device=dev)
    _need(out, "out", (torch.int32,), dev)
    with torch.cuda.device(dev):
        st = lib.dsa_topk_merge(_ptr(cand_scores), _ptr(cand_cols), T, C, int(k), _ptr(out),
                                _stream(dev))
    _check(st, "dsa_topk_merge")
    return out


def topk_merge_ranks(cand_scores, cand_cols, k, *, out=None):
    """[W, T, kr] rank-major (score, global column) candidates -> the [T, k]
    global top-k, ascending columns, -1 padding."""
    dev = cand_scores.device
    _need(cand_scores, "cand_scores", (torch.float32,), dev)
    _need(cand_cols, "cand_cols", (torch.int32,), dev)
    W, T, kr = cand_scores.shape
    if tuple(cand_cols.shape) != (W, T, kr):
        raise ValueError("cand_scores and cand_cols must have the same [W, T, kr] shape")
    if out is None:
        out = torch.empty((T, k), dtype=torch.int32, device=dev)
    _need(out, "out", (torch.int32,), dev)
    with torch.cuda.device(dev):
        st = lib.dsa_topk_merge_ranks(_ptr(cand_scores), _ptr(cand_cols), W, T, kr, int(k),
                                      _ptr(out), _stream(dev))
    _check(st, "dsa_topk_merge_ranks")
    return out


def topk_dcp_candidates(logits, row_starts, row_ends, k, rank, world, interleave, *, S=None,
                        scores=None, cols=None, workspace=None):
    """A rank's masked top-k of its local logits [T, ld] as (score, global
    position) pairs, [T, k] each (-inf / -1 in empty slots)."""
    T, ld = logits.shape
    S = ld if S is None else S
    dev = logits.device
    _need(logits, "logits", (torch.float32,), dev)
    _need(row_starts, "row_starts", (torch.int32,), dev)
    _need(row_ends, "row_ends", (torch.int32,), dev)
    if scores is None:
        scores = torch.empty((T, k), dtype=torch.float32, device=dev)
    if cols is None:
        cols = torch.empty((T, k), dtype=torch.int32, device=dev)
    _need(scores, "scores", (torch.float32,), dev)
    _need(cols, "cols", (torch.int32,), dev)
    nbytes = workspace_bytes(DSA_OP_TOPK, T, S, k)
    ws = _workspace(nbytes, dev, workspace)
    with torch.cuda.device(dev):
        st = lib.dsa_topk_dcp_candidates(_ptr(logits), ld, _ptr(row_starts), _ptr(row_ends), T, S,
                                         int(k), int(rank), int(world), int(interleave),
                                         _ptr(scores), _ptr(cols), _ptr(ws) if nbytes else None,
                                         nbytes, _stream(dev))
    _check(st, "dsa_topk_dcp_candidates")
    return scores, cols


def q_quant_fold_weights(q, weights, weight_scale, padded_heads=None, *, q_fp8=None,
                         weights_out=None):
    """bf16 q [T,H,128] -> (e4m3 q [T,Hp,128], fp32 weights [T,Hp]) with each
    row's UE8M0 scale and weight_scale folded into the weights."""
    dev = q.device
    _need(q, "q", (torch.bfloat16,), dev)
    _need(weights, "weights", (torch.float32,), dev)
    T, H, D = q.shape
    Hp = H if padded_heads is None else int(padded_heads)
    if q_fp8 is None:
        q_fp8 = torch.empty((T, Hp, D), dtype=torch.float8_e4m3fn, device=dev)
    if weights_out is None:
        weights_out = torch.empty((T, Hp), dtype=torch.float32, device=dev)
    _need(q_fp8, "q_fp8", (torch.float8_e4m3fn, torch.uint8), dev)
    _need(weights_out, "weights_out", (torch.float32,), dev)
    with torch.cuda.device(dev):
        st = lib.dsa_q_quant_fold_weights(_ptr(q), _ptr(weights), float(weight_scale), T, H, D, Hp,
                                          _ptr(q_fp8), _ptr(weights_out), _stream(dev))
    _check(st, "dsa_q_quant_fold_weights")
    return q_fp8, weights_out


def k_norm_quant_insert(k, ln_weight, ln_bias, eps, slot_mapping, k_cache, k_scale=None):
    """LayerNorm the new keys k [T,128] (bf16) and write them to their slots of
    the paged cache k_cache [num_blocks, block_size, 128]: bf16, or e4m3 codes
    with k_scale [num_blocks*block_size] for an e4m3 cache.  In place."""
    dev = k.device
    _need(k, "k", (torch.bfloat16,), dev)
    _need(ln_weight, "ln_weight", (torch.float32,), dev)
    _need(ln_bias, "ln_bias", (torch.float32,), dev)
    _need(slot_mapping, "slot_mapping", (torch.int64,), dev)
    _need(k_cache, "k_cache", (torch.bfloat16, torch.float8_e4m3fn, torch.uint8), dev)
    _need(k_scale, "k_scale", (torch.float32,), dev)
    T, D = k.shape
    num_blocks, block_size = k_cache.shape[0], k_cache.shape[1]
    dt = DSA_BF16 if k_cache.dtype == torch.bfloat16 else DSA_E4M3
    with torch.cuda.device(dev):
        st = lib.dsa_k_norm_quant_insert(_ptr(k), _ptr(ln_weight), _ptr(ln_bias), float(eps),
                                         _ptr(slot_mapping), T, D, dt, _ptr(k_cache), _ptr(k_scale),
                                         num_blocks, block_size, _stream(dev))
    _check(st, "dsa_k_norm_quant_insert")
    return k_cache, k_scale


def last_device_error() -> int:
    """Synchronise and return (then clear) the device error word as a status."""
    return int(lib.dsa_get_last_device_error())


def selftest_wait_timeout(timeout_ns: int, device=None):
    dev = torch.device("cuda") if device is None else device
    _check(lib.dsa_selftest_wait_timeout(int(timeout_ns), _stream(dev)),
           "dsa_selftest_wait_timeout")
