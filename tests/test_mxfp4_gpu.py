"""MXFP4 queries and keys (E2M1 elements, E8M0 scales per 32 elements) on the
GPU through the C ABI, against the oracle.

Bars as for the other element types: logits within 2e-2 relative + 1e-3
absolute of the fp64 oracle on the decoded operands; the top-k bit-exact with
the oracle's top-k of the GPU's own logits.
"""
import numpy as np
import pytest
import torch

import oracle
from top_selection_dsa_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

RTOL, ATOL = 2e-2, 1e-3


@pytest.fixture(scope="module")
def api():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from top_selection_dsa_gb300 import api as _api
    return _api


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def inputs(p):
    return (dev(p.q), dev(p.q_sf), dev(p.k), dev(p.k_sf), dev(p.w), dev(p.row_starts),
            dev(p.row_ends))


def assert_close(gpu, ref, what):
    g = np.asarray(gpu, np.float64)
    r = np.asarray(ref, np.float64)
    ninf = np.isneginf(r)
    assert (np.isneginf(g) == ninf).all(), f"{what}: -inf pattern"
    err = np.abs(g[~ninf] - r[~ninf])
    bound = ATOL + RTOL * np.abs(r[~ninf])
    assert (err <= bound).all(), f"{what}: max excess {float((err - bound).max()):.3g}"


def oracle_logits(p, rows=None):
    return oracle.logits_mxfp4(p.q, p.q_sf, p.k, p.k_sf, p.w, p.row_starts, p.row_ends, rows=rows)


@pytest.mark.parametrize("T", [333, 334, 335])   # groups of three rows: all three remainders
def test_mxfp4_small_causal_ragged(api, T):
    p = wl.prefill_mx(T, T, 64, 128, 40, seed=50)         # several tiles, ragged tail
    t = inputs(p)
    lg = api.indexer_logits_mxfp4(*t, clean=True)
    g = lg.cpu().numpy()
    assert_close(g, oracle_logits(p), "mxfp4 causal")
    got = api.indexer_topk_mxfp4(*t, p.topk).cpu().numpy()
    assert np.array_equal(got, oracle.topk(g, p.row_starts, p.row_ends, p.topk))


def test_mxfp4_ranges_thd_and_unclean_buffer(api):
    lens = [130, 1, 400, 257]
    rs, re = wl.thd_ranges(lens)
    T = sum(lens)
    p = wl.prefill_mx(T, T, 64, 128, 64, rs, re, seed=51)
    t = inputs(p)
    buf = torch.full((T, T + 5), 7.0, device="cuda")          # ld > S, dirty
    api.indexer_logits_mxfp4(*t, logits=buf)
    g = buf.cpu().numpy()[:, :T]
    ref = oracle_logits(p)
    for r in range(T):
        assert_close(g[r, rs[r]:re[r]], ref[r, rs[r]:re[r]], f"row {r}")
    assert (buf.cpu().numpy()[:, T:] == 7.0).all()
    got = api.indexer_topk_mxfp4(*t, p.topk).cpu().numpy()
    assert np.array_equal(got, oracle.topk(g, rs, re, p.topk, S=T))


def test_mxfp4_extreme_block_scales(api):
    # Blocks whose scales span a wide range (one block per row dominates),
    # zero blocks, and negative zeros: the scales must be applied per block.
    p = wl.prefill_mx(200, 200, 64, 128, 16, seed=52)
    rng = np.random.default_rng(53)
    p.q_sf[:] = rng.integers(100, 150, p.q_sf.shape).astype(np.uint8)
    p.k_sf[:] = rng.integers(100, 150, p.k_sf.shape).astype(np.uint8)
    p.q[::7, :, :16] = 0x88                                     # -0 codes in block 0
    p.k[::5, 16:32] = 0                                         # zero block 1
    t = inputs(p)
    g = api.indexer_logits_mxfp4(*t, clean=True).cpu().numpy()
    assert_close(g, oracle_logits(p), "extreme scales")


def test_mxfp4_32768_full_size(api):
    p = wl.prefill_mxfp4()
    t = inputs(p)
    ws = torch.empty(api.workspace_bytes(api.DSA_OP_INDEXER_TOPK, p.T, p.S, p.topk),
                     dtype=torch.uint8, device="cuda")
    got = api.indexer_topk_mxfp4(*t, p.topk, workspace=ws).cpu().numpy()
    ld = (p.S + 3) // 4 * 4
    lg = ws[:p.T * ld * 4].view(torch.float32).view(p.T, ld)[:, :p.S]
    edges = set(range(64)) | set(range(p.T - 64, p.T))
    rng = np.random.default_rng(54)
    rows = np.array(sorted(edges | set(int(x) for x in rng.choice(p.T, 16, replace=False))))
    g = lg[torch.from_numpy(rows).cuda()].cpu().numpy()
    ref = oracle_logits(p, rows)
    for i, r in enumerate(rows):
        assert_close(g[i, :r + 1], ref[i, :r + 1], f"row {r}")
    for r0 in range(0, p.T, 2048):                              # every row's top-k
        chunk = lg[r0:r0 + 2048].cpu().numpy()
        ref_idx = oracle.topk(chunk, p.row_starts[r0:r0 + 2048], p.row_ends[r0:r0 + 2048],
                              p.topk, S=p.S)
        assert np.array_equal(got[r0:r0 + 2048], ref_idx), f"rows {r0}.."
    unfused = api.indexer_logits_mxfp4(*t)
    for r in (0, 777, 20000, p.T - 1):
        assert torch.equal(unfused[r, :r + 1], lg[r, :r + 1])
    assert api.last_device_error() == api.DSA_OK
