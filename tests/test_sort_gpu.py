"""dsa_topk_sort_by_score against the oracle's score order (GPU).

The scores the sort reads are the GPU's own logits, and the expected order is
oracle.sort_by_score on those same fp32 values: equal scores must come out in
ascending column order, so the comparison is exact.
"""
import numpy as np
import pytest
import torch

import oracle
from top_selection_dsa_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from top_selection_dsa_gb300 import api as _api
    return _api


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def test_sort_after_prefill_topk(api):
    p = wl.tiny_causal()
    q = dev(p.q.view(np.int16)).view(torch.bfloat16)
    k = dev(p.k.view(np.int16)).view(torch.bfloat16)
    w, rs, re = dev(p.w), dev(p.row_starts), dev(p.row_ends)
    lg = api.indexer_logits(q, k, w, rs, re, clean=True)
    top = api.topk(lg, rs, re, p.topk)
    want = oracle.sort_by_score(lg.cpu().numpy(), top.cpu().numpy())
    got = api.topk_sort_by_score(lg, top.clone())
    assert np.array_equal(got.cpu().numpy(), want)
    assert api.last_device_error() == api.DSA_OK


@pytest.mark.parametrize("S,k", [(1, 1), (50, 64), (3000, 2048), (9000, 4096), (12000, 8192)])
def test_sort_ties_padding_and_sizes(api, S, k):
    rng = np.random.default_rng(S + k)
    T = 6
    lg = np.round(rng.standard_normal((T, S)), 1).astype(np.float32)   # many equal scores
    lg[0, : S // 2] = 0.0
    lg[0, S // 2:] = -0.0                                              # -0.0 equals +0.0
    lg[1, ::3] = -np.inf
    rs = np.zeros(T, np.int32)
    re = np.array([S, S, S // 2, 0, S, max(S - 7, 0)], np.int32)       # short and empty rows
    top = oracle.topk(lg, rs, re, k)
    got = api.topk_sort_by_score(dev(lg), dev(top))
    assert np.array_equal(got.cpu().numpy(), oracle.sort_by_score(lg, top))


def test_sort_reads_paged_logits_from_the_workspace(api):
    p = wl.paged_decode(B=4, next_n=2, ctx_lo=3000, ctx_hi=20000, topk=300, seed=7)
    q = dev(p.q.view(np.int16)).view(torch.bfloat16)
    kc = dev(p.k_cache.view(np.int16)).view(torch.bfloat16)
    w, bt, cl = dev(p.w), dev(p.block_table), dev(p.context_lens)
    max_ctx = p.max_ctx()
    ws = torch.empty(api.workspace_bytes(api.DSA_OP_INDEXER_TOPK_PAGED, p.R, max_ctx, p.topk),
                     dtype=torch.uint8, device="cuda")
    top = api.indexer_topk_paged(q, w, kc, bt, cl, p.topk, next_n=p.next_n, workspace=ws)
    ld = (max_ctx + 3) // 4 * 4
    lg = ws[:p.R * ld * 4].view(torch.float32).view(p.R, ld)          # the composed call's logits
    want = oracle.sort_by_score(lg.cpu().numpy(), top.cpu().numpy())
    assert np.array_equal(api.topk_sort_by_score(lg, top.clone()).cpu().numpy(), want)


def test_sort_index_past_the_row_is_padding_and_reported(api):
    lg = dev(np.arange(40, dtype=np.float32).reshape(2, 20))
    top = dev(np.array([[3, 7, 25, -1], [0, 19, 1, 2]], np.int32))
    got = api.topk_sort_by_score(lg, top).cpu().numpy()
    assert got.tolist() == [[7, 3, -1, -1], [19, 2, 1, 0]]
    assert api.last_device_error() == api.DSA_ERR_INVALID_ARG
    assert api.last_device_error() == api.DSA_OK
