"""The rank merge and the decode-context-parallel top-k on one GPU.

dsa_topk_merge is checked against oracle.topk_merge on candidate sets with
ties, empty slots and invalid scores.  The W-rank protocol is emulated on one
device (each rank's keys are its interleaved share of the row): local top-k
with the library's top-k, global columns, concatenation as the exchange would
produce it, merge -- which must equal the oracle's top-k of the whole row.
"""
import numpy as np
import pytest
import torch

import oracle
from top_selection_dsa_gb300 import dcp

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from top_selection_dsa_gb300 import api as _api
    return _api


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


@pytest.mark.parametrize("C,k", [(1, 1), (16, 8), (300, 256), (4096, 2048), (16384, 2048),
                                 (16384, 16384)])
def test_merge_matches_oracle(api, C, k):
    rng = np.random.default_rng(C + k)
    T = 5
    sc = np.round(rng.standard_normal((T, C)), 1).astype(np.float32)    # many ties
    cols = np.stack([rng.permutation(4 * C)[:C] for _ in range(T)]).astype(np.int32)
    cols[0, ::5] = -1                                                   # empty slots
    sc[1, ::7] = -np.inf
    sc[2, ::11] = np.nan
    sc[3, : C // 2] = -0.0
    got = api.topk_merge(dev(sc), dev(cols), k).cpu().numpy()
    assert np.array_equal(got, oracle.topk_merge(sc, cols, k))


@pytest.mark.parametrize("world,inter", [(2, 1), (4, 64), (8, 64), (3, 5)])
def test_emulated_ranks_give_the_global_topk(api, world, inter):
    # Each rank: one dsa_topk_dcp_candidates call on its share of the row;
    # the exchange's [W, T, k] layout; one dsa_topk_merge_ranks call.
    rng = np.random.default_rng(world * 100 + inter)
    T, S, k = 16, 40000, 2048
    lg = np.round(rng.standard_normal((T, S)) * 4, 0).astype(np.float32)   # heavy ties
    L = np.exp(rng.uniform(np.log(3000), np.log(S), T)).astype(np.int32)
    L[0] = 100                                                          # fewer than k keys
    L[1] = 0                                                            # empty
    cand_s, cand_c = [], []
    for r in range(world):
        pos = dcp.owned_positions(S, r, world, inter).numpy()
        loc = lg[:, pos]
        ln = np.array([dcp.local_len(int(x), r, world, inter) for x in L], np.int32)
        s_r, c_r = dcp.local_candidates(dev(loc), dev(ln), k, r, world, inter)
        # The pairs: the oracle's local top-k, its scores, its global positions.
        top = oracle.topk(loc, np.zeros(T, np.int32), ln, k)
        want_c = np.where(top >= 0, pos[np.maximum(top, 0)], -1)
        want_s = np.where(top >= 0, np.take_along_axis(loc, np.maximum(top, 0), 1), -np.inf)
        assert np.array_equal(c_r.cpu().numpy(), want_c)
        assert np.array_equal(s_r.cpu().numpy(), want_s.astype(np.float32))
        cand_s.append(s_r)
        cand_c.append(c_r)
    all_s, all_c = torch.stack(cand_s), torch.stack(cand_c)            # [W, T, k]
    merged = api.topk_merge_ranks(all_s, all_c, k).cpu().numpy()
    assert np.array_equal(merged, oracle.topk(lg, np.zeros(T, np.int32), L, k))
    assert api.last_device_error() == api.DSA_OK


@pytest.mark.parametrize("W,kr,k", [(1, 300, 256), (4, 512, 2048), (8, 2048, 2048), (3, 7, 16)])
def test_merge_ranks_matches_oracle(api, W, kr, k):
    # [W, T, kr] candidates equal dsa_topk_merge of the same candidates as
    # [T, W * kr] rows (the oracle's merge).
    rng = np.random.default_rng(W * kr + k)
    T = 6
    sc = np.round(rng.standard_normal((W, T, kr)), 1).astype(np.float32)
    cols = np.stack([rng.permutation(4 * W * kr)[:W * kr] for _ in range(T)]).astype(np.int32)
    cols = cols.reshape(T, W, kr).transpose(1, 0, 2).copy()
    cols[0, 0, ::3] = -1                                                 # empty slots
    sc[W - 1, 1, ::5] = -np.inf
    sc[0, 2, ::4] = np.nan
    flat_s = sc.transpose(1, 0, 2).reshape(T, W * kr)
    flat_c = cols.transpose(1, 0, 2).reshape(T, W * kr)
    got = api.topk_merge_ranks(dev(sc), dev(cols), k).cpu().numpy()
    assert np.array_equal(got, oracle.topk_merge(flat_s, flat_c, k))


def test_dcp_candidates_large_positions(api):
    # Local column j of rank r maps to ((j / i) * W + r) * i + j % i; a
    # position past INT32_MAX is refused before any launch.
    T, S, k = 2, 5000, 64
    lg = dev(np.random.default_rng(5).standard_normal((T, S)).astype(np.float32))
    z = torch.zeros(T, dtype=torch.int32, device="cuda")
    e = torch.full((T,), S, dtype=torch.int32, device="cuda")
    s_, c_ = api.topk_dcp_candidates(lg, z, e, k, 3, 4, 1000)
    top = api.topk(lg, z, e, k).cpu().numpy().astype(np.int64)
    want = ((top // 1000) * 4 + 3) * 1000 + top % 1000
    assert np.array_equal(c_.cpu().numpy(), want)
    with pytest.raises(api.DSAError):
        api.topk_dcp_candidates(lg, z, e, k, 0, 1 << 20, 1 << 10)
