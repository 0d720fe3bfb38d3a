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


@pytest.mark.parametrize("world,inter", [(2, 1), (4, 64), (8, 64)])
def test_emulated_ranks_give_the_global_topk(api, world, inter):
    rng = np.random.default_rng(world * 100 + inter)
    T, S, k = 16, 40000, 2048
    lg = np.round(rng.standard_normal((T, S)) * 4, 0).astype(np.float32)   # heavy ties
    L = np.exp(rng.uniform(np.log(3000), np.log(S), T)).astype(np.int32)
    L[0] = 100                                                          # fewer than k keys
    cand_s, cand_c = [], []
    for r in range(world):
        pos = dcp.owned_positions(S, r, world, inter).numpy()
        loc = dev(lg[:, pos])
        ln = dcp.local_len(dev(L).long(), r, world, inter)
        s_r, c_r = dcp.local_candidates(loc, ln, k, r, world, inter)
        cand_s.append(s_r)
        cand_c.append(c_r)
    merged = api.topk_merge(torch.cat(cand_s, 1), torch.cat(cand_c, 1), k).cpu().numpy()
    assert np.array_equal(merged, oracle.topk(lg, np.zeros(T, np.int32), L, k))
    assert api.last_device_error() == api.DSA_OK
