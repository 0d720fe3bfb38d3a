"""The composed entry points captured in a CUDA graph and replayed.

Shapes are fixed at capture (rows, key capacity, k); row ranges and context
lengths are device data, so one graph serves every step of a decode loop.
Each replay must give exactly what an eager call gives on the same inputs
(both are checked against the oracle elsewhere).  The library's per-device
lookups run on the first call, so every test calls once before capturing.
"""
import numpy as np
import pytest
import torch

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


def capture(fn):
    """fn() once on a side stream (warm-up), then captured into a graph."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def test_paged_decode_graph_replays_with_new_context_lengths(api):
    # 16 rows with contexts above 16384 keys: the split top-k (a memset and
    # three dependent launches) runs inside the graph.
    p = wl.paged_decode(B=8, next_n=2, ctx_lo=17000, ctx_hi=40000, topk=512, seed=11)
    q = dev(p.q.view(np.int16)).view(torch.bfloat16)
    kc = dev(p.k_cache.view(np.int16)).view(torch.bfloat16)
    w, bt, cl = dev(p.w), dev(p.block_table), dev(p.context_lens)
    R, max_ctx = p.R, p.max_ctx()
    ws = torch.empty(api.workspace_bytes(api.DSA_OP_INDEXER_TOPK_PAGED, R, max_ctx, p.topk),
                     dtype=torch.uint8, device="cuda")
    out = torch.empty((R, p.topk), dtype=torch.int32, device="cuda")

    def step():
        api.indexer_topk_paged(q, w, kc, bt, cl, p.topk, next_n=p.next_n, out=out, workspace=ws)

    ref1 = api.indexer_topk_paged(q, w, kc, bt, cl, p.topk, next_n=p.next_n).clone()
    g = capture(step)
    out.fill_(-7)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref1)
    # Shorter contexts (their blocks are in the table): same graph, new data.
    lens2 = np.maximum(p.context_lens // 3, p.next_n).astype(np.int32)
    lens2[0] = p.next_n                                  # a row of a single key
    cl.copy_(dev(lens2))
    out.fill_(-7)
    g.replay()
    torch.cuda.synchronize()
    ref2 = api.indexer_topk_paged(q, w, kc, bt, dev(lens2), p.topk, next_n=p.next_n)
    assert torch.equal(out, ref2)
    assert not torch.equal(ref1, ref2)
    assert api.last_device_error() == api.DSA_OK


def test_prefill_graph_replays_with_new_row_ranges(api):
    rng = np.random.default_rng(9)
    a0 = rng.integers(0, 1500, size=512).astype(np.int32)
    b0 = np.minimum(a0 + rng.integers(0, 1200, size=512), 1500).astype(np.int32)
    p = wl.prefill(T=512, S=1500, H=64, D=128, topk=300, row_starts=a0, row_ends=b0, seed=4)
    q = dev(p.q.view(np.int16)).view(torch.bfloat16)
    k = dev(p.k.view(np.int16)).view(torch.bfloat16)
    w, rs, re = dev(p.w), dev(p.row_starts), dev(p.row_ends)
    ws = torch.empty(api.workspace_bytes(api.DSA_OP_INDEXER_TOPK, p.T, p.S, p.topk),
                     dtype=torch.uint8, device="cuda")
    out = torch.empty((p.T, p.topk), dtype=torch.int32, device="cuda")

    def step():
        api.indexer_topk(q, k, w, rs, re, p.topk, out=out, workspace=ws)

    ref1 = api.indexer_topk(q, k, w, rs, re, p.topk).clone()
    g = capture(step)
    out.fill_(-7)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref1)
    a = rng.integers(0, p.S, size=p.T).astype(np.int32)
    b = np.minimum(a + rng.integers(0, 900, size=p.T), p.S).astype(np.int32)
    rs.copy_(dev(a))
    re.copy_(dev(b))
    out.fill_(-7)
    g.replay()
    torch.cuda.synchronize()
    ref2 = api.indexer_topk(q, k, w, dev(a), dev(b), p.topk)
    assert torch.equal(out, ref2)
    assert api.last_device_error() == api.DSA_OK
