"""dsa_indexer_topk_host: host inputs, chunked upload / compute / download.

The indices must equal those of the device entry point dsa_indexer_topk bit
for bit (both pick the unique masked top-k under the lower-index tie rule),
and, on a small case, the oracle's top-k of the GPU's own logits.
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
        pytest.skip("no CUDA device")
    from top_selection_dsa_gb300 import api as _api
    return _api


def host(x, pin=True):
    t = torch.from_numpy(np.ascontiguousarray(x))
    return t.pin_memory() if pin else t


def host_qk(p, pin=True):
    if p.dtype == wl.BF16:
        return (host(p.q.view(np.int16), pin).view(torch.bfloat16),
                host(p.k.view(np.int16), pin).view(torch.bfloat16))
    return host(p.q, pin).view(torch.float8_e4m3fn), host(p.k, pin).view(torch.float8_e4m3fn)


def run_host(api, p, pin=True):
    q, k = host_qk(p, pin)
    ks = host(p.k_scale, pin) if p.k_scale is not None else None
    return api.indexer_topk_host(q, k, host(p.w, pin), host(p.row_starts, pin),
                                 host(p.row_ends, pin), p.topk, k_scale=ks)


def run_device(api, p):
    q, k = (t.cuda() for t in host_qk(p, False))
    ks = torch.from_numpy(p.k_scale).cuda() if p.k_scale is not None else None
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    out = api.indexer_topk(q, k, d(p.w), d(p.row_starts), d(p.row_ends), p.topk, k_scale=ks)
    torch.cuda.synchronize()
    return out.cpu()


def test_small_case_matches_oracle_topk_of_gpu_logits(api):
    # T = 700: two chunks (384 + 316 rows)
    p = wl.prefill(700, 700, 8, 64, 64, seed=3, name="host_small")
    got = run_host(api, p)
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    q, k = (t.cuda() for t in host_qk(p, False))
    lg = api.indexer_logits(q, k, d(p.w), d(p.row_starts), d(p.row_ends), clean=True)
    want = oracle.topk(lg.cpu().numpy(), p.row_starts, p.row_ends, p.topk)
    assert np.array_equal(got.numpy(), want)


# 4096 and 1000 rows: chunks of whole multiples of 64 rows; 8192 rows at 64
# heads: chunks of whole scoring rounds (4 rows x the SM count) after a
# shorter first chunk.
@pytest.mark.parametrize("T", [4096, 1000, 8192])
def test_causal_bf16_equals_device_entry_point(api, T):
    p = wl.prefill_causal(T=T, H=64, D=128, topk=2048, seed=1)
    assert torch.equal(run_host(api, p), run_device(api, p))


def test_e4m3_with_key_scales_equals_device_entry_point(api):
    p = wl.prefill(1536, 1536, 64, 128, 512, seed=2, dtype=wl.E4M3, name="host_e4m3")
    assert torch.equal(run_host(api, p), run_device(api, p))


def test_chunks_of_few_long_rows(api):
    # 4700 rows of up to 40000 keys in chunks of at most 512 rows, which the
    # top-k takes with one 1024-thread CTA per row, but for a 28-row chunk
    # that takes the split top-k; the device entry point runs all 4700 rows
    # on 256-thread CTAs.
    T, S = 4700, 40000
    rng = np.random.default_rng(7)
    ends = rng.integers(1, S + 1, size=T).astype(np.int32)
    starts = (ends * rng.uniform(0, 0.3, size=T)).astype(np.int32)
    p = wl.prefill(T, S, 8, 64, 2048, starts, ends, seed=4, name="host_split_tail")
    assert torch.equal(run_host(api, p), run_device(api, p))


def test_query_scales_go_up_too(api):
    p = wl.prefill(900, 900, 16, 128, 64, seed=8, name="host_qscale")
    qs = np.random.default_rng(8).uniform(0.5, 2.0, size=(900, 16)).astype(np.float32)
    q, k = host_qk(p)
    got = api.indexer_topk_host(q, k, host(p.w), host(p.row_starts), host(p.row_ends), p.topk,
                                q_scale=host(qs))
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    want = api.indexer_topk(q.cuda(), k.cuda(), d(p.w), d(p.row_starts), d(p.row_ends), p.topk,
                            q_scale=d(qs))
    torch.cuda.synchronize()
    assert torch.equal(got, want.cpu())


def test_pageable_host_memory(api):
    p = wl.prefill(640, 640, 16, 128, 128, seed=5, name="host_pageable")
    assert torch.equal(run_host(api, p, pin=False), run_device(api, p))


def test_no_rows(api):
    p = wl.prefill(0, 64, 8, 64, 16, np.zeros(0, np.int32), np.zeros(0, np.int32), seed=6,
                   name="host_empty")
    out = run_host(api, p)
    assert out.shape == (0, 16)
