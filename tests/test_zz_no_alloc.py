"""dsa_indexer_topk_noalloc, called through the C ABI (needs a GPU).

This entry point serves callers that cannot allocate device memory when they
call the indexer: plugins whose host framework owns every device allocation,
and serving loops that cannot afford cudaMalloc's implicit synchronisation.  It keeps the logits in a
fixed 64 MiB device array of the library instead of a caller workspace.

The test runs it twice in a row on different inputs (so the second call finds
the first call's logits still in the shared array) and compares each result
with dsa_indexer_topk, which takes a caller workspace: the indices must be
identical.  A second case uses the shape where the workspace entry point
splits long rows over many CTAs and the no-alloc one does not.  The file is
named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

from top_selection_dsa_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from top_selection_dsa_gb300 import api as _api
    f = _api.lib.dsa_indexer_topk_noalloc
    P, I = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [P, P, P, P, I, P, P, P, I, I, I, I, I, P, P]
    f.restype = I
    return _api


def _inputs(p):
    cuda = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    q = cuda(p.q.view(np.int16)).view(torch.bfloat16)
    k = cuda(p.k.view(np.int16)).view(torch.bfloat16)
    return q, k, cuda(p.w), cuda(p.row_starts), cuda(p.row_ends)


def _noalloc(api, p, q, k, w, rs, re):
    out = torch.full((p.T, p.topk), -7, dtype=torch.int32, device="cuda")
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = api.lib.dsa_indexer_topk_noalloc(ptr(q), None, ptr(k), None, api.DSA_BF16, ptr(w),
                                          ptr(rs), ptr(re), p.T, p.S, p.H, p.D, p.topk,
                                          ptr(out), stream)
    assert st == api.DSA_OK, api.status_string(st)
    return out


def test_noalloc_matches_workspace_entry_point_on_two_calls(api):
    first = wl.prefill_causal(T=2048, H=64, D=128, topk=512, seed=21)
    lens = [700, 1, 1300]
    rs, re = wl.thd_ranges(lens)
    second = wl.prefill(sum(lens), sum(lens), 64, 128, 300, rs, re, seed=22)
    for p in (first, second):
        q, k, w, rs_d, re_d = _inputs(p)
        got = _noalloc(api, p, q, k, w, rs_d, re_d)
        want = api.indexer_topk(q, k, w, rs_d, re_d, p.topk)
        torch.cuda.synchronize()
        assert torch.equal(got, want)
    assert api.last_device_error() == api.DSA_OK


@pytest.mark.parametrize("T", [24, 256])
def test_noalloc_matches_where_the_workspace_call_splits_rows(api, T):
    # 24 rows of up to 32768 keys: dsa_indexer_topk takes the split top-k
    # (many CTAs per row, scratch in its workspace), the no-alloc call the
    # 256-thread per-row kernel (its array holds only the logits).  256 rows:
    # both take one 1024-thread CTA per row (256 * 32768 * 4 bytes = 32 MiB of
    # logits).  Both must select the same columns, ties and clamped or empty
    # ranges included.
    S = 32768
    rng = np.random.default_rng(23)
    rs = rng.integers(-100, S // 2, T).astype(np.int32)
    re = (rs + rng.integers(0, S + 200, T)).astype(np.int32)   # some past S
    re[:4] = rs[:4]                                            # empty rows
    rs[4:8], re[4:8] = -5, S + 9                               # whole, clamped
    p = wl.prefill(T, S, 64, 128, 2048, rs, re, seed=24)
    p.k[:] = p.k[np.arange(S) % 97]       # repeated key rows: exact ties
    q, k, w, rs_d, re_d = _inputs(p)
    for _ in range(2):
        got = _noalloc(api, p, q, k, w, rs_d, re_d)
        want = api.indexer_topk(q, k, w, rs_d, re_d, p.topk)
        torch.cuda.synchronize()
        assert torch.equal(got, want)
    assert (got[:4] == -1).all()
    assert api.last_device_error() == api.DSA_OK


def test_noalloc_rejects_requests_larger_than_its_array(api):
    fake = ctypes.c_void_p(0x10000)   # never dereferenced: rejected on the host
    T, S = 8192, 4096                 # 8192 * 4096 * 4 bytes = 128 MiB > 64 MiB
    st = api.lib.dsa_indexer_topk_noalloc(fake, None, fake, None, api.DSA_BF16, fake, fake,
                                          fake, T, S, 64, 128, 2048, fake, None)
    assert st == api.DSA_ERR_UNSUPPORTED
