"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Two bars, fixed for the lightning-indexer path:
  * logits: |gpu - oracle| <= 1e-3 + 2e-2 * |oracle| for every finite oracle
    value, and -inf exactly where the oracle has -inf;
  * top-k: bit-exact with the oracle's top-k run on the GPU's own logits.
Full-size workloads compare sampled rows (the oracle computes them one by
one) and check the top-k of every row the oracle can afford.
"""
import math

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
    t = torch.from_numpy(np.ascontiguousarray(x))
    return t.cuda()


def qk_tensors(p):
    if p.dtype == wl.BF16:
        return dev(p.q.view(np.int16)).view(torch.bfloat16), dev(p.k.view(np.int16)).view(torch.bfloat16)
    return dev(p.q).view(torch.float8_e4m3fn), dev(p.k).view(torch.float8_e4m3fn)


def prefill_inputs(p):
    q, k = qk_tensors(p)
    ks = dev(p.k_scale) if p.k_scale is not None else None
    return q, k, dev(p.w), dev(p.row_starts), dev(p.row_ends), ks


def assert_logits_close(gpu, ref, what=""):
    g = np.asarray(gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape
    ninf = np.isneginf(r)
    bad_inf = np.isneginf(g) != ninf
    assert not bad_inf.any(), f"{what}: -inf mismatch at {np.argwhere(bad_inf)[:5].tolist()}"
    fin = ~ninf
    err = np.abs(g[fin] - r[fin])
    bound = ATOL + RTOL * np.abs(r[fin])
    if not (err <= bound).all():
        i = int(np.argmax(err - bound))
        raise AssertionError(f"{what}: logits differ: max excess {float((err - bound)[i]):.3g}, "
                             f"gpu {g[fin][i]!r} oracle {r[fin][i]!r}; "
                             f"{int((err > bound).sum())} of {err.size} outside tolerance")


def oracle_logits(p, rows=None):
    return oracle.logits(p.q, p.k, p.w, p.row_starts, p.row_ends, dtype=p.dtype,
                         k_scale=p.k_scale, rows=rows)


def sample_rows(T, n, seed=0, always=()):
    rng = np.random.default_rng(seed)
    rows = set(int(r) for r in rng.choice(T, size=min(n, T), replace=False))
    rows.update(r for r in always if 0 <= r < T)
    return np.array(sorted(rows), dtype=np.int64)


# ------------------------------------------------------------ failure detection

def test_bounded_wait_reports_timeout(api):
    assert api.last_device_error() == api.DSA_OK
    api.selftest_wait_timeout(2_000_000)          # 2 ms; nothing ever arrives
    assert api.last_device_error() == api.DSA_ERR_TIMEOUT
    assert api.last_device_error() == api.DSA_OK  # the word is cleared
    x = torch.ones(4, device="cuda")              # the context is still usable
    assert float(x.sum()) == 4.0


# ---------------------------------------------------------------- small parity

def test_tiny_causal_logits_and_topk(api):
    p = wl.tiny_causal()
    q, k, w, rs, re, ks = prefill_inputs(p)
    lg = api.indexer_logits(q, k, w, rs, re, clean=True)
    g = lg.cpu().numpy()
    assert_logits_close(g, oracle_logits(p), "tiny")
    ref_idx = oracle.topk(g, p.row_starts, p.row_ends, p.topk)
    got = api.topk(lg, rs, re, p.topk).cpu().numpy()
    assert np.array_equal(got, ref_idx)
    fused = api.indexer_topk(q, k, w, rs, re, p.topk).cpu().numpy()
    assert np.array_equal(fused, ref_idx)
    assert (fused[:p.topk - 1, -1] == -1).all()          # early rows padded


@pytest.mark.parametrize("H,D", [(64, 128), (32, 128), (16, 64), (8, 128), (4, 64), (2, 128),
                                 (1, 64)])
def test_logits_heads_and_dims_ragged(api, H, D):
    T = S = 333   # several key tiles, ragged tail, partial last token group
    p = wl.prefill(T, S, H, D, 16, seed=H + D)
    q, k, w, rs, re, ks = prefill_inputs(p)
    g = api.indexer_logits(q, k, w, rs, re, clean=True).cpu().numpy()
    assert_logits_close(g, oracle_logits(p), f"H={H} D={D}")
    got = api.indexer_topk(q, k, w, rs, re, p.topk).cpu().numpy()
    assert np.array_equal(got, oracle.topk(g, p.row_starts, p.row_ends, p.topk))


def test_logits_non_causal_ranges_and_unclean_buffer(api):
    T, S = 97, 1000
    rng = np.random.default_rng(7)
    rs = rng.integers(-50, S, T).astype(np.int32)
    re = (rs + rng.integers(-20, 700, T)).astype(np.int32)
    p = wl.prefill(T, S, 64, 128, 64, rs, re, seed=8)
    q, k, w, rs_d, re_d, _ = prefill_inputs(p)
    buf = torch.full((T, S + 3), 7.0, device="cuda")            # ld > S
    api.indexer_logits(q, k, w, rs_d, re_d, logits=buf)
    g = buf.cpu().numpy()[:, :S]
    ref = oracle_logits(p)
    for t in range(T):                                           # in-range columns only
        lo, hi = max(rs[t], 0), min(max(re[t], 0), S)
        if hi > lo:
            assert_logits_close(g[t, lo:hi], ref[t, lo:hi], f"row {t}")
    assert (buf.cpu().numpy()[:, S:] == 7.0).all()               # padding columns untouched
    got = api.topk(buf, rs_d, re_d, p.topk, S=S).cpu().numpy()
    assert np.array_equal(got, oracle.topk(buf.cpu().numpy(), rs, re, p.topk, S=S))


def test_thd_small(api):
    lens = [130, 1, 400, 257]
    rs, re = wl.thd_ranges(lens)
    T = sum(lens)
    p = wl.prefill(T, T, 64, 128, 100, rs, re, seed=9)
    q, k, w, rs_d, re_d, _ = prefill_inputs(p)
    g = api.indexer_logits(q, k, w, rs_d, re_d, clean=True).cpu().numpy()
    assert_logits_close(g, oracle_logits(p), "thd")
    got = api.indexer_topk(q, k, w, rs_d, re_d, p.topk).cpu().numpy()
    ref = oracle.topk(g, rs, re, p.topk)
    assert np.array_equal(got, ref)
    sel = got[got >= 0]
    owner = np.repeat(np.arange(len(lens)), lens)
    rows = np.nonzero(got >= 0)[0]
    assert (owner[sel] == owner[rows]).all()                     # indices stay in-sequence


def test_fp8_small(api):
    p = wl.prefill(300, 300, 64, 128, 32, seed=10, dtype=wl.E4M3)
    q, k, w, rs, re, ks = prefill_inputs(p)
    g = api.indexer_logits(q, k, w, rs, re, k_scale=ks, clean=True).cpu().numpy()
    assert_logits_close(g, oracle_logits(p), "fp8")
    got = api.indexer_topk(q, k, w, rs, re, p.topk, k_scale=ks).cpu().numpy()
    assert np.array_equal(got, oracle.topk(g, p.row_starts, p.row_ends, p.topk))


@pytest.mark.parametrize("H", [32, 16, 8, 4, 1])
def test_fp8_head_counts_ragged(api, H):
    # e4m3 instances below 64 heads: registers-held weights (H >= 16) and the
    # scalar head sum (H < 16), several key tiles with a ragged tail
    T = S = 333
    p = wl.prefill(T, S, H, 128, 16, seed=40 + H, dtype=wl.E4M3)
    q, k, w, rs, re, ks = prefill_inputs(p)
    g = api.indexer_logits(q, k, w, rs, re, k_scale=ks, clean=True).cpu().numpy()
    assert_logits_close(g, oracle_logits(p), f"fp8 H={H}")
    got = api.indexer_topk(q, k, w, rs, re, p.topk, k_scale=ks).cpu().numpy()
    assert np.array_equal(got, oracle.topk(g, p.row_starts, p.row_ends, p.topk))


def test_q_scale_argument(api):
    p = wl.prefill(130, 130, 16, 128, 8, seed=11)
    q, k, w, rs, re, _ = prefill_inputs(p)
    sq = np.exp2(np.random.default_rng(12).integers(-2, 3, (130, 16))).astype(np.float32)
    g = api.indexer_logits(q, k, w, rs, re, q_scale=dev(sq), clean=True).cpu().numpy()
    ref = oracle.logits(p.q, p.k, p.w, p.row_starts, p.row_ends, q_scale=sq)
    assert_logits_close(g, ref, "q_scale")


# ---------------------------------------------------------------- top-k alone

def test_topk_edge_cases(api):
    rng = np.random.default_rng(13)
    T, S, k = 12, 5000, 64
    lg = rng.standard_normal((T, S)).astype(np.float32)
    lg[1] = 0.0                                   # all ties
    lg[2, ::2] = -0.0                              # signed-zero ties
    lg[2, 1::2] = 0.0
    lg[3, :] = -np.inf                             # nothing valid
    lg[4, rng.random(S) < 0.5] = np.nan            # NaN never selected
    lg[5] = np.round(lg[5] * 2) / 2                # heavy ties
    lg[6, 100:200] = np.inf
    rs = np.array([0, 0, 0, 0, 0, 0, 0, 10, 4000, 30, -5, 2], np.int32)
    re = np.array([S, S, S, S, S, S, S, 10 + k, 4000 + k - 1, 20, 10 ** 6, 2], np.int32)
    dirty = lg.copy()
    for t in range(T):                             # garbage outside the ranges
        dirty[t, :max(rs[t], 0)] = 1e30
        dirty[t, min(max(re[t], 0), S):] = np.inf
    got = api.topk(dev(dirty), dev(rs), dev(re), k).cpu().numpy()
    ref = oracle.topk(dirty, rs, re, k)
    assert np.array_equal(got, ref)
    assert (got[3] == -1).all() and (got[9] == -1).all() and (got[11] == -1).all()
    assert (got[7] == np.arange(10, 10 + k)).all()


# Rows of several chunks whose threshold bin (top 11 key bits) sits at an
# edge of the value order, where the bin's bounds are compared as floats:
# the +0 bin with -0 and positive subnormals, the bin just below it
# (negative subnormals, with the zeros above it), the +inf bin, the bin of
# -FLT_MAX, and a NaN-heavy row.  Every bin holds more keys than are still
# needed, so each row lists its bin's keys and refines them.  Both row
# kernels: 256 threads (3 chunks of 4096) and 1024 threads (4 of 16384).
@pytest.mark.parametrize("S,T", [(10000, 10), (50000, 40)])
def test_topk_threshold_bin_at_value_edges(api, S, T):
    rng = np.random.default_rng(S + T)
    k = 80
    f = lambda bits: np.array(bits, np.uint32).view(np.float32)
    lg = np.full((T, S), -1.0, np.float32)
    kind = np.arange(T) % 5
    for t in range(T):
        cols = rng.permutation(S)
        big, mid = cols[:30], cols[30:30 + 150]
        if kind[t] == 0:    # bin of +0: zeros of both signs and positive subnormals
            lg[t, big] = 1.0
            lg[t, mid[:50]] = f(rng.integers(1, 0x200000, 50))
            lg[t, mid[50:100:2]] = 0.0
            lg[t, mid[51:100:2]] = -0.0
        elif kind[t] == 1:  # bin below it: negative subnormals under 20 zeros
            lg[t, big] = 1.0
            lg[t, mid[:20]] = -0.0
            lg[t, mid[20:90]] = f(0x80000000 + rng.integers(1, 0x200000, 70))
            lg[t, mid[90:95]] = f(0x80000001)          # -(smallest subnormal)
        elif kind[t] == 2:  # bin of +inf
            lg[t, mid[:100]] = np.inf
        elif kind[t] == 3:  # bin of -FLT_MAX, the rest -inf
            lg[t] = -np.inf
            lg[t, big] = 3.0e38
            lg[t, mid[:90]] = f(0xFF7FFFFF - rng.integers(0, 0x100000, 90))
            lg[t, mid[90:100]] = f(0xFF7FFFFF)
        else:               # NaN everywhere but 150 tied keys and 30 larger ones
            lg[t] = np.nan
            lg[t, big] = 2.0
            lg[t, mid] = 1.5
    rs = np.zeros(T, np.int32)
    re = np.full(T, S, np.int32)
    got = api.topk(dev(lg), dev(rs), dev(re), k).cpu().numpy()
    assert np.array_equal(got, oracle.topk(lg, rs, re, k))


# A row of several chunks goes out from shared memory four columns a store
# when k is a multiple of 4 and the output row is 16-byte aligned, else one
# column a store: k = 6 and 2050, and k = 2048 into an output that starts 4
# bytes past a 16-byte boundary, each with rows shorter than k (padding) and
# a NaN-heavy row.
@pytest.mark.parametrize("k,offset", [(6, 0), (2050, 0), (2048, 1), (2048, 0)])
def test_topk_output_store_widths(api, k, offset):
    rng = np.random.default_rng(k + offset)
    T, S = 40, 10000
    lg = rng.standard_normal((T, S)).astype(np.float32)
    lg[5] = np.round(lg[5] * 2) / 2                       # ties
    lg[6, rng.random(S) < 0.9] = np.nan                   # about 1000 valid keys
    rs = np.zeros(T, np.int32)
    re = np.full(T, S, np.int32)
    re[7], rs[9], re[11] = 3000, 5000, 1500               # 1500 keys: fewer than k
    flat = torch.full((T * k + 4,), 7, dtype=torch.int32, device="cuda")
    out = flat[offset:offset + T * k].view(T, k)
    got = api.topk(dev(lg), dev(rs), dev(re), k, out=out).cpu().numpy()
    assert np.array_equal(got, oracle.topk(lg, rs, re, k))
    assert (flat[:offset] == 7).all() and (flat[offset + T * k:] == 7).all()


# Rows of at most 4096 columns take the persistent short-row kernel, which
# loops over rows (more rows than its CTAs here) and prefetches two rows ahead:
# every edge case on many rows, with ranges and garbage around them.
@pytest.mark.parametrize("S,k", [(4096, 2048), (3000, 64), (4096, 4096), (700, 1)])
def test_topk_short_rows_many(api, S, k):
    rng = np.random.default_rng(S + k)
    T = 1500
    lg = rng.standard_normal((T, S)).astype(np.float32)
    kind = np.arange(T) % 8
    lg[kind == 1] = 0.0                                          # all ties
    lg[kind == 2] = np.round(lg[kind == 2] * 2) / 2              # heavy ties
    lg[kind == 3] = -np.inf                                      # nothing valid
    sub = lg[kind == 4]
    sub[rng.random(sub.shape) < 0.3] = np.nan
    lg[kind == 4] = sub
    lg[kind == 5, ::3] = -0.0                                    # signed zeros
    ends = rng.integers(0, S + 1, size=T)
    starts = (ends * rng.uniform(0, 0.5, size=T)).astype(np.int64)
    rs = starts.astype(np.int32)
    re = ends.astype(np.int32)
    re[kind == 6] = S + 100                                      # clamped to S
    rs[kind == 7] = re[kind == 7]                                # empty
    dirty = lg.copy()
    for t in range(T):
        dirty[t, :max(rs[t], 0)] = 1e30
        dirty[t, min(max(re[t], 0), S):] = np.inf
    got = api.topk(dev(dirty), dev(rs), dev(re), k).cpu().numpy()
    assert np.array_equal(got, oracle.topk(dirty, rs, re, k))


# Row lengths that reach every top-k path: with few rows (7) the per-row
# kernel's one-chunk rows (S <= 4096) and two-chunk rows, then the split path
# (S > 16384); with more than 512 rows the per-row kernel's multi-chunk
# bitmap path (gathered threshold bin, or digit passes when the bin is too
# large, as in the tie-heavy rows) and, past 262144 columns, the streaming
# kernel.
@pytest.mark.parametrize("S,k,T", [(100, 1, 7), (2048, 2048, 7), (2049, 2048, 7),
                                   (4096, 4096, 7), (8000, 2048, 7), (16384, 3000, 7),
                                   (30000, 2048, 7), (60000, 2048, 7), (131072, 2048, 7),
                                   (200000, 5000, 7), (300000, 2048, 7), (40000, 2048, 520),
                                   (270000, 2048, 520)])
def test_topk_row_lengths(api, S, k, T):
    rng = np.random.default_rng(S + k + T)
    lg = (rng.standard_normal((T, S)) * 4).round().astype(np.float32)   # many ties
    lg[6::7] = rng.standard_normal((len(range(6, T, 7)), S)).astype(np.float32)  # few ties
    rs = np.tile(np.array([0, 0, 0, 0, 0, 0, S // 3], np.int32), T // 7 + 1)[:T]
    re = np.tile(np.array([S, S - 1, S // 2, k, k - 1, 1, S], np.int32), T // 7 + 1)[:T]
    got = api.topk(dev(lg), dev(rs), dev(re), k).cpu().numpy()
    assert np.array_equal(got, oracle.topk(lg, rs, re, k))


# Few long rows (some longer than 16384 columns) over rows of every kind:
# empty, one key, exactly one or two 4096-key units, all ties, nothing valid,
# NaN, signed zeros, ranges starting mid-row or clamped.  24 rows take the
# split path (each resident CTA walking several units), 40 rows one
# 1024-thread CTA per row.
@pytest.mark.parametrize("T", [24, 40])
def test_topk_few_long_rows_edge_rows(api, T):
    rng = np.random.default_rng(77 + T)
    S, k = 50000, 2048
    lg = rng.standard_normal((T, S)).astype(np.float32)
    kind = np.arange(T) % 10
    lg[kind == 1] = 0.0                                           # all ties
    lg[kind == 2] = np.round(lg[kind == 2] * 2) / 2               # heavy ties
    lg[kind == 3] = -np.inf                                       # nothing valid
    sub = lg[kind == 4]
    sub[rng.random(sub.shape) < 0.4] = np.nan
    lg[kind == 4] = sub
    lg[kind == 5, ::2] = -0.0                                     # signed zeros
    lg[kind == 5, 1::2] = 0.0
    starts = np.zeros(T, np.int64)
    ends = np.full(T, S, np.int64)
    ends[kind == 6] = 4096                                        # one whole unit
    ends[kind == 7] = 8192 + 1                                    # two units and a key
    starts[kind == 8] = 12345                                     # mid-row start
    ends[kind == 8] = S + 1000                                    # clamped end
    ends[0] = 0                                                   # empty
    starts[10], ends[10] = 777, 778                               # one key
    starts[20], ends[20] = 100, 100 + k                           # exactly k keys
    rs, re = starts.astype(np.int32), ends.astype(np.int32)
    dirty = lg.copy()
    for t in range(T):
        dirty[t, :max(rs[t], 0)] = 1e30
        dirty[t, min(max(re[t], 0), S):] = np.inf
    got = api.topk(dev(dirty), dev(rs), dev(re), k).cpu().numpy()
    assert np.array_equal(got, oracle.topk(dirty, rs, re, k))
    assert (got[0] == -1).all() and got[10, 0] == 777 and (got[10, 1:] == -1).all()
    assert (got[20] == np.arange(100, 100 + k)).all()
    ws = api.workspace_bytes(api.DSA_OP_TOPK, T, S, k)
    assert (ws > 0) == (T < 32)                    # split scratch for the split path only


def test_topk_reads_ranges_written_just_before_on_the_stream(api):
    # dsa_topk's row ranges come out of kernels queued immediately before it
    # on the same stream (with stale zero ranges in the buffers beforehand):
    # the top-k must see the new ranges, not the stale ones.
    rng = np.random.default_rng(31)
    T, S, k = 2048, 6000, 256
    lg = rng.standard_normal((T, S)).astype(np.float32)
    rs = rng.integers(-10, S // 2, T).astype(np.int32)
    re = (rs + rng.integers(0, S // 2 + 20, T)).astype(np.int32)
    lg_d, rs_src, re_src = dev(lg), dev(rs), dev(re)
    ref = oracle.topk(lg, rs, re, k)
    rs_d = torch.zeros(T, dtype=torch.int32, device="cuda")
    re_d = torch.zeros(T, dtype=torch.int32, device="cuda")
    big = torch.ones(1 << 24, device="cuda")
    for _ in range(5):
        rs_d.zero_()
        re_d.zero_()
        big.mul_(1.0)                               # a long kernel ahead of the writers
        torch.add(rs_src, 0, out=rs_d)              # elementwise kernels, the second
        torch.add(re_src, 0, out=re_d)              # queued right before dsa_topk
        got = api.topk(lg_d, rs_d, re_d, k)
        assert np.array_equal(got.cpu().numpy(), ref)


# --------------------------------------------------------------------- paged

@pytest.mark.parametrize("next_n,block_size,H,fp8", [(2, 64, 64, False), (1, 16, 64, False),
                                                     (3, 128, 32, False), (4, 32, 64, False),
                                                     (2, 64, 64, True), (1, 8, 16, True)])
def test_paged_small(api, next_n, block_size, H, fp8):
    ctx = np.array([1, next_n, 129, 500, 1000, 2047, 2048, 2049, 4000], np.int32)
    ctx = np.maximum(ctx, next_n)
    p = wl.paged_decode(next_n=next_n, block_size=block_size, H=H, D=128, topk=256,
                        ctx_hi=4096, seed=next_n * block_size + H, context_lens=ctx,
                        dtype=wl.E4M3 if fp8 else wl.BF16)
    check_paged(api, p, rows=None)


# Paged rows long enough for the few-long-rows top-k (a context above 16384
# keys; 8 to 40 rows: the split path below 32 rows, a 1024-thread CTA per row
# from 32), one to five query tokens a request: empty and one-key rows,
# contexts ending inside a 4096-key unit and inside a block, e4m3 and bf16, 8
# to 64 heads.
@pytest.mark.parametrize("next_n,block_size,H,fp8", [(1, 16, 64, False), (2, 64, 64, True),
                                                     (4, 32, 8, False), (3, 128, 16, True),
                                                     (5, 64, 32, False), (4, 64, 64, True)])
def test_paged_split_topk(api, next_n, block_size, H, fp8):
    ctx = np.array([0, 1, next_n, 4097, 16385, 20003, 33000, 40960], np.int32)
    p = wl.paged_decode(next_n=next_n, block_size=block_size, H=H, D=128, topk=2048,
                        ctx_hi=40960, seed=7 * next_n + H, context_lens=ctx,
                        dtype=wl.E4M3 if fp8 else wl.BF16)
    check_paged(api, p, rows=None)


def paged_tensors(p):
    if p.dtype == wl.BF16:
        q = dev(p.q.view(np.int16)).view(torch.bfloat16)
        kc = dev(p.k_cache.view(np.int16)).view(torch.bfloat16)
    else:
        q = dev(p.q).view(torch.float8_e4m3fn)
        kc = dev(p.k_cache).view(torch.float8_e4m3fn)
    ks = dev(p.k_scale.reshape(-1)) if p.k_scale is not None else None
    return q, dev(p.w), kc, dev(p.block_table), dev(p.context_lens), ks


def check_paged(api, p, rows=None):
    q, w, kc, bt, cl, ks = paged_tensors(p)
    lg = api.indexer_logits_paged(q, w, kc, bt, cl, next_n=p.next_n, k_scale=ks)
    g = lg.cpu().numpy()
    ref = oracle.logits_paged(p.q, p.w, p.k_cache, p.block_table, p.context_lens,
                              next_n=p.next_n, dtype=p.dtype, k_scale=p.k_scale,
                              ld=p.max_ctx(), rows=rows)
    gg = g if rows is None else g[rows]
    rs, re = oracle.paged_row_ranges(p.context_lens, p.next_n)
    rr = np.arange(p.R) if rows is None else rows
    for i, r in enumerate(rr):                     # the visited part of each row
        hi = int(p.context_lens[r // p.next_n])
        assert_logits_close(gg[i, :hi], ref[i, :hi], f"paged row {r}")
    got = api.indexer_topk_paged(q, w, kc, bt, cl, p.topk, next_n=p.next_n, k_scale=ks)
    got = got.cpu().numpy()
    assert np.array_equal(got, oracle.topk(g, rs, re, p.topk))
    assert api.last_device_error() == api.DSA_OK


def test_paged_bad_block_id_is_reported_not_dereferenced(api):
    p = wl.paged_decode(B=2, next_n=1, ctx_lo=200, ctx_hi=300, block_size=64, H=64,
                        topk=16, seed=3)
    bt = p.block_table.copy()
    bt[1, 1] = 10 ** 6                              # past the cache
    q, w, kc, _, cl, _ = paged_tensors(p)
    api.indexer_logits_paged(q, w, kc, dev(bt), cl, next_n=1)
    assert api.last_device_error() == api.DSA_ERR_INVALID_ARG
    assert api.last_device_error() == api.DSA_OK


# -------------------------------------------------------- full-size workloads

def edge_rows(starts, lens, n=64):
    """The first and last n rows of every sequence (packed at the given starts)."""
    rows = set()
    for a, L in zip(starts, lens):
        rows.update(range(a, a + min(n, L)))
        rows.update(range(a + max(L - n, 0), a + L))
    return rows


def check_topk_all_rows(got, lg, p, chunk=2048):
    """The GPU's top-k of every row against the oracle's top-k of the same
    (GPU) logits, brought to the host a row chunk at a time."""
    for r0 in range(0, p.T, chunk):
        r1 = min(p.T, r0 + chunk)
        g = lg[r0:r1].cpu().numpy()
        ref = oracle.topk(g, p.row_starts[r0:r1], p.row_ends[r0:r1], p.topk, S=p.S)
        if not np.array_equal(got[r0:r1], ref):
            bad = np.nonzero((got[r0:r1] != ref).any(axis=1))[0]
            raise AssertionError(f"top-k differs on {bad.size} rows of [{r0}, {r1}), "
                                 f"first row {r0 + int(bad[0])}")


def fused_with_logits(api, p, q, k, w, rs, re, ks=None):
    """dsa_indexer_topk, and the logits it left at the start of its workspace."""
    ws = torch.empty(api.workspace_bytes(api.DSA_OP_INDEXER_TOPK, p.T, p.S, p.topk),
                     dtype=torch.uint8, device="cuda")
    out = api.indexer_topk(q, k, w, rs, re, p.topk, k_scale=ks, workspace=ws)
    ld = (p.S + 3) // 4 * 4
    lg = ws[:p.T * ld * 4].view(torch.float32).view(p.T, ld)[:, :p.S]
    return out.cpu().numpy(), lg


def check_rows_logits(lg, p, rows, what):
    g = lg[torch.from_numpy(rows).cuda()].cpu().numpy()
    ref = oracle_logits(p, rows)
    for i, t in enumerate(rows):                   # the row's own range
        lo, hi = max(int(p.row_starts[t]), 0), min(int(p.row_ends[t]), p.S)
        assert_logits_close(g[i, lo:hi], ref[i, lo:hi], f"{what} row {t}")


def test_prefill_causal_4096_full_size(api):
    p = wl.prefill_causal()
    q, k, w, rs, re, _ = prefill_inputs(p)
    lg = api.indexer_logits(q, k, w, rs, re, clean=True)
    g = lg.cpu().numpy()
    rows = sample_rows(p.T, 24, seed=1, always=edge_rows([0], [p.T]) | {2047, 2048})
    assert_logits_close(g[rows], oracle_logits(p, rows), "prefill 4096")
    ref = oracle.topk(g, p.row_starts, p.row_ends, p.topk)
    fused, flg = fused_with_logits(api, p, q, k, w, rs, re)
    assert np.array_equal(fused, ref)
    cols = torch.arange(p.S, device="cuda")
    mask = (cols[None, :] >= rs[:, None]) & (cols[None, :] < re[:, None])
    assert torch.equal(flg[mask], lg[mask])        # the fused call's logits, bit for bit
    assert np.array_equal(api.topk(lg, rs, re, p.topk).cpu().numpy(), ref)
    assert (ref[2047:] != -1).all() and (ref[:2047, -1] == -1).all()


def test_prefill_thd_full_size(api):
    p = wl.prefill_thd()
    q, k, w, rs, re, _ = prefill_inputs(p)
    fused, lg = fused_with_logits(api, p, q, k, w, rs, re)
    offs = np.cumsum([0] + p.seq_lens)
    rows = sample_rows(p.T, 24, seed=2, always=edge_rows(offs[:-1], p.seq_lens))
    check_rows_logits(lg, p, rows, "thd")
    check_topk_all_rows(fused, lg, p)


def test_paged_decode_full_size(api):
    p = wl.paged_decode()
    check_paged(api, p, rows=None)                 # every row: logits and top-k


def test_prefill_fp8_32768_full_size(api):
    # Every row's top-k (bit-exact against the oracle's top-k of the fused
    # call's own logits); the logits of the first and last 64 rows and a
    # seeded sample (the oracle's fp64 logits take ~0.5 GFLOP per long row).
    p = wl.prefill_fp8()
    q, k, w, rs, re, ks = prefill_inputs(p)
    fused, lg = fused_with_logits(api, p, q, k, w, rs, re, ks)
    rows = sample_rows(p.T, 16, seed=4, always=edge_rows([0], [p.T]) | {2047, 2048})
    check_rows_logits(lg, p, rows, "fp8")
    check_topk_all_rows(fused, lg, p)
    unfused = api.indexer_logits(q, k, w, rs, re, k_scale=ks)
    for t in (0, 1000, 2047, 20000, 32767):          # the unfused call: same logits
        assert torch.equal(unfused[t, :t + 1], lg[t, :t + 1])
