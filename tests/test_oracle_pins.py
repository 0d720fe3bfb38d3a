"""Pins of the CPU oracle to things other than itself (CPU only).

Each test checks the oracle against what the pages and the mathematics fix:
hand-worked examples (tests/golden, each with its citation), closed forms,
invariants, brute force on tiny inputs and independent library routines
(torch's own bf16/e4m3 decoders, numpy's stable sort).  They are chosen so that
a plausible slip in the oracle -- a dropped ReLU, a weight applied inside the
ReLU, a transposed operand or index, a wrong mask bound, a wrong tie-break,
an off-by-one in the paged addressing -- fails at least one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from top_selection_dsa_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _num(v):
    if isinstance(v, str):
        return {"-inf": -math.inf, "inf": math.inf, "nan": math.nan,
                "-0.0": -0.0}[v]
    return float(v)


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def bf16(x):
    return wl.to_bf16_bits(np.asarray(x, dtype=np.float32))


# ------------------------------------------------------------------ decoders

def test_e4m3_decoder_exhaustive_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(mine[ok], ref[ok])
    assert np.array_equal(np.signbit(mine[ok]), np.signbit(ref[ok]))
    assert np.isnan(mine).sum() == 2          # S.1111.111 only


def test_e4m3_decoder_golden_codes():
    g = _load("e4m3_codes.json")
    for code, val in g["codes"].items():
        got = oracle.e4m3_to_f64([int(code, 16)])[0]
        want = _num(val)
        if math.isnan(want):
            assert math.isnan(got), code
        else:
            assert got == want and math.copysign(1, got) == math.copysign(1, want), code


def test_bf16_decoder_matches_torch():
    rng = np.random.default_rng(1)
    bits = np.concatenate([
        rng.integers(0, 1 << 16, 4096).astype(np.uint16),
        np.array([0x0000, 0x8000, 0x7F80, 0xFF80, 0x0001, 0x7F7F, 0x3F80], np.uint16)])
    mine = oracle.bf16_to_f64(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(mine[ok], ref[ok])


# -------------------------------------------------------------------- logits

def test_logits_hand_example():
    g = _load("logits_hand_example.json")
    got = oracle.logits(bf16(g["q"]), bf16(g["k"]), np.array(g["w"], np.float32),
                        np.array(g["row_starts"], np.int32),
                        np.array(g["row_ends"], np.int32))
    want = np.array([[_num(v) for v in r] for r in g["logits"]])
    assert np.array_equal(got, want)


def test_logits_one_hot_is_kronecker_delta():
    # H=1, w=1, q[t]=e_i(t), k[s]=e_j(s)  =>  logit = [i(t) == j(s)]
    rng = np.random.default_rng(2)
    T, S, D = 9, 13, 16
    it = rng.integers(0, D, T)
    js = rng.integers(0, D, S)
    q = np.zeros((T, 1, D), np.float32)
    q[np.arange(T), 0, it] = 1
    k = np.zeros((S, D), np.float32)
    k[np.arange(S), js] = 1
    rs = np.zeros(T, np.int32)
    re = np.full(T, S, np.int32)
    got = oracle.logits(bf16(q), bf16(k), np.ones((T, 1), np.float32), rs, re)
    assert np.array_equal(got, (it[:, None] == js[None, :]).astype(np.float64))


def test_logits_relu_factor_closed_form():
    # q[t,h,:] = (h+1) e0, k[s,:] = (s-c) e0: all dots share the sign of s-c,
    # so logit[t,s] = max(0, s-c) * sum_h (h+1) w[t,h]  (zero for s <= c).
    T, S, H, D, c = 5, 12, 4, 8, 6
    rng = np.random.default_rng(3)
    q = np.zeros((T, H, D), np.float32)
    q[:, :, 0] = np.arange(1, H + 1)[None, :]
    k = np.zeros((S, D), np.float32)
    k[:, 0] = np.arange(S) - c
    w = rng.integers(-8, 9, (T, H)).astype(np.float32) / 4
    got = oracle.logits(bf16(q), bf16(k), w, np.zeros(T, np.int32), np.full(T, S, np.int32))
    W = (w.astype(np.float64) * np.arange(1, H + 1)).sum(1)
    want = np.maximum(0, np.arange(S) - c)[None, :] * W[:, None]
    assert np.array_equal(got, want)


def test_logits_alternating_heads_closed_form():
    # q[t,h,:] = (-1)^h e0, k[s,:] = b_s e0: the ReLU keeps the even heads when
    # b_s > 0 and the odd heads when b_s < 0, so
    # logit = |b_s| * sum_{h even} w  or  |b_s| * sum_{h odd} w.
    T, S, H, D = 3, 6, 6, 4
    q = np.zeros((T, H, D), np.float32)
    q[:, :, 0] = np.array([(-1) ** h for h in range(H)])[None, :]
    b = np.array([2, -3, 0.5, -1, 0, 4], np.float32)
    k = np.zeros((S, D), np.float32)
    k[:, 0] = b
    w = np.array([[1, 2, 3, 4, 5, 6], [-1, 0, 2, 0, -3, 1], [0.5, -0.5, 1, -1, 2, -2]],
                 np.float32)
    got = oracle.logits(bf16(q), bf16(k), w, np.zeros(T, np.int32), np.full(T, S, np.int32))
    even = w[:, 0::2].astype(np.float64).sum(1)
    odd = w[:, 1::2].astype(np.float64).sum(1)
    want = np.where(b[None, :] > 0, b[None, :] * even[:, None],
                    np.abs(b)[None, :] * odd[:, None])
    assert np.array_equal(got, want)


def test_logits_negative_weights_give_nonpositive_scores():
    # w < 0 multiplies a ReLU output, so every logit is <= 0 (applying the
    # weight inside the ReLU would make them >= 0 instead).
    p = wl.prefill(16, 16, 4, 64, 4, seed=4)
    w = -np.abs(p.w)
    got = oracle.logits(p.q, p.k, w, p.row_starts, p.row_ends)
    fin = np.isfinite(got)
    assert fin.sum() == p.valid_pairs()
    assert (got[fin] <= 0).all() and (got[fin] < 0).any()


def test_logits_all_negative_dots_are_exact_zero():
    T, S, H, D = 4, 5, 3, 8
    q = np.abs(np.random.default_rng(5).standard_normal((T, H, D))).astype(np.float32)
    k = -np.abs(np.random.default_rng(6).standard_normal((S, D))).astype(np.float32)
    w = np.random.default_rng(7).standard_normal((T, H)).astype(np.float32)
    got = oracle.logits(bf16(q), bf16(k), w, np.zeros(T, np.int32), np.full(T, S, np.int32))
    assert np.array_equal(got, np.zeros((T, S)))


def test_logits_masking_and_clamping():
    T, S = 6, 10
    p = wl.prefill(T, S, 2, 64, 4, np.zeros(T, np.int32), np.full(T, S, np.int32), seed=8)
    rs = np.array([0, 3, -4, 7, 5, 2], np.int32)
    re = np.array([10, 5, 2, 30, 5, 1], np.int32)
    full = oracle.logits(p.q, p.k, p.w, np.zeros(T, np.int32), np.full(T, S, np.int32))
    got = oracle.logits(p.q, p.k, p.w, rs, re)
    for t in range(T):
        lo, hi = max(rs[t], 0), min(re[t], S)
        for s in range(S):
            if lo <= s < hi:
                assert got[t, s] == full[t, s]
            else:
                assert got[t, s] == -math.inf
    assert np.isneginf(got[4]).all() and np.isneginf(got[5]).all()


def test_logits_linear_in_weights():
    p = wl.prefill(12, 12, 8, 64, 4, seed=9)
    w2 = np.random.default_rng(10).standard_normal(p.w.shape).astype(np.float32)
    a = oracle.logits(p.q, p.k, p.w, p.row_starts, p.row_ends)
    b = oracle.logits(p.q, p.k, w2, p.row_starts, p.row_ends)
    c = oracle.logits(p.q, p.k, p.w.astype(np.float64) + w2, p.row_starts, p.row_ends)
    fin = np.isfinite(a)
    # w1 + w2 is rounded to fp32 by the call; compare within that rounding.
    assert np.allclose(c[fin], (a + b)[fin], rtol=1e-6, atol=1e-9)


def test_logits_positive_homogeneity_in_keys():
    p = wl.prefill(8, 8, 4, 64, 4, seed=11)
    k2 = wl.to_bf16_bits(2 * wl.bf16_bits_to_f32(p.k))      # exact in bf16
    a = oracle.logits(p.q, p.k, p.w, p.row_starts, p.row_ends)
    b = oracle.logits(p.q, k2, p.w, p.row_starts, p.row_ends)
    fin = np.isfinite(a)
    assert np.array_equal(b[fin], 2 * a[fin])


def test_logits_e4m3_equals_bf16_of_the_same_values():
    # Every e4m3 value is exact in bf16; torch converts codes -> bf16
    # independently of the oracle's decoder.  The block scales enter as the
    # k_scale/q_scale arguments on both sides.
    p = wl.prefill(10, 10, 4, 128, 4, seed=12, dtype=wl.E4M3)
    qb = torch.from_numpy(p.q).view(torch.float8_e4m3fn).to(torch.bfloat16)
    kb = torch.from_numpy(p.k).view(torch.float8_e4m3fn).to(torch.bfloat16)
    qb = qb.view(torch.int16).numpy().view(np.uint16)
    kb = kb.view(torch.int16).numpy().view(np.uint16)
    sq = np.exp2(np.random.default_rng(13).integers(-3, 3, (10, 4))).astype(np.float32)
    a = oracle.logits(p.q, p.k, p.w, p.row_starts, p.row_ends, dtype=oracle.E4M3,
                      q_scale=sq, k_scale=p.k_scale)
    b = oracle.logits(qb, kb, p.w, p.row_starts, p.row_ends, dtype=oracle.BF16,
                      q_scale=sq, k_scale=p.k_scale)
    assert np.array_equal(a, b)


def test_logits_scale_commutes_with_relu():
    # relu(s*x) = s*relu(x) for s > 0: a power-of-two key scale multiplies
    # the logit exactly.
    p = wl.prefill(8, 8, 4, 128, 4, seed=14, dtype=wl.E4M3)
    one = np.ones_like(p.k_scale)
    a = oracle.logits(p.q, p.k, p.w, p.row_starts, p.row_ends, dtype=oracle.E4M3,
                      k_scale=one)
    b = oracle.logits(p.q, p.k, p.w, p.row_starts, p.row_ends, dtype=oracle.E4M3,
                      k_scale=p.k_scale)
    fin = np.isfinite(a)
    sk = np.broadcast_to(p.k_scale[None, :].astype(np.float64), a.shape)
    assert np.array_equal(b[fin], a[fin] * sk[fin])


# --------------------------------------------------------------------- paged

def test_paged_hand_example():
    g = _load("paged_hand_example.json")
    kc = bf16(g["k_cache"])
    got = oracle.logits_paged(bf16(g["q"]), np.array(g["w"], np.float32), kc,
                              np.array(g["block_table"], np.int32),
                              np.array(g["context_lens"], np.int32),
                              next_n=g["next_n"], ld=3)
    want = np.array([[_num(v) for v in r] for r in g["logits"]])
    assert np.array_equal(got, want)
    rs, re = oracle.paged_row_ranges(np.array(g["context_lens"], np.int32), g["next_n"])
    assert rs.tolist() == g["row_starts"] and re.tolist() == g["row_ends"]
    for kk, exp in g["topk"].items():
        assert oracle.topk(got.astype(np.float32), rs, re, int(kk)).tolist() == exp


def test_paged_row_ranges_closed_form():
    rs, re = oracle.paged_row_ranges(np.array([5, 1, 100], np.int32), 3)
    assert rs.tolist() == [0] * 9
    assert re.tolist() == [3, 4, 5, 0, 0, 1, 98, 99, 100]


def test_paged_equals_contiguous_on_gathered_keys():
    p = wl.paged_decode(B=3, next_n=2, ctx_lo=40, ctx_hi=300, block_size=16,
                        H=4, D=64, topk=8, seed=15)
    ld = p.max_ctx()
    got = oracle.logits_paged(p.q, p.w, p.k_cache, p.block_table, p.context_lens,
                              next_n=2, ld=ld)
    rs, re = oracle.paged_row_ranges(p.context_lens, 2)
    for b in range(p.B):
        L = int(p.context_lens[b])
        pos = np.arange(L)
        kg = p.k_cache[p.block_table[b, pos // 16], pos % 16]     # [L, D]
        rows = slice(2 * b, 2 * b + 2)
        ref = oracle.logits(p.q[rows], kg, p.w[rows], rs[rows], re[rows])
        assert np.array_equal(got[rows, :L], ref)
        assert np.isneginf(got[rows, L:]).all()


def test_paged_identity_table_equals_contiguous_causal_tail():
    # One request, identity block table: the next_n rows are the last next_n
    # rows of a causal prefill over the same keys.
    L, n, bs = 50, 3, 8
    p = wl.prefill(L, L, 2, 64, 4, seed=16)
    nb = -(-L // bs)
    kc = np.zeros((nb * bs, 64), np.uint16)
    kc[:L] = p.k
    got = oracle.logits_paged(p.q[L - n:], p.w[L - n:], kc.reshape(nb, bs, 64),
                              np.arange(nb, dtype=np.int32)[None, :],
                              np.array([L], np.int32), next_n=n, ld=L)
    ref = oracle.logits(p.q, p.k, p.w, p.row_starts, p.row_ends)[L - n:]
    assert np.array_equal(got, ref)


# --------------------------------------------------------------------- top-k

def test_topk_hand_examples():
    g = _load("topk_semantics.json")
    for c in g["cases"]:
        row = np.array([[_num(v) for v in c["logits"]]], np.float32)
        got = oracle.topk(row, np.array([c["row_start"]], np.int32),
                          np.array([c["row_end"]], np.int32), c["k"])
        assert got[0].tolist() == c["expect"], c["why"]
    h = _load("logits_hand_example.json")
    lg = np.array([[_num(v) for v in r] for r in h["logits"]], np.float32)
    for kk, exp in h["topk"].items():
        got = oracle.topk(lg, np.array(h["row_starts"], np.int32),
                          np.array(h["row_ends"], np.int32), int(kk))
        assert got.tolist() == exp


def _brute_force_topk(row, lo, hi, k):
    """Enumerate every subset of the valid columns: keep the one whose values,
    sorted high to low, are largest, and among equal value lists the one whose
    columns, sorted, are smallest."""
    valid = [c for c in range(lo, hi) if not (math.isnan(row[c]) or row[c] == -math.inf)]
    m = min(k, len(valid))
    best = None
    for sub in itertools.combinations(valid, m):
        vals = sorted((float(row[c]) for c in sub), reverse=True)
        key = (vals, [-c for c in sorted(sub)])
        if best is None or key > best[0]:
            best = (key, sorted(sub))
    return best[1] + [-1] * (k - m)


def test_topk_brute_force_on_tie_heavy_rows():
    rng = np.random.default_rng(17)
    pool = np.array([-1.0, 0.0, -0.0, 1.0, 2.0, np.inf, -np.inf, np.nan, 0.5], np.float32)
    for trial in range(300):
        n = int(rng.integers(1, 10))
        row = pool[rng.integers(0, len(pool), n)]
        lo = int(rng.integers(-2, n))
        hi = int(rng.integers(lo, n + 3))
        k = int(rng.integers(1, n + 3))
        got = oracle.topk(row[None, :], np.array([lo], np.int32),
                          np.array([hi], np.int32), k)[0].tolist()
        want = _brute_force_topk(row, max(lo, 0), min(hi, n), k)
        assert got == want, (row, lo, hi, k)


def test_topk_matches_numpy_stable_sort():
    rng = np.random.default_rng(18)
    T, S = 40, 300
    lg = rng.integers(-20, 20, (T, S)).astype(np.float32) / 4   # many ties
    rs = rng.integers(0, S, T).astype(np.int32)
    re = (rs + rng.integers(0, S, T)).astype(np.int32)
    for k in (1, 7, 64, 299):
        got = oracle.topk(lg, rs, re, k)
        for t in range(T):
            lo, hi = rs[t], min(re[t], S)
            cols = np.arange(lo, hi)
            order = np.argsort(-lg[t, lo:hi], kind="stable")   # desc, ties by column
            pick = np.sort(cols[order[:k]])
            want = np.full(k, -1, np.int32)
            want[:len(pick)] = pick
            assert np.array_equal(got[t], want)


def test_topk_invariants_random():
    rng = np.random.default_rng(19)
    T, S, k = 64, 500, 50
    lg = rng.standard_normal((T, S)).astype(np.float32)
    lg[rng.random((T, S)) < 0.05] = -np.inf
    rs = rng.integers(-10, S, T).astype(np.int32)
    re = (rs + rng.integers(-5, 120, T)).astype(np.int32)
    out = oracle.topk(lg, rs, re, k)
    for t in range(T):
        lo, hi = max(rs[t], 0), min(max(re[t], 0), S)
        valid = [c for c in range(lo, hi) if np.isfinite(lg[t, c]) or lg[t, c] == np.inf]
        sel = [c for c in out[t] if c != -1]
        assert len(sel) == min(k, len(valid))
        assert all(c == -1 for c in out[t][len(sel):])             # -1 only at tail
        assert sel == sorted(set(sel))                              # ascending, unique
        assert all(lo <= c < hi for c in sel)
        unsel = set(valid) - set(sel)
        for i in sel:                                               # exchange property
            for j in unsel:
                assert lg[t, i] > lg[t, j] or (lg[t, i] == lg[t, j] and i < j)


def test_topk_never_selects_dirty_columns_outside_range():
    # vime PR #502 review: garbage in invalid columns must not be picked.
    T, S, k = 8, 64, 16
    rng = np.random.default_rng(20)
    lg = rng.standard_normal((T, S)).astype(np.float32)
    rs = np.arange(T, dtype=np.int32) * 4
    re = rs + 10
    dirty = lg.copy()
    for t in range(T):
        dirty[t, :rs[t]] = np.inf
        dirty[t, re[t]:] = 1e30
    a = oracle.topk(lg, rs, re, k)
    b = oracle.topk(dirty, rs, re, k)
    assert np.array_equal(a, b)
    assert (b[:, 10:] == -1).all()


def test_topk_closed_forms():
    S = 100
    inc = np.arange(S, dtype=np.float32)[None, :]
    dec = -inc
    const = np.zeros((1, S), np.float32)
    rs, re = np.array([10], np.int32), np.array([90], np.int32)
    assert oracle.topk(inc, rs, re, 5)[0].tolist() == [85, 86, 87, 88, 89]
    assert oracle.topk(dec, rs, re, 5)[0].tolist() == [10, 11, 12, 13, 14]
    assert oracle.topk(const, rs, re, 5)[0].tolist() == [10, 11, 12, 13, 14]
    assert oracle.topk(inc, rs, re, 80)[0].tolist() == list(range(10, 90))
    assert oracle.topk(inc, rs, re, 83)[0].tolist() == list(range(10, 90)) + [-1] * 3


# ------------------------------------------------------------ score order

def test_sort_by_score_hand_example():
    # torch.topk's order (vime PR #502, torch_dsa_topk): descending value;
    # equal values keep the lower column first, -0.0 equals +0.0, and the -1
    # padding stays at the tail.
    lg = np.array([[1.0, 3.0, 2.0, 3.0, -0.0, 0.0]], np.float32)
    assert oracle.sort_by_score(lg, np.array([[0, 1, 2, 3, 4, 5]], np.int32)).tolist() == \
        [[1, 3, 2, 0, 4, 5]]
    assert oracle.sort_by_score(lg, np.array([[5, 4, 2, -1, -1]], np.int32)).tolist() == \
        [[2, 4, 5, -1, -1]]
    # -inf and NaN (never selected by a top-k) are equal and lowest.
    lg2 = np.array([[np.nan, -np.inf, 1.0, np.nan, 2.0]], np.float32)
    assert oracle.sort_by_score(lg2, np.array([[0, 1, 2, 3, 4]], np.int32)).tolist() == \
        [[4, 2, 0, 1, 3]]


def test_sort_by_score_values_match_torch_topk():
    # The sorted scores are exactly torch.topk's (sorted=True) values; the
    # order among equal scores is checked by the invariant below.
    rng = np.random.default_rng(5)
    for _ in range(20):
        S, k = int(rng.integers(5, 300)), int(rng.integers(1, 40))
        lg = rng.standard_normal((3, S)).astype(np.float32)
        lg[:, rng.integers(0, S, size=S // 4)] = np.round(lg[:, :S // 4], 1)  # ties
        rs = np.zeros(3, np.int32)
        re_ = np.full(3, S, np.int32)
        top = oracle.topk(lg, rs, re_, k)
        srt = oracle.sort_by_score(lg, top)
        for t in range(3):
            n = int((srt[t] >= 0).sum())
            want = torch.topk(torch.from_numpy(lg[t]), n).values.numpy()
            assert np.array_equal(lg[t, srt[t, :n]], want)
            # the same set of columns, padding at the tail
            assert sorted(srt[t, :n].tolist()) == sorted(top[t][top[t] >= 0].tolist())
            assert (srt[t, n:] == -1).all()
            # equal scores in ascending column order
            v, c = lg[t, srt[t, :n]], srt[t, :n]
            assert all(v[i] > v[i + 1] or (v[i] == v[i + 1] and c[i] < c[i + 1])
                       for i in range(n - 1))


# -------------------------------------------------- prologue (q quant, K insert)

def test_e4m3_encoder_round_trip_and_ties():
    # Every finite code decodes and encodes back to itself ([OCP-FP8]).
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    vals = oracle.e4m3_to_f64(codes)
    assert np.array_equal(oracle.f64_to_e4m3(vals), codes)
    # Midpoints between neighbouring positive codes go to the even code.
    pos = np.arange(0, 0x7E, dtype=np.uint8)
    a, b = oracle.e4m3_to_f64(pos), oracle.e4m3_to_f64(pos + 1)
    mids = oracle.f64_to_e4m3((a + b) / 2)
    assert np.array_equal(mids, np.where(pos % 2 == 0, pos, pos + 1))
    # Saturation and signed zero.
    assert oracle.f64_to_e4m3([448.0, 460.0, 1e6, -1e6, -0.0]).tolist() == [0x7E, 0x7E, 0x7E, 0xFE, 0x80]


def test_e4m3_encoder_matches_torch_cast():
    rng = np.random.default_rng(3)
    v = (rng.standard_normal(4000) * rng.choice([1e-3, 0.05, 1.0, 60.0], 4000)).clip(-440, 440)
    got = oracle.f64_to_e4m3(v)
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, ref)


def test_q_quant_fold_closed_forms():
    D = 128
    rows = np.zeros((1, 5, D), np.float32)
    rows[0, 0, 0] = 448.0                     # amax = 448: scale 1
    rows[0, 1, 3] = -452.0                    # just above (exact in bf16): scale 2
    rows[0, 2, :] = 0.0                       # all zero: scale 1, codes 0
    rows[0, 3, :] = np.linspace(-1, 1, D)     # amax 1: scale 2^-8 (1 <= 448 * 2^-8 = 1.75)
    rows[0, 4, 7] = 2.0 ** -20                # tiny: scale 2^-28 (2^-20 <= 448 * 2^-28)
    q = bf16(rows)
    w = np.array([[1.0, -2.0, 3.0, 0.5, 4.0]], np.float32)
    q8, wo = oracle.q_quant_fold(q, w, 0.25, padded_heads=8)
    scales = np.array([1.0, 2.0, 1.0, 2.0 ** -8, 2.0 ** -28])
    assert np.array_equal(wo[0, :5], (w[0] * np.float32(0.25)).astype(np.float32) * scales.astype(np.float32))
    assert (wo[0, 5:] == 0).all() and (q8[0, 5:] == 0).all()            # padded heads
    assert q8[0, 0, 0] == 0x7E and q8[0, 1, 3] == oracle.f64_to_e4m3([-226.0])[0] == 0xF6
    assert (q8[0, 2] == 0).all()
    deq = oracle.e4m3_to_f64(q8[0, 3]) * 2.0 ** -8
    src = oracle.bf16_to_f64(q[0, 3])
    assert np.all(np.abs(deq - src) <= np.maximum(np.abs(src) * 2.0 ** -4, 2.0 ** -18))
    assert oracle.e4m3_to_f64(q8[0, 4, 7:8])[0] * 2.0 ** -28 == 2.0 ** -20


def test_q_quant_fold_matches_torch_quantisation():
    # The input generator quantises with torch's own e4m3 cast and the same
    # UE8M0 rule: an independent implementation of the same definition.
    rng = np.random.default_rng(1)
    src = wl.bf16_bits_to_f32(bf16(rng.standard_normal((6, 4, 128)) * 0.1))
    q8_ref, s_ref = wl.quantize_e4m3_blocks(src.reshape(24, 128))
    q8, wo = oracle.q_quant_fold(bf16(src), np.ones((6, 4), np.float32), 1.0, padded_heads=4)
    assert np.array_equal(q8.reshape(24, 128), q8_ref)
    assert np.array_equal(wo.reshape(24), s_ref)


def test_k_norm_insert_layer_norm_and_slots():
    rng = np.random.default_rng(2)
    T, D = 6, 128
    k = rng.standard_normal((T, D)) * 0.3
    k[1] = 0.7                                                 # constant row: output is the bias
    kb = bf16(k)
    g = (1 + 0.1 * rng.standard_normal(D)).astype(np.float32)
    b = (0.05 * rng.standard_normal(D)).astype(np.float32)
    slots = np.array([5, 0, -1, 11, 3, 9], np.int64)           # -1: a padding token
    cache = np.full((3, 4, D), 0x7FC0, np.uint16)              # sentinel bf16 NaN
    oracle.k_norm_insert(kb, g, b, 1e-6, slots, cache)
    flat = cache.reshape(12, D)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(wl.bf16_bits_to_f32(kb)).double(), (D,),
                                         torch.from_numpy(g).double(), torch.from_numpy(b).double(),
                                         1e-6).numpy()
    for t, s in enumerate(slots):
        if s < 0:
            continue
        got = oracle.bf16_to_f64(flat[s])
        assert np.all(np.abs(got - ref[t]) <= np.abs(ref[t]) * 2.0 ** -8 + 1e-30)
    assert np.array_equal(oracle.bf16_to_f64(flat[0]), oracle.bf16_to_f64(bf16(b)))   # constant row
    untouched = [i for i in range(12) if i not in set(slots.tolist())]
    assert (flat[untouched] == 0x7FC0).all()
    # e4m3 cache: the bf16 row quantised with its UE8M0 scale
    c8 = np.zeros((3, 4, D), np.uint8)
    sc = np.zeros(12, np.float32)
    oracle.k_norm_insert(kb, g, b, 1e-6, slots, c8, sc)
    for t, s in enumerate(slots):
        if s < 0:
            continue
        row = oracle.bf16_to_f64(flat[s])
        q8, wo = oracle.q_quant_fold(flat[s][None, None, :], np.ones((1, 1), np.float32), 1.0, 1)
        assert np.array_equal(c8.reshape(12, D)[s], q8[0, 0]) and sc[s] == wo[0, 0]


def test_k_layer_norm_is_torch_layer_norm_in_double():
    # The unrounded LayerNorm the insert rounds: torch's own fp64 layer_norm
    # on the same bf16 inputs, to double rounding; a constant row gives the
    # bias exactly; the insert's bf16 output is within half a bf16 step of it.
    rng = np.random.default_rng(3)
    T, D = 9, 128
    k = rng.standard_normal((T, D)) * rng.choice([0.01, 0.3, 20.0], (T, 1)) + 0.2
    k[4] = -2.5                                                # constant row
    kb = bf16(k)
    g = (1 + 0.1 * rng.standard_normal(D)).astype(np.float32)
    b = (0.05 * rng.standard_normal(D)).astype(np.float32)
    got = oracle.k_layer_norm(kb, g, b, 1e-6)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(wl.bf16_bits_to_f32(kb)).double(), (D,),
                                         torch.from_numpy(g).double(), torch.from_numpy(b).double(),
                                         1e-6).numpy()
    assert np.all(np.abs(got - ref) <= 1e-9 * (np.abs(ref) + 1.0))   # rows of tiny variance amplify rounding
    assert np.array_equal(got[4], b.astype(np.float64))
    cache = np.zeros((1, T, D), np.uint16)
    oracle.k_norm_insert(kb, g, b, 1e-6, np.arange(T, dtype=np.int64), cache)
    rounded = oracle.bf16_to_f64(cache.reshape(T * D)).reshape(T, D)
    assert np.all(np.abs(rounded - got) <= np.abs(got) * 2.0 ** -8 + 1e-30)


# ----------------------------------------------------------- rank merge

def test_topk_merge_hand_example_and_whole_row():
    sc = np.array([[0.5, 2.0, 2.0, -np.inf, 1.0, 0.0, -0.0, np.nan]], np.float32)
    cc = np.array([[10, 7, 3, 4, -1, 2, 1, 9]], np.int32)     # -1: an empty slot
    # 2.0 at columns 3 and 7 (3 first), then 0.5 (10), then 0.0 / -0.0 (1 before 2)
    assert oracle.topk_merge(sc, cc, 4).tolist() == [[1, 3, 7, 10]]
    assert oracle.topk_merge(sc, cc, 8).tolist() == [[1, 2, 3, 7, 10, -1, -1, -1]]
    # All columns of a row as one candidate set: the masked top-k itself.
    rng = np.random.default_rng(8)
    lg = np.round(rng.standard_normal((4, 90)), 1).astype(np.float32)
    cols = np.tile(np.arange(90, dtype=np.int32), (4, 1))
    assert np.array_equal(oracle.topk_merge(lg, cols, 17),
                          oracle.topk(lg, np.zeros(4, np.int32), np.full(4, 90, np.int32), 17))


def test_topk_merge_of_interleaved_local_topk_is_the_global_topk():
    # Every column of the global top-k is in its own rank's local top-k, so
    # merging the local top-ks reproduces the global one, ties included.
    from top_selection_dsa_gb300 import dcp
    rng = np.random.default_rng(4)
    for world, inter in ((2, 1), (3, 4), (4, 64)):
        S, T, k = 700, 5, 40
        lg = np.round(rng.standard_normal((T, S)), 1).astype(np.float32)
        L = rng.integers(1, S + 1, T).astype(np.int32)
        cand_s, cand_c = [], []
        for r in range(world):
            pos = dcp.owned_positions(S, r, world, inter).numpy()
            loc = lg[:, pos]
            ln = np.array([dcp.local_len(int(x), r, world, inter) for x in L], np.int32)
            top = oracle.topk(loc, np.zeros(T, np.int32), ln, k)
            g = np.where(top >= 0, pos[np.maximum(top, 0)], -1)
            cand_s.append(np.where(top >= 0, np.take_along_axis(loc, np.maximum(top, 0), 1), -np.inf))
            cand_c.append(g)
        merged = oracle.topk_merge(np.concatenate(cand_s, 1), np.concatenate(cand_c, 1), k)
        assert np.array_equal(merged, oracle.topk(lg, np.zeros(T, np.int32), L, k))


# ------------------------------------------------------------------ MXFP4

def _golden_json(name):
    import json
    import os
    with open(os.path.join(os.path.dirname(__file__), "golden", name)) as f:
        return json.load(f)


def test_e2m1_and_e8m0_decoders_match_the_mx_definition():
    g = _golden_json("e2m1_codes.json")
    got = oracle.e2m1_to_f64(range(16))
    for c in range(16):
        want = g["e2m1"][str(c)]
        assert got[c] == want and np.signbit(got[c]) == np.signbit(want), c
    codes = [int(c) for c in g["e8m0"]]
    got = oracle.e8m0_to_f64(codes)
    assert np.array_equal(got, np.array([g["e8m0"][str(c)] for c in codes]))
    assert np.isnan(oracle.e8m0_to_f64([255])[0])
    # every code: the value doubles with the exponent field
    assert np.array_equal(oracle.e8m0_to_f64(range(1, 255)), 2.0 * oracle.e8m0_to_f64(range(0, 254)))


def test_mxfp4_logits_hand_example():
    g = _golden_json("mxfp4_hand_example.json")
    q = np.zeros((1, 1, 32), np.uint8)
    k = np.zeros((2, 32), np.uint8)
    for i, v in g["q_bytes"].items():
        q[0, 0, int(i)] = v
    for row, key in ((0, "k0_bytes"), (1, "k1_bytes")):
        for i, v in g[key].items():
            k[row, int(i)] = v
    q_sf = np.array(g["q_sf"], np.uint8).reshape(1, 1, 2)
    k_sf = np.array([g["k0_sf"], g["k1_sf"]], np.uint8)
    w = np.full((1, 1), g["w"], np.float32)
    got = oracle.logits_mxfp4(q, q_sf, k, k_sf, w, np.zeros(1, np.int32), np.full(1, 2, np.int32))
    assert got.tolist() == [g["logits"]]


def _decode_mx_with_table(packed, sf):
    """Decoded values from the golden E2M1 table (independent of the oracle)."""
    g = _golden_json("e2m1_codes.json")
    table = np.array([g["e2m1"][str(c)] for c in range(16)])
    codes = np.empty(packed.shape[:-1] + (2 * packed.shape[-1],), np.uint8)
    codes[..., 0::2] = packed & 15
    codes[..., 1::2] = packed >> 4
    scale = np.ldexp(1.0, sf.astype(np.int64) - 127)
    return table[codes] * np.repeat(scale, 32, axis=-1)


def test_mxfp4_logits_equal_the_bf16_oracle_on_the_decoded_values():
    # E2M1 values times powers of two near 1 are exact in bf16: the MXFP4
    # logits must equal the (separately pinned) bf16 oracle's on those values,
    # bit for bit (same fp64 sums in the same order).
    rng = np.random.default_rng(21)
    T, S, H, D = 9, 70, 4, 64
    q = rng.integers(0, 256, (T, H, D // 2)).astype(np.uint8)
    k = rng.integers(0, 256, (S, D // 2)).astype(np.uint8)
    q_sf = rng.integers(120, 135, (T, H, D // 32)).astype(np.uint8)
    k_sf = rng.integers(120, 135, (S, D // 32)).astype(np.uint8)
    w = rng.standard_normal((T, H)).astype(np.float32)
    rs = rng.integers(-3, 40, T).astype(np.int32)
    re = (rs + rng.integers(0, 50, T)).astype(np.int32)
    qv = _decode_mx_with_table(q, q_sf)
    kv = _decode_mx_with_table(k, k_sf)
    assert np.array_equal(wl.bf16_bits_to_f32(bf16(qv)), qv)      # exact in bf16
    assert np.array_equal(wl.bf16_bits_to_f32(bf16(kv)), kv)
    ref = oracle.logits(bf16(qv), bf16(kv), w, rs, re)
    got = oracle.logits_mxfp4(q, q_sf, k, k_sf, w, rs, re)
    assert np.array_equal(got, ref)


def test_mxfp4_quantiser_of_the_input_generator():
    # Encoding only (the generator's job): the decoded block is the nearest
    # E2M1 value times the block scale, ties to the even code, and the scale
    # is the smallest power of two with amax <= 6 * scale.
    rng = np.random.default_rng(22)
    x = rng.standard_normal((40, 128)) * rng.choice([1e-3, 0.1, 3.0, 500.0], (40, 1))
    x[0, :32] = 0.0                                   # an all-zero block
    x[1, :32] = 6.0                                   # amax exactly 6 -> scale 1
    x[2, :4] = [0.25, 0.75, 1.25, 2.5]                # ties (with amax 6 below)
    x[2, 4] = 6.0
    packed, sf = wl.quantize_mxfp4_blocks(x)
    dec = _decode_mx_with_table(packed, sf)
    scale = np.ldexp(1.0, sf.astype(np.int64) - 127)
    amax = np.abs(x.reshape(40, 4, 32)).max(-1)
    assert np.all(amax <= 6 * scale) and np.all((amax == 0) | (amax > 3 * scale))
    assert sf[0, 0] == 127 and sf[1, 0] == 127
    assert dec[2, :4].tolist() == [0.0, 1.0, 1.0, 2.0]  # ties go to the even code
    grid = np.concatenate([-wl.E2M1_GRID[::-1], wl.E2M1_GRID])
    y = x / np.repeat(scale, 32, axis=1)
    nearest = grid[np.abs(y[..., None] - grid).argmin(-1)]
    err_best = np.abs(y - nearest)
    assert np.all(np.abs(dec / np.repeat(scale, 32, axis=1) - y) <= err_best + 1e-12)
