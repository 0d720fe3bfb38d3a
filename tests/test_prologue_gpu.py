"""The steps before the indexer on the GPU against the oracle.

q quantisation + weight fold is bit-exact (the scale is an exact power of two
and the codes round the same exact value).  The key LayerNorm runs in fp32 on
the GPU and in double in the oracle: each bf16 output may differ by one bf16
step, and an e4m3 code by one step where its bf16 input did.
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


def bf16_dev(bits):
    return dev(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def q_rows(rng, T, H):
    x = rng.standard_normal((T, H, 128)) * rng.choice([1e-4, 0.05, 1.0, 300.0], (T, H, 1))
    flat = x.reshape(T * H, 128)
    special = [np.zeros(128),                    # all-zero row
               np.full(128, -0.0),               # negative zeros
               np.where(np.arange(128) == 5, 448.0, 0.01),          # amax exactly 448 * 2^0
               np.where(np.arange(128) == 9, 896.0, -3.0)]          # amax exactly 448 * 2^1
    for i, row in enumerate(special[:T * H]):
        flat[i] = row
    return wl.to_bf16_bits(x.astype(np.float32))


@pytest.mark.parametrize("T,H,Hp", [(1, 1, 1), (37, 64, 64), (50, 24, 32), (300, 64, 64)])
def test_q_quant_fold_bit_exact(api, T, H, Hp):
    rng = np.random.default_rng(T * 100 + H)
    q = q_rows(rng, T, H)
    w = rng.standard_normal((T, H)).astype(np.float32)
    ws = float(np.float32(128 ** -0.5 * H ** -0.5))
    q8, wo = api.q_quant_fold_weights(bf16_dev(q), dev(w), ws, Hp)
    r8, ro = oracle.q_quant_fold(q, w, ws, Hp)
    assert np.array_equal(q8.view(torch.uint8).cpu().numpy(), r8)
    assert np.array_equal(wo.cpu().numpy(), ro)


def test_q_quant_fold_full_size_sampled(api):
    # The e4m3 workload's query: T=32768 rows of 64 heads, every row checked
    # against the oracle on a sample.
    T, H = 32768, 64
    rng = np.random.default_rng(7)
    q = wl.to_bf16_bits((rng.standard_normal((T, H, 128)) / np.sqrt(128)).astype(np.float32))
    w = (rng.standard_normal((T, H)) / 8).astype(np.float32)
    ws = float(np.float32(128 ** -0.5 * 64 ** -0.5))
    q8, wo = api.q_quant_fold_weights(bf16_dev(q), dev(w), ws, 64)
    rows = np.unique(np.concatenate([rng.integers(0, T, 48), [0, 1, T - 1]]))
    r8, ro = oracle.q_quant_fold(q[rows], w[rows], ws, 64)
    assert np.array_equal(q8.view(torch.uint8)[dev(rows).long()].cpu().numpy(), r8)
    assert np.array_equal(wo[dev(rows).long()].cpu().numpy(), ro)


def ln_inputs(rng, T):
    k = rng.standard_normal((T, 128)) * 0.5 + 0.1
    k[0] = 1.25                                  # constant row
    kb = wl.to_bf16_bits(k.astype(np.float32))
    g = (1 + 0.2 * rng.standard_normal(128)).astype(np.float32)
    b = (0.1 * rng.standard_normal(128)).astype(np.float32)
    return kb, g, b


def test_k_norm_insert_bf16_cache(api):
    rng = np.random.default_rng(5)
    T, nb, bs = 200, 8, 64
    kb, g, b = ln_inputs(rng, T)
    slots = rng.permutation(nb * bs)[:T].astype(np.int64)
    slots[3] = -1                                # padding token
    cache = torch.full((nb, bs, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    api.k_norm_quant_insert(bf16_dev(kb), dev(g), dev(b), 1e-6, dev(slots), cache)
    got = cache.view(torch.int16).cpu().numpy().view(np.uint16).reshape(nb * bs, 128)
    ref = np.full((nb, bs, 128), 0x7FC0, np.uint16)
    oracle.k_norm_insert(kb, g, b, 1e-6, slots, ref)
    ref = ref.reshape(nb * bs, 128)
    live = slots[slots >= 0]
    gv, rv = oracle.bf16_to_f64(got[live]), oracle.bf16_to_f64(ref[live])
    assert np.all(np.abs(gv - rv) <= np.abs(rv) * 2.0 ** -7 + 1e-30)    # at most one bf16 step
    assert np.mean(got[live] == ref[live]) > 0.999
    idle = np.setdiff1d(np.arange(nb * bs), live)
    assert np.all(np.isnan(oracle.bf16_to_f64(got[idle])))              # nothing else written


def test_k_norm_insert_e4m3_cache_and_bad_slot(api):
    rng = np.random.default_rng(6)
    T, nb, bs = 300, 5, 64
    kb, g, b = ln_inputs(rng, T)
    slots = rng.permutation(nb * bs)[:T].astype(np.int64)
    slots[7] = nb * bs + 3                       # past the cache: skipped and reported
    c8 = torch.zeros((nb, bs, 128), dtype=torch.uint8, device="cuda")
    sc = torch.zeros(nb * bs, dtype=torch.float32, device="cuda")
    api.k_norm_quant_insert(bf16_dev(kb), dev(g), dev(b), 1e-6, dev(slots), c8, sc)
    assert api.last_device_error() == api.DSA_ERR_INVALID_ARG
    r8 = np.zeros((nb, bs, 128), np.uint8)
    rs = np.zeros(nb * bs, np.float32)
    oracle.k_norm_insert(kb, g, b, 1e-6, slots, r8, rs)
    live = slots[(slots >= 0) & (slots < nb * bs)]
    got8 = c8.cpu().numpy().reshape(nb * bs, 128)[live]
    ref8 = r8.reshape(nb * bs, 128)[live]
    gs, rsl = sc.cpu().numpy()[live], rs[live]
    assert np.mean(gs == rsl) > 0.99                                   # same UE8M0 scale
    same = gs == rsl
    gd = oracle.e4m3_to_f64(got8[same].ravel()).reshape(-1, 128) * gs[same, None]
    rd = oracle.e4m3_to_f64(ref8[same].ravel()).reshape(-1, 128) * rsl[same, None]
    step = np.abs(rd) * 2.0 ** -3 + rsl[same, None] * 2.0 ** -9        # one e4m3 step
    assert np.all(np.abs(gd - rd) <= step)
    assert np.mean(got8[same] == ref8[same]) > 0.995
