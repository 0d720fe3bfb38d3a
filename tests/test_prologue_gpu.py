"""The steps before the indexer on the GPU against the oracle.

q quantisation + weight fold is bit-exact (the scale is an exact power of two
and the codes round the same exact value).  The key LayerNorm runs in fp32 on
the GPU (the page's F.layer_norm on x.float()) and in double in the oracle:
every bf16 output must be the nearest-even rounding of the exact value, except
where the exact value lies within the fp32 computation's error bound of a
rounding midpoint; the e4m3 cache must hold exactly the oracle's quantisation
of those bf16 rows.
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


def ln_error_bound(kb, g, b, eps):
    """Bound on |fp32 LayerNorm - exact LayerNorm| per element, from the
    operations the fp32 computation rounds: the mean (a sum of 128 terms, at
    most 11 roundings deep), the variance and rsqrt (a few ulp), and the
    products and the bias add (one rounding each), with a wide margin."""
    x = wl.bf16_bits_to_f32(kb).astype(np.float64)
    mean = x.mean(axis=1, keepdims=True)
    rstd = 1.0 / np.sqrt(((x - mean) ** 2).mean(axis=1, keepdims=True) + eps)
    p = (x - mean) * rstd * g
    mean_err = np.abs(x).mean(axis=1, keepdims=True) * rstd * np.abs(g)
    return 2.0 ** -17 * (np.abs(p) + np.abs(b)) + 2.0 ** -18 * mean_err


def assert_bf16_rounding_of(got_bits, v64, delta, what):
    """Every bf16 in got_bits is the nearest-even bf16 of the exact value v64,
    except where v64 lies within delta (the fp32 computation's error bound)
    of the midpoint between its two bf16 neighbours: there either neighbour
    is a correct rounding of a value the fp32 computation may produce."""
    got = oracle.bf16_to_f64(got_bits.ravel()).reshape(v64.shape)
    _, e = np.frexp(np.abs(v64))                       # |v| in [2^(e-1), 2^e)
    ulp = np.ldexp(1.0, e - 8)                         # bf16 spacing there
    lo = np.floor(v64 / ulp) * ulp
    hi = lo + ulp
    mid = lo + ulp / 2
    even_lo = (np.round(np.abs(lo) / ulp).astype(np.int64) % 2) == 0
    nearest = np.where(v64 - lo < hi - v64, lo, np.where(hi - v64 < v64 - lo, hi,
                                                         np.where(even_lo, lo, hi)))
    nearest = np.where(v64 == 0, 0.0, nearest)
    exact = got == nearest
    near_mid = (np.abs(v64 - mid) <= delta) & ((got == lo) | (got == hi))
    bad = ~(exact | near_mid)
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} bf16 values are neither "
                           f"the rounding of the exact LayerNorm nor a midpoint case; first "
                           f"at {np.argwhere(bad)[0].tolist()}: got {got[bad][0]!r}, exact "
                           f"{v64[bad][0]!r}")
    return int((~exact).sum())


def test_k_norm_insert_bf16_cache(api):
    rng = np.random.default_rng(5)
    T, nb, bs = 200, 8, 64
    kb, g, b = ln_inputs(rng, T)
    slots = rng.permutation(nb * bs)[:T].astype(np.int64)
    slots[3] = -1                                # padding token
    cache = torch.full((nb, bs, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    api.k_norm_quant_insert(bf16_dev(kb), dev(g), dev(b), 1e-6, dev(slots), cache)
    got = cache.view(torch.int16).cpu().numpy().view(np.uint16).reshape(nb * bs, 128)
    live_t = np.nonzero(slots >= 0)[0]
    v64 = oracle.k_layer_norm(kb, g, b, 1e-6)[live_t]
    delta = ln_error_bound(kb, g, b, 1e-6)[live_t]
    assert_bf16_rounding_of(got[slots[live_t]], v64, delta, "bf16 cache")
    ref = np.full((nb, bs, 128), 0x7FC0, np.uint16)          # the oracle's own insert
    oracle.k_norm_insert(kb, g, b, 1e-6, slots, ref)
    assert np.mean(got[slots[live_t]] == ref.reshape(nb * bs, 128)[slots[live_t]]) > 0.99
    idle = np.setdiff1d(np.arange(nb * bs), slots[live_t])
    assert np.all(np.isnan(oracle.bf16_to_f64(got[idle])))    # nothing else written


def test_k_norm_insert_e4m3_cache_and_bad_slot(api):
    # The e4m3 cache holds the bf16 LayerNorm output quantised with its
    # UE8M0 scale: the same rows written to a bf16 cache (checked against the
    # exact LayerNorm as above) must quantise, by the oracle's rule, to
    # exactly the codes and scales of the e4m3 cache.
    rng = np.random.default_rng(6)
    T, nb, bs = 300, 5, 64
    kb, g, b = ln_inputs(rng, T)
    slots = rng.permutation(nb * bs)[:T].astype(np.int64)
    slots[7] = nb * bs + 3                       # past the cache: skipped and reported
    c8 = torch.zeros((nb, bs, 128), dtype=torch.uint8, device="cuda")
    sc = torch.zeros(nb * bs, dtype=torch.float32, device="cuda")
    api.k_norm_quant_insert(bf16_dev(kb), dev(g), dev(b), 1e-6, dev(slots), c8, sc)
    assert api.last_device_error() == api.DSA_ERR_INVALID_ARG
    c16 = torch.zeros((nb, bs, 128), dtype=torch.bfloat16, device="cuda")
    api.k_norm_quant_insert(bf16_dev(kb), dev(g), dev(b), 1e-6, dev(slots), c16)
    assert api.last_device_error() == api.DSA_ERR_INVALID_ARG
    live_t = np.nonzero((slots >= 0) & (slots < nb * bs))[0]
    live = slots[live_t]
    rows16 = c16.view(torch.int16).cpu().numpy().view(np.uint16).reshape(nb * bs, 128)[live]
    assert_bf16_rounding_of(rows16, oracle.k_layer_norm(kb, g, b, 1e-6)[live_t],
                            ln_error_bound(kb, g, b, 1e-6)[live_t], "e4m3 path's bf16 rows")
    r8, rs = oracle.q_quant_fold(rows16[:, None, :], np.ones((len(live), 1), np.float32), 1.0, 1)
    assert np.array_equal(c8.cpu().numpy().reshape(nb * bs, 128)[live], r8[:, 0])
    assert np.array_equal(sc.cpu().numpy()[live], rs[:, 0])
    untouched = np.setdiff1d(np.arange(nb * bs), live)
    assert (c8.cpu().numpy().reshape(nb * bs, 128)[untouched] == 0).all()
