"""The seeded input generators produce the shapes and structure they promise."""
import numpy as np

from top_selection_dsa_gb300 import workloads as wl


def test_tiny_causal_shapes_and_ranges():
    p = wl.tiny_causal()
    assert (p.T, p.S, p.H, p.D, p.topk) == (256, 256, 4, 64, 32)
    assert p.q.dtype == np.uint16 and p.k.dtype == np.uint16 and p.w.dtype == np.float32
    assert (p.row_starts == 0).all() and (p.row_ends == np.arange(1, 257)).all()
    assert p.valid_pairs() == 256 * 257 // 2
    again = wl.tiny_causal()
    assert np.array_equal(again.q, p.q) and np.array_equal(again.w, p.w)


def test_distribution_scales():
    p = wl.prefill(512, 512, 16, 128, 8, seed=3)
    q = wl.bf16_bits_to_f32(p.q)
    assert abs(q.std() - 128 ** -0.5) < 0.01 * 128 ** -0.5 * 10
    assert abs(p.w.std() - (1 / 4) * 128 ** -0.5) < 0.1 * (1 / 4) * 128 ** -0.5


def test_thd_ranges():
    lens = wl.thd_seq_lens(8, 512, 8192, seed=0)
    assert len(lens) == 8 and all(512 <= L <= 8192 for L in lens)
    rs, re = wl.thd_ranges([3, 2])
    assert rs.tolist() == [0, 0, 0, 3, 3] and re.tolist() == [1, 2, 3, 4, 5]


def test_paged_block_table_is_a_permutation():
    p = wl.paged_decode(B=6, next_n=2, ctx_lo=100, ctx_hi=1000, block_size=16,
                        H=2, D=64, topk=8, seed=4)
    used = []
    for b in range(p.B):
        n = -(-int(p.context_lens[b]) // 16)
        used.extend(p.block_table[b, :n].tolist())
    assert sorted(used) == list(range(p.k_cache.shape[0]))
    assert ((p.context_lens >= 100) & (p.context_lens <= 1000)).all()
    assert p.max_blocks == -(-1000 // 16)


def test_e4m3_block_quantisation():
    rng = np.random.default_rng(5)
    x = wl.bf16_bits_to_f32(wl.to_bf16_bits(rng.standard_normal((300, 128)).astype(np.float32) * 0.1))
    x[7] = 0
    codes, sc = wl.quantize_e4m3_blocks(x)
    m, e = np.frexp(sc)
    assert (m == 0.5).all()                                # powers of two
    assert sc[7] == 1.0
    import torch
    deq = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy() * sc[:, None]
    assert not np.isnan(deq).any()
    amax = np.abs(x).max(1)
    assert (amax / sc <= 448).all() and (amax[amax > 0] / sc[amax > 0] > 224).all()
    assert np.allclose(deq, x, rtol=2 ** -4, atol=1e-30 + 2 ** -9 * sc[:, None].max())
