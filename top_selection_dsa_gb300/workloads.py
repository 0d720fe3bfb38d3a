"""Seeded synthetic inputs for the DSA lightning-indexer path.

This module is shared by the CUDA path's tests/benchmark and by the CPU oracle.
It holds none of the method's arithmetic: it only draws random numbers,
encodes them into the input formats (bf16, or e4m3 with power-of-two block
scales) and lays out row ranges, packed sequences and block tables.

Workloads (shapes and distributions of the lightning-indexer configurations):
  tiny_causal      T=S=256, H=4, D=64, k=32, single causal sequence
  prefill_causal   T=S=4096, H=64, D=128, k=2048, single causal sequence
  prefill_thd      8 packed sequences, lengths U[512, 8192], H=64, D=128, k=2048
  paged_decode     64 requests x 2 query tokens, contexts log-U[4096, 131072],
                   bf16 K cache in 64-token blocks behind a permuted block table
  prefill_fp8      T=S=32768, H=64, D=128, k=2048, e4m3 q/k with UE8M0 scales
  prefill_mxfp4    T=S=32768, H=64, D=128, k=2048, MXFP4 q/k (E2M1 elements,
                   one E8M0 scale per 32-element block)

Distributions: q, k ~ N(0, 1/D) rounded to bf16; weights ~ N(0,1)/sqrt(H),
times D^-0.5 for every workload but the tiny one (the index softmax scale that
KimiK3DSAIndexer.score folds into the weights, vLLM page
"vllm.models.kimi_k3.nvidia.dsa").

FP8 inputs: each block of D=128 elements (one key row, or one (token, head)
query row; quant_block_size = index_head_dim on the same page) gets the scale
2^ceil(log2(amax/448)) (1 when amax is 0), stored as fp32; the element is
x/scale rounded to nearest-even e4m3 (never saturates, since |x/scale| <= 448).
The query scale is folded into the weights (w' = w * scale_q, exact for a
power of two), as the page's score() does before calling the indexer op, so
the query side carries no scale of its own.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

BF16 = 0
E4M3 = 1
MXFP4 = 2
E4M3_MAX = 448.0
E2M1_MAX = 6.0
MX_BLOCK = 32
# E2M1 magnitudes of codes 0..7 (OCP Microscaling Formats, E2M1: bias 1).
E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


@dataclass
class Prefill:
    """Contiguous-key workload: q [T,H,D], k [S,D], w [T,H], ranges [T]."""
    name: str
    dtype: int
    q: np.ndarray                 # uint16 (bf16 bits) or uint8 (e4m3 codes)
    k: np.ndarray
    w: np.ndarray                 # float32 [T, H]
    row_starts: np.ndarray        # int32 [T]
    row_ends: np.ndarray          # int32 [T]
    topk: int
    k_scale: np.ndarray | None = None   # float32 [S] (e4m3 only)
    seq_lens: list = field(default_factory=list)

    @property
    def T(self):
        return self.q.shape[0]

    @property
    def H(self):
        return self.q.shape[1]

    @property
    def D(self):
        return self.q.shape[2]

    @property
    def S(self):
        return self.k.shape[0]

    def valid_pairs(self) -> int:
        lo = np.clip(self.row_starts.astype(np.int64), 0, self.S)
        hi = np.clip(self.row_ends.astype(np.int64), 0, self.S)
        return int(np.maximum(hi - lo, 0).sum())


@dataclass
class PrefillMX:
    """Contiguous-key workload with MXFP4 operands: packed E2M1 q [T,H,D/2]
    and k [S,D/2] (uint8, low nibble = even element), E8M0 block scales
    q_sf [T,H,D/32] and k_sf [S,D/32] (uint8), fp32 weights [T,H] without
    the query scale (it stays in q_sf)."""
    name: str
    q: np.ndarray
    q_sf: np.ndarray
    k: np.ndarray
    k_sf: np.ndarray
    w: np.ndarray
    row_starts: np.ndarray
    row_ends: np.ndarray
    topk: int
    dtype: int = MXFP4
    seq_lens: list = field(default_factory=list)

    @property
    def T(self):
        return self.q.shape[0]

    @property
    def H(self):
        return self.q.shape[1]

    @property
    def D(self):
        return 2 * self.q.shape[2]

    @property
    def S(self):
        return self.k.shape[0]

    def valid_pairs(self) -> int:
        lo = np.clip(self.row_starts.astype(np.int64), 0, self.S)
        hi = np.clip(self.row_ends.astype(np.int64), 0, self.S)
        return int(np.maximum(hi - lo, 0).sum())


@dataclass
class Paged:
    """Paged decode workload over a block-table-addressed K cache."""
    name: str
    dtype: int
    q: np.ndarray                 # [B*next_n, H, D]
    w: np.ndarray                 # float32 [B*next_n, H]
    k_cache: np.ndarray           # [num_blocks, block_size, D]
    block_table: np.ndarray       # int32 [B, max_blocks]
    context_lens: np.ndarray      # int32 [B]
    next_n: int
    topk: int
    k_scale: np.ndarray | None = None   # float32 [num_blocks, block_size]

    @property
    def B(self):
        return self.block_table.shape[0]

    @property
    def H(self):
        return self.q.shape[1]

    @property
    def D(self):
        return self.q.shape[2]

    @property
    def block_size(self):
        return self.k_cache.shape[1]

    @property
    def max_blocks(self):
        return self.block_table.shape[1]

    @property
    def R(self):
        return self.q.shape[0]

    def max_ctx(self) -> int:
        return self.max_blocks * self.block_size

    def valid_pairs(self) -> int:
        L = self.context_lens.astype(np.int64)
        n = self.next_n
        return int(sum(max(int(l) - n + j + 1, 0) for l in L for j in range(n)))


# ----------------------------------------------------------------- encoders

def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest-even); return the uint16 bit patterns."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def ue8m0_scale(amax: np.ndarray) -> np.ndarray:
    """Power-of-two scale 2^ceil(log2(amax/448)); 1 where amax == 0."""
    ratio = np.asarray(amax, dtype=np.float64) / E4M3_MAX
    m, e = np.frexp(ratio)                  # ratio = m * 2^e, m in [0.5, 1)
    e = np.where(m == 0.5, e - 1, e)        # exact powers of two stay put
    s = np.ldexp(1.0, e).astype(np.float32)
    return np.where(ratio > 0, s, np.float32(1.0)).astype(np.float32)


def quantize_e4m3_blocks(x: np.ndarray):
    """Quantise rows of x [..., D] (one block per row) to e4m3 + fp32 scale."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    amax = np.abs(x).max(axis=-1)
    scale = ue8m0_scale(amax)
    xs = x / scale[..., None]
    codes = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return codes, scale


def quantize_mxfp4_blocks(x: np.ndarray):
    """Quantise rows of x [rows, D] (D a multiple of 32) to MXFP4: per block
    of 32 elements the E8M0 scale 2^e, e = ceil(log2(amax / 6)) (0 for an
    all-zero block), and each element x / 2^e rounded to the nearest E2M1
    value, ties to the even code (|x / 2^e| <= 6, so nothing saturates).
    Returns (packed [rows, D/2] uint8 with the even element in the low
    nibble, scales [rows, D/32] uint8)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    rows, D = x.shape
    blocks = x.reshape(rows, D // MX_BLOCK, MX_BLOCK)
    amax = np.abs(blocks).max(axis=-1)
    m, e = np.frexp(amax / E2M1_MAX)
    e = np.where(m == 0.5, e - 1, e)
    e = np.where(amax > 0, e, 0)
    e = np.clip(e, -127, 127)
    y = blocks / np.ldexp(1.0, e)[..., None]
    mag = np.abs(y)
    hi = np.clip(np.searchsorted(E2M1_GRID, mag, side="left"), 0, 7)
    lo = np.clip(hi - 1, 0, 7)
    dlo, dhi = mag - E2M1_GRID[lo], E2M1_GRID[hi] - mag
    code = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(lo % 2 == 0, lo, hi)))
    code = (code | np.where(np.signbit(y), 8, 0)).astype(np.uint8).reshape(rows, D)
    packed = (code[:, 0::2] | (code[:, 1::2] << 4)).astype(np.uint8)
    return packed, (e + 127).astype(np.uint8)


def _normal_bf16(rng, shape, std, chunk_rows=1 << 16):
    """N(0, std^2) rounded to bf16, generated in row chunks to bound memory."""
    rows = shape[0]
    inner = int(np.prod(shape[1:]))
    out = np.empty((rows, inner), dtype=np.uint16)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        x = rng.standard_normal((r1 - r0, inner), dtype=np.float32) * np.float32(std)
        out[r0:r1] = to_bf16_bits(x)
    return out.reshape(shape)


def _weights(rng, T, H, softmax_scale):
    w = rng.standard_normal((T, H), dtype=np.float32) / np.float32(math.sqrt(H))
    if softmax_scale:
        w = w * np.float32(1.0 / math.sqrt(softmax_scale))
    return w.astype(np.float32)


def causal_ranges(T: int):
    rs = np.zeros(T, dtype=np.int32)
    re = np.arange(1, T + 1, dtype=np.int32)
    return rs, re


def thd_ranges(seq_lens):
    """Packed sequences: row t of sequence i sees [off_i, off_i + pos + 1)."""
    rs, re = [], []
    off = 0
    for L in seq_lens:
        rs.append(np.full(L, off, dtype=np.int32))
        re.append(off + np.arange(1, L + 1, dtype=np.int32))
        off += L
    return np.concatenate(rs), np.concatenate(re)


# ---------------------------------------------------------------- workloads

def prefill(T, S, H, D, topk, row_starts=None, row_ends=None, *, seed=0,
            softmax_scale=True, name="prefill", dtype=BF16) -> Prefill:
    """Generic contiguous-key workload (causal ranges unless given)."""
    rng = _rng(seed)
    if row_starts is None:
        assert T == S, "default ranges are causal and need T == S"
        row_starts, row_ends = causal_ranges(T)
    std = 1.0 / math.sqrt(D)
    w = _weights(rng, T, H, D if softmax_scale else 0)
    if dtype == BF16:
        q = _normal_bf16(rng, (T, H, D), std)
        k = _normal_bf16(rng, (S, D), std)
        return Prefill(name, BF16, q, k, w, np.asarray(row_starts, np.int32),
                       np.asarray(row_ends, np.int32), topk)
    # e4m3: bf16 sources, then per-row block quantisation; q scale into w.
    qsrc = bf16_bits_to_f32(_normal_bf16(rng, (T * H, D), std))
    ksrc = bf16_bits_to_f32(_normal_bf16(rng, (S, D), std))
    q8, sq = quantize_e4m3_blocks(qsrc)
    k8, sk = quantize_e4m3_blocks(ksrc)
    del qsrc, ksrc
    w = (w * sq.reshape(T, H)).astype(np.float32)
    return Prefill(name, E4M3, q8.reshape(T, H, D), k8, w,
                   np.asarray(row_starts, np.int32), np.asarray(row_ends, np.int32),
                   topk, k_scale=sk)


def prefill_mx(T, S, H, D, topk, row_starts=None, row_ends=None, *, seed=0,
               name="prefill_mxfp4") -> PrefillMX:
    """MXFP4 workload: q, k ~ N(0, 1/D) rounded to bf16, then quantised to
    MXFP4 by blocks of 32; w ~ N(0,1)/sqrt(H) * D^-0.5 (the softmax scale;
    the query's block scales stay separate, as mxfp4_q_quant returns them)."""
    rng = _rng(seed)
    if row_starts is None:
        assert T == S, "default ranges are causal and need T == S"
        row_starts, row_ends = causal_ranges(T)
    std = 1.0 / math.sqrt(D)
    w = _weights(rng, T, H, D)
    qsrc = bf16_bits_to_f32(_normal_bf16(rng, (T * H, D), std))
    ksrc = bf16_bits_to_f32(_normal_bf16(rng, (S, D), std))
    q4, qsf = quantize_mxfp4_blocks(qsrc)
    del qsrc
    k4, ksf = quantize_mxfp4_blocks(ksrc)
    return PrefillMX(name, q4.reshape(T, H, D // 2), qsf.reshape(T, H, D // MX_BLOCK), k4, ksf,
                     w, np.asarray(row_starts, np.int32), np.asarray(row_ends, np.int32), topk)


def prefill_mxfp4(T=32768, H=64, D=128, topk=2048, seed=0) -> PrefillMX:
    return prefill_mx(T, T, H, D, topk, seed=seed, name=f"prefill_mxfp4_T{T}_H{H}_D{D}_k{topk}")


def tiny_causal(seed=0) -> Prefill:
    """T=S=256, H=4, D=64, k=32; w ~ N(0,1)/sqrt(H) (no D^-0.5)."""
    return prefill(256, 256, 4, 64, 32, seed=seed, softmax_scale=False,
                   name="tiny_causal_T256_H4_D64_k32")


def prefill_causal(T=4096, H=64, D=128, topk=2048, seed=0) -> Prefill:
    return prefill(T, T, H, D, topk, seed=seed,
                   name=f"prefill_causal_T{T}_H{H}_D{D}_k{topk}")


def thd_seq_lens(n_seqs=8, lo=512, hi=8192, seed=0):
    return [int(x) for x in _rng(seed).integers(lo, hi + 1, size=n_seqs)]


def prefill_thd(n_seqs=8, lo=512, hi=8192, H=64, D=128, topk=2048, seed=0) -> Prefill:
    lens = thd_seq_lens(n_seqs, lo, hi, seed)
    rs, re = thd_ranges(lens)
    T = int(sum(lens))
    p = prefill(T, T, H, D, topk, rs, re, seed=seed + 1,
                name=f"prefill_thd_{n_seqs}seqs_U{lo}-{hi}_H{H}_D{D}_k{topk}")
    p.seq_lens = lens
    return p


def prefill_fp8(T=32768, H=64, D=128, topk=2048, seed=0) -> Prefill:
    return prefill(T, T, H, D, topk, seed=seed, dtype=E4M3,
                   name=f"prefill_fp8_T{T}_H{H}_D{D}_k{topk}")


def decode_context_lens(B=64, lo=4096, hi=131072, seed=0):
    u = _rng(seed).uniform(math.log(lo), math.log(hi), size=B)
    return np.clip(np.round(np.exp(u)), lo, hi).astype(np.int32)


def paged_decode(B=64, next_n=2, ctx_lo=4096, ctx_hi=131072, block_size=64,
                 H=64, D=128, topk=2048, seed=0, dtype=BF16,
                 context_lens=None) -> Paged:
    """Paged K cache in blocks of block_size tokens, block table permuted."""
    if context_lens is None:
        context_lens = decode_context_lens(B, ctx_lo, ctx_hi, seed)
    context_lens = np.asarray(context_lens, dtype=np.int32)
    B = context_lens.shape[0]
    rng = _rng(seed + 1)
    max_blocks = -(-ctx_hi // block_size)
    nblk = [-(-int(L) // block_size) for L in context_lens]
    total = int(sum(nblk))
    perm = rng.permutation(total).astype(np.int32)
    block_table = np.zeros((B, max_blocks), dtype=np.int32)
    pos = 0
    for b, n in enumerate(nblk):
        block_table[b, :n] = perm[pos:pos + n]
        pos += n
    std = 1.0 / math.sqrt(D)
    R = B * next_n
    w = _weights(rng, R, H, D)
    if dtype == BF16:
        q = _normal_bf16(rng, (R, H, D), std)
        kc = _normal_bf16(rng, (total * block_size, D), std).reshape(total, block_size, D)
        return Paged(f"paged_decode_B{B}x{next_n}_ctx{ctx_lo}-{ctx_hi}_blk{block_size}"
                     f"_H{H}_D{D}_k{topk}", BF16, q, w, kc, block_table,
                     context_lens, next_n, topk)
    qsrc = bf16_bits_to_f32(_normal_bf16(rng, (R * H, D), std))
    ksrc = bf16_bits_to_f32(_normal_bf16(rng, (total * block_size, D), std))
    q8, sq = quantize_e4m3_blocks(qsrc)
    k8, sk = quantize_e4m3_blocks(ksrc)
    w = (w * sq.reshape(R, H)).astype(np.float32)
    return Paged(f"paged_decode_fp8_B{B}x{next_n}_blk{block_size}_H{H}_D{D}_k{topk}",
                 E4M3, q8.reshape(R, H, D), w, k8.reshape(total, block_size, D),
                 block_table, context_lens, next_n, topk,
                 k_scale=sk.reshape(total, block_size))


WORKLOADS = {
    "tiny_causal": tiny_causal,
    "prefill_causal": prefill_causal,
    "prefill_thd": prefill_thd,
    "paged_decode": paged_decode,
    "prefill_fp8": prefill_fp8,
    "prefill_mxfp4": prefill_mxfp4,
}
