// dsa_score.cuh -- lightning-indexer scoring kernel for sm_103a.
//
// Computes  logit[t,s] = sum_h w[t,h] * max(0, q[t,h,:] . k[s,:])  (times the
// e4m3 key scale when the operands are fp8), the index score that
// KimiK3DSAIndexer.score hands to sparse_attn_indexer (vLLM API docs,
// "vllm.models.kimi_k3.nvidia.dsa"), and writes it for the columns of each
// row's range, -inf for the other columns of the key tiles it visits.
//
// Layout of the contraction: keys sit on the MMA M dimension (128 TMEM lanes
// = 128 keys of a tile) and the group's query tokens x heads on N (up to 256
// columns, e.g. 4 tokens x 64 heads).  Each epilogue thread therefore owns
// one key and reduces over the heads of its own TMEM lane in registers.
//
// CTA roles (one CTA per SM; 192 or 320 threads):
//   warp 0      TMA producer: the group's q tile once, then K tiles into an
//               NST-deep ring of shared-memory stages (prefill: 2-D boxes of
//               the [S, D] key matrix; paged: 3-D boxes of
//               [num_blocks, block_size, D] through the block table)
//   warp 1      TMEM allocator + single-thread tcgen05.mma issuer into one of
//               two TMEM accumulators (double buffer)
//   warps 2..   epilogue: tcgen05.ld of the accumulator, ReLU, head-weighted
//               sum in ascending head order, key scale, range mask, store
#pragma once

#include "dsa_common.cuh"
#include "dsa_internal.h"

namespace dsa {

template <int H, int N, int D, bool kFp8, bool kPaged>
struct ScoreCfg {
  static constexpr int ESZ = kFp8 ? 1 : 2;
  static constexpr int ROW_BYTES = D * ESZ;
  static constexpr int ATOMS = ROW_BYTES / 128;     // 128-byte swizzle atoms along K
  static constexpr int ATOM_ELEMS = 128 / ESZ;
  static constexpr int KSTEPS = ROW_BYTES / 32;     // one MMA consumes 32 bytes of K
  static constexpr int TILE = 128;                  // keys per tile = MMA M
  static constexpr int TOK = N / H;                 // query rows per group
  static constexpr int EPI_WG = (N / 2 >= H) ? 2 : 1;
  static constexpr int EPI_COLS = N / EPI_WG;       // accumulator columns per epilogue thread
  static constexpr int EPI_TOK = EPI_COLS / H;
  static constexpr int THREADS = 64 + 128 * EPI_WG;
  static constexpr int Q_BYTES = ATOMS * N * 128;
  static constexpr int STAGE_BYTES = ATOMS * TILE * 128;
  static constexpr int MISC_BYTES = 4096;
  static constexpr int SMEM_LIMIT = 232448;
  static constexpr int NST_FIT = (SMEM_LIMIT - 1024 - MISC_BYTES - Q_BYTES) / STAGE_BYTES;
  static constexpr int NST = NST_FIT > 8 ? 8 : NST_FIT;
  static constexpr int SMEM = 1024 + Q_BYTES + NST * STAGE_BYTES + MISC_BYTES;
  static constexpr uint32_t TMEM_COLS = 2u * N;
  static constexpr uint32_t IDESC = mma_idesc(kFp8 ? 0u : 1u, TILE, N);

  static_assert(ROW_BYTES % 128 == 0, "a key row must be a whole number of swizzle atoms");
  static_assert(N % 16 == 0 && N >= 32 && N <= 256, "MMA N for M=128");
  static_assert(N % H == 0 && EPI_COLS % H == 0 && EPI_COLS % 32 == 0, "column split");
  static_assert(TMEM_COLS <= 512 && (TMEM_COLS & (TMEM_COLS - 1)) == 0, "TMEM allocation");
  static_assert(NST >= 2 && NST <= 8, "pipeline depth");
  static_assert(SMEM <= SMEM_LIMIT, "shared memory");
};

// Shared-memory carve-up of the MISC region.
struct ScoreMisc {
  static constexpr int W = 0;           // float w_s[N]      (<= 1024 B)
  static constexpr int RS = 1024;       // int rs_s[TOK]     (<= 1024 B)
  static constexpr int RE = 2048;       // int re_s[TOK]     (<= 1024 B)
  static constexpr int BARS = 3072;     // full[8], empty[8], qfull, accf[2], acce[2]
  static constexpr int TMEM_SLOT = 3072 + 256;
  static constexpr int INFO = 3072 + 272;   // int[4]: kt_begin, kt_end
  static constexpr int ABORT = 3072 + 304;  // uint32 abort flag
};

template <int H, int N, int D, bool kFp8, bool kPaged>
__global__ void __launch_bounds__(ScoreCfg<H, N, D, kFp8, kPaged>::THREADS, 1)
    score_kernel(const __grid_constant__ ScoreParams p) {
  using C = ScoreCfg<H, N, D, kFp8, kPaged>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* q_s = smem;
  uint8_t* k_s = smem + C::Q_BYTES;
  uint8_t* misc = k_s + C::NST * C::STAGE_BYTES;
  float* w_s = reinterpret_cast<float*>(misc + ScoreMisc::W);
  int* rs_s = reinterpret_cast<int*>(misc + ScoreMisc::RS);
  int* re_s = reinterpret_cast<int*>(misc + ScoreMisc::RE);
  uint64_t* bars = reinterpret_cast<uint64_t*>(misc + ScoreMisc::BARS);
  uint64_t* full = bars;
  uint64_t* empty = bars + 8;
  uint64_t* qfull = bars + 16;
  uint64_t* accf = bars + 17;
  uint64_t* acce = bars + 19;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + ScoreMisc::TMEM_SLOT);
  int* info = reinterpret_cast<int*>(misc + ScoreMisc::INFO);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(misc + ScoreMisc::ABORT);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---------------------------------------------------------------- work item
  int row0, ntok, b = 0, L = 0, key_lo = 0, key_hi = 0;
  if constexpr (kPaged) {
    b = blockIdx.x / p.chunks_per_req;
    const int c = blockIdx.x % p.chunks_per_req;
    const int Lraw = p.context_lens[b];
    const int cap = p.max_blocks * p.block_size;
    L = Lraw < 0 ? 0 : (Lraw > cap ? cap : Lraw);
    key_lo = c * p.chunk_keys;
    key_hi = min(L, key_lo + p.chunk_keys);
    if (c == 0 && threadIdx.x == 0 && (Lraw < 0 || Lraw > cap)) record_error(p.err, kErrBadIndex);
    if (key_lo >= key_hi) return;  // whole CTA, before any barrier or TMEM use
    row0 = b * p.next_n;
    ntok = p.next_n;
  } else {
    const int g = static_cast<int>(gridDim.x) - 1 - static_cast<int>(blockIdx.x);
    row0 = g * C::TOK;
    ntok = min(C::TOK, p.R - row0);
  }

  // -------------------------------------------------------------------- setup
  for (int i = threadIdx.x; i < N; i += C::THREADS) {
    const int tok = i / H, h = i % H;
    float wv = 0.f;
    if (tok < ntok) {
      const int64_t r = row0 + tok;
      wv = p.weights[r * H + h];
      if (p.q_scale) wv *= p.q_scale[r * H + h];
    }
    w_s[i] = wv;
  }
  for (int i = threadIdx.x; i < C::TOK; i += C::THREADS) {
    int lo = 0, hi = 0;
    if (i < ntok) {
      if constexpr (kPaged) {
        const int end = L - p.next_n + i + 1;
        hi = end < 0 ? 0 : end;
      } else {
        lo = min(max(p.row_starts[row0 + i], 0), p.S);
        hi = min(max(p.row_ends[row0 + i], 0), p.S);
        if (hi < lo) hi = lo;
      }
    }
    rs_s[i] = lo;
    re_s[i] = hi;
  }
  if (warp == 0) {
    // Union of the group's key ranges -> tile range.
    int lo = 0x7fffffff, hi = 0;
    if constexpr (kPaged) {
      lo = key_lo;
      hi = key_hi;
    } else {
      for (int i = lane; i < ntok; i += 32) {
        const int a = min(max(p.row_starts[row0 + i], 0), p.S);
        const int e = min(max(p.row_ends[row0 + i], 0), p.S);
        if (e > a) {
          lo = min(lo, a);
          hi = max(hi, e);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
        hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
      }
    }
    if (lane == 0) {
      if (hi > lo) {
        info[0] = lo / C::TILE;
        info[1] = (hi + C::TILE - 1) / C::TILE;
      } else {
        info[0] = 0;
        info[1] = 0;
      }
      for (int s = 0; s < C::NST; ++s) {
        mbar_init(&full[s], 1);
        mbar_init(&empty[s], 1);
      }
      mbar_init(qfull, 1);
      for (int i = 0; i < 2; ++i) {
        mbar_init(&accf[i], 1);
        mbar_init(&acce[i], 128 * C::EPI_WG);
      }
      *abort_flag = 0;
      fence_barrier_init();
    }
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  const int kt_begin = info[0], kt_end = info[1];

  // -------------------------------------------------------------------- roles
  if (warp == 0) {
    if (lane == 0 && kt_end > kt_begin) {
      tma_prefetch_desc(&p.tmap_q);
      tma_prefetch_desc(&p.tmap_k);
      mbar_arrive_expect_tx(qfull, C::Q_BYTES);
#pragma unroll
      for (int a = 0; a < C::ATOMS; ++a)
        tma_load_2d(q_s + a * N * 128, &p.tmap_q, qfull, a * C::ATOM_ELEMS, row0 * H);
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      for (int kt = kt_begin; kt < kt_end; ++kt) {
        if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
        uint8_t* dst = k_s + stage * C::STAGE_BYTES;
        if constexpr (!kPaged) {
#pragma unroll
          for (int a = 0; a < C::ATOMS; ++a)
            tma_load_2d(dst + a * C::TILE * 128, &p.tmap_k, &full[stage], a * C::ATOM_ELEMS,
                        kt * C::TILE);
        } else {
          const int bs = p.block_size;
          const int nblk = (L + bs - 1) / bs;
          const int per_tile = C::TILE / bs;
          for (int i = 0; i < per_tile; ++i) {
            int lb = kt * per_tile + i;
            if (lb > nblk - 1) lb = nblk - 1;
            int pb = p.block_table[static_cast<int64_t>(b) * p.max_blocks + lb];
            if (pb < 0 || pb >= p.num_blocks) {
              record_error(p.err, kErrBadIndex);
              pb = 0;
            }
#pragma unroll
            for (int a = 0; a < C::ATOMS; ++a)
              tma_load_3d(dst + a * C::TILE * 128 + i * bs * 128, &p.tmap_k, &full[stage],
                          a * C::ATOM_ELEMS, 0, pb);
          }
        }
        ++issued;
        if (++stage == C::NST) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) {
        *abort_flag = 1;
        record_error(p.err, kErrTimeout);
        // Let the copies already in flight land before the CTA retires.
        mbar_wait_bounded(qfull, 0, nullptr, 100000000ull);
        const int first = issued > C::NST ? issued - C::NST : 0;
        for (int i = first; i < issued; ++i)
          mbar_wait_bounded(&full[i % C::NST], (i / C::NST) & 1u, nullptr, 100000000ull);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && kt_end > kt_begin) {
      bool ok = mbar_wait_bounded(qfull, 0, abort_flag);
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      const uint32_t q_addr = smem_u32(q_s);
      for (int kt = kt_begin; ok && kt < kt_end; ++kt) {
        const int it = kt - kt_begin;
        const int buf = it & 1;
        const uint32_t aphase = static_cast<uint32_t>(it >> 1) & 1u;
        if (!mbar_wait_bounded(&acce[buf], aphase ^ 1u, abort_flag) ||
            !mbar_wait_bounded(&full[stage], phase, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * N);
        const uint32_t k_addr = smem_u32(k_s + stage * C::STAGE_BYTES);
#pragma unroll
        for (int ks = 0; ks < C::KSTEPS; ++ks) {
          const int atom = ks / 4, within = ks % 4;
          const uint64_t adesc = sw128_kmajor_desc(k_addr + atom * C::TILE * 128 + within * 32);
          const uint64_t bdesc = sw128_kmajor_desc(q_addr + atom * N * 128 + within * 32);
          mma_ss<kFp8>(d_tmem, adesc, bdesc, C::IDESC, ks > 0 ? 1u : 0u);
        }
        mma_commit(&empty[stage]);
        mma_commit(&accf[buf]);
        ++issued;
        if (++stage == C::NST) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) {
        *abort_flag = 1;
        record_error(p.err, kErrTimeout);
        if (issued > 0) {
          // The last commit covers every MMA issued before it.
          const int last = issued - 1;
          mbar_wait_bounded(&accf[last & 1], static_cast<uint32_t>(last >> 1) & 1u, nullptr,
                            100000000ull);
        }
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int ew = warp - 2;
    const int wg = ew >> 2;       // which column half
    const int quarter = warp & 3;  // the TMEM lane quarter this warp may access
    const int key_in_tile = quarter * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    for (int kt = kt_begin; kt < kt_end; ++kt) {
      const int it = kt - kt_begin;
      const int buf = it & 1;
      const uint32_t aphase = static_cast<uint32_t>(it >> 1) & 1u;
      if (!mbar_wait_bounded(&accf[buf], aphase, abort_flag)) {
        *abort_flag = 1;
        record_error(p.err, kErrTimeout);
        break;
      }
      tc_fence_after_sync();
      float v[C::EPI_COLS];
#pragma unroll
      for (int c = 0; c < C::EPI_COLS; c += 32) {
        float chunk[32];
        tmem_load32(tmem_base + lane_addr + static_cast<uint32_t>(buf * N + wg * C::EPI_COLS + c),
                    chunk);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[c + i] = chunk[i];
      }
      tc_fence_before_sync();
      mbar_arrive(&acce[buf]);

      const int s = kt * C::TILE + key_in_tile;
      float kscale = 1.f;
      if constexpr (kFp8) {
        if constexpr (kPaged) {
          const int bs = p.block_size;
          const int nblk = (L + bs - 1) / bs;
          int lb = s / bs;
          if (lb > nblk - 1) lb = nblk - 1;
          int pb = p.block_table[static_cast<int64_t>(b) * p.max_blocks + lb];
          if (pb < 0 || pb >= p.num_blocks) pb = 0;
          kscale = p.k_scale[static_cast<int64_t>(pb) * bs + (s % bs)];
        } else {
          kscale = s < p.S ? p.k_scale[s] : 0.f;
        }
      }
      const bool col_ok = s < p.S;
#pragma unroll
      for (int j = 0; j < C::EPI_TOK; ++j) {
        const int tok = wg * C::EPI_TOK + j;
        const float* wt = w_s + tok * H;
        float acc = 0.f;
#pragma unroll
        for (int h = 0; h < H; ++h) acc = fmaf(wt[h], fmaxf(v[j * H + h], 0.f), acc);
        if constexpr (kFp8) acc *= kscale;
        if (tok < ntok && col_ok) {
          const float val = (s >= rs_s[tok] && s < re_s[tok]) ? acc : -INFINITY;
          p.logits[static_cast<int64_t>(row0 + tok) * p.ld + s] = val;
        }
      }
    }
  }

  // ------------------------------------------------------------------ teardown
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

template <int H, int N, int D, bool kFp8, bool kPaged>
cudaError_t launch_score_instance(const ScoreParams& p, int grid, cudaStream_t st) {
  using C = ScoreCfg<H, N, D, kFp8, kPaged>;
  auto kern = score_kernel<H, N, D, kFp8, kPaged>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  if (grid <= 0) return cudaSuccess;
  kern<<<grid, C::THREADS, C::SMEM, st>>>(p);
  return cudaGetLastError();
}

}  // namespace dsa
