// dsa_score.cuh -- lightning-indexer scoring kernel for sm_103a.
//
// Computes  logit[t,s] = sum_h w[t,h] * max(0, q[t,h,:] . k[s,:])  (times the
// e4m3 key scale when the operands are fp8), the index score that
// KimiK3DSAIndexer.score hands to sparse_attn_indexer (vLLM API docs,
// "vllm.models.kimi_k3.nvidia.dsa"), and writes it for the columns of each
// row's range, -inf for the other columns of the key tiles it visits.
//
// Layout of the contraction: keys sit on the MMA M dimension (128 TMEM lanes
// = 128 keys of a tile) and a group of query tokens x heads on N (up to 256
// columns, e.g. 4 tokens x 64 heads).  Each epilogue thread therefore owns
// one key and reduces over the heads of its own TMEM lane in registers.
//
// Persistent CTAs (one per SM) walk a static list of work items -- a group of
// TOK query rows (prefill) or one chunk of one request's keys (paged decode)
// -- in snake order, so that the long causal groups spread evenly.  Roles:
//   warp 0      TMA producer: each group's q tile into one of two q buffers,
//               then its K tiles into an NST-deep ring of shared-memory stages
//               (prefill: 2-D boxes of [S, D]; paged: 3-D boxes of
//               [num_blocks, block_size, D] through the block table)
//   warp 1      TMEM allocator + single-thread tcgen05.mma issuer into one of
//               two TMEM accumulators
//   warps 2..   EPI_WG epilogue warpgroups, each owning EPI_COLS accumulator
//               columns (whole tokens): one batched tcgen05.ld per tile, ReLU,
//               head-weighted sum, key scale, range mask, store
//
// The head sum uses min(8, H) interleaved fp32 partial sums (head h goes to
// partial h % 8, each accumulated in ascending h) combined pairwise.  The
// order is fixed, so every entry point that scores the same inputs produces
// bit-identical logits.
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
  static constexpr int MINCOLS = H > 32 ? H : 32;
  static constexpr int EPI_WG = (N / MINCOLS) < 4 ? (N / MINCOLS) : 4;
  static constexpr int EPI_COLS = N / EPI_WG;       // accumulator columns per epilogue thread
  static constexpr int EPI_TOK = EPI_COLS / H;
  // Paged decode has few columns: up to four warpgroups form EPI_SETS
  // independent epilogue sets that take alternate tiles (tile i goes to set
  // i % EPI_SETS), with NBUF TMEM accumulators in flight.
  static constexpr int EPI_SETS = (kPaged && EPI_WG < 4) ? 4 / EPI_WG : 1;
  static constexpr int NBUF = 2 * EPI_SETS;
  static constexpr int EPI_THREADS = 128 * EPI_WG * EPI_SETS;
  static constexpr int NPART = H < 8 ? H : 8;       // partial sums of the head reduction
  static constexpr int THREADS = 64 + EPI_THREADS;
  static constexpr int Q_BYTES = ATOMS * N * 128;
  static constexpr int STAGE_BYTES = ATOMS * TILE * 128;
  // misc: w_s[N] | rs_s[TOK] | re_s[TOK] | paged block-table slices for the
  // producer and the epilogue (BT entries each) | 36 barriers | tmem slot + abort
  static constexpr int BT = kPaged ? 256 : 0;  // >= chunk keys / smallest block (2048 / 8)
  static constexpr int PFX = kPaged ? kMaxPagedRequests + 1 : 0;  // work-list prefix sums
  static constexpr int MISC_W = 0;
  static constexpr int MISC_RS = N * 4;
  static constexpr int MISC_RE = MISC_RS + TOK * 4;
  static constexpr int MISC_BTP = MISC_RE + TOK * 4;
  static constexpr int MISC_BTE = MISC_BTP + BT * 4;
  static constexpr int MISC_PFX = MISC_BTE + BT * 4;
  static constexpr int MISC_BARS = (MISC_PFX + PFX * 4 + 7) / 8 * 8;
  static constexpr int MISC_SLOT = MISC_BARS + 36 * 8;
  static constexpr int MISC_BYTES = (MISC_SLOT + 16 + 127) / 128 * 128;
  // One persistent CTA per SM with two q buffers (the next group's q tile
  // loads while the current group runs).
  static constexpr int QBUF = 2;
  static constexpr int SMEM_LIMIT = 232448;
  static constexpr int NST_FIT = (SMEM_LIMIT - 1024 - MISC_BYTES - QBUF * Q_BYTES) / STAGE_BYTES;
  static constexpr int NST = NST_FIT > 8 ? 8 : NST_FIT;
  static constexpr int SMEM = 1024 + QBUF * Q_BYTES + NST * STAGE_BYTES + MISC_BYTES;
  static constexpr uint32_t TMEM_COLS = static_cast<uint32_t>(NBUF * N);
  static constexpr uint32_t IDESC = mma_idesc(kFp8 ? 0u : 1u, TILE, N);

  static_assert(ROW_BYTES % 128 == 0, "a key row must be a whole number of swizzle atoms");
  static_assert(N % 16 == 0 && N >= 32 && N <= 256, "MMA N for M=128");
  static_assert(N % H == 0 && EPI_COLS % H == 0 && (EPI_COLS == 32 || EPI_COLS == 64 ||
                EPI_COLS == 128), "column split");
  static_assert(TMEM_COLS <= 512 && (TMEM_COLS & (TMEM_COLS - 1)) == 0, "TMEM allocation");
  static_assert(NST >= 2 && NST <= 8, "pipeline depth");
  static_assert(SMEM <= SMEM_LIMIT, "shared memory");
};

// One work item, as every role derives it.
struct ScoreGroup {
  int row0;      // first query row
  int ntok;      // valid query rows (<= TOK)
  int kt_begin;  // first key tile (prefill: absolute; paged: logical within the request)
  int kt_end;    // one past the last key tile; kt_end <= kt_begin means nothing to do
  int b;         // paged: request
  int L;         // paged: clamped context length
  bool bad_len;  // paged: context length was out of range
};

// Work item `slot`.  Must be called by all 32 lanes of a warp.  Paged decode:
// slot indexes the CTA's compacted list of non-empty (request, chunk) items,
// pfx[b] being the number of items of requests before b.
template <int TOK, bool kPaged>
__device__ __forceinline__ ScoreGroup score_group(const ScoreParams& p, int slot, int lane,
                                                  const int* pfx) {
  ScoreGroup g;
  g.bad_len = false;
  if constexpr (kPaged) {
    const int B = p.R / p.next_n;
    int lo_b = 0, hi_b = B;  // largest b with pfx[b] <= slot
    while (hi_b - lo_b > 1) {
      const int mid = (lo_b + hi_b) >> 1;
      if (pfx[mid] <= slot) lo_b = mid; else hi_b = mid;
    }
    g.b = lo_b;
    const int c = slot - pfx[lo_b];
    const int Lraw = p.context_lens[g.b];
    const int cap = p.max_blocks * p.block_size;
    g.L = Lraw < 0 ? 0 : (Lraw > cap ? cap : Lraw);
    const int lo = c * p.chunk_keys;
    const int hi = min(g.L, lo + p.chunk_keys);
    g.row0 = g.b * p.next_n;
    g.ntok = p.next_n;
    g.kt_begin = lo / 128;
    g.kt_end = hi > lo ? (hi + 127) / 128 : g.kt_begin;
  } else {
    const int G = (p.R + TOK - 1) / TOK;
    const int grp = G - 1 - slot;  // later causal groups carry more keys: start with them
    g.b = 0;
    g.L = 0;
    g.row0 = grp * TOK;
    g.ntok = min(TOK, p.R - g.row0);
    int lo = 0x7fffffff, hi = 0;
    for (int i = lane; i < g.ntok; i += 32) {
      const int a = min(max(p.row_starts[g.row0 + i], 0), p.S);
      const int e = min(max(p.row_ends[g.row0 + i], 0), p.S);
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
    g.kt_begin = hi > lo ? lo / 128 : 0;
    g.kt_end = hi > lo ? (hi + 127) / 128 : 0;
  }
  return g;
}

// ReLU of head h's dot product, as the epilogue takes it.  Some heads use
// max(x, 0) (ALU pipe), the others x + |x| = 2 max(x, 0) (one add on the FMA
// pipe) with their weight staged halved, so that both forms give the same
// products w * relu(x) bit for bit while the two pipes share the work: every
// fourth head takes the add form for bf16, every second for e4m3 (whose
// epilogue, with its weights in registers, leans harder on the ALU pipe).
template <bool kFp8>
__host__ __device__ constexpr bool relu_by_add(int h) {
  return kFp8 ? (h & 1) == 1 : (h & 3) == 3;
}

template <bool kFp8>
__device__ __forceinline__ float relu_term(int h, float x) {
  return relu_by_add<kFp8>(h) ? x + fabsf(x) : fmaxf(x, 0.f);
}

// Snake order over work items: round r visits CTAs 0..P-1 forward when r is
// even and backward when r is odd.
__device__ __forceinline__ int snake_slot(int r, int P, int cta) {
  return r * P + ((r & 1) ? (P - 1 - cta) : cta);
}

template <int COLS>
__device__ __forceinline__ void tmem_load_cols(uint32_t taddr, float (&v)[COLS]) {
  static_assert(COLS == 32 || COLS == 64 || COLS == 128, "tcgen05.ld width");
  if constexpr (COLS == 32) {
    tmem_load32(taddr, v);
  } else if constexpr (COLS == 64) {
    tmem_load64(taddr, v);
  } else {
    float* lo = v;
    float* hi = v + 64;
    tmem_load64(taddr, *reinterpret_cast<float(*)[64]>(lo));
    tmem_load64(taddr + 64, *reinterpret_cast<float(*)[64]>(hi));
  }
}

template <int H, int N, int D, bool kFp8, bool kPaged>
__global__ void __launch_bounds__(ScoreCfg<H, N, D, kFp8, kPaged>::THREADS, 1)
    score_kernel(const __grid_constant__ ScoreParams p) {
  using C = ScoreCfg<H, N, D, kFp8, kPaged>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* q_s = smem;                         // QBUF x Q_BYTES
  uint8_t* k_s = smem + C::QBUF * C::Q_BYTES;  // NST x STAGE_BYTES
  uint8_t* misc = k_s + C::NST * C::STAGE_BYTES;
  float* w_s = reinterpret_cast<float*>(misc + C::MISC_W);
  int* rs_s = reinterpret_cast<int*>(misc + C::MISC_RS);
  int* re_s = reinterpret_cast<int*>(misc + C::MISC_RE);
  uint64_t* bars = reinterpret_cast<uint64_t*>(misc + C::MISC_BARS);
  uint64_t* full = bars;         // [8]
  uint64_t* empty = bars + 8;    // [8]
  uint64_t* qfull = bars + 16;   // [2]
  uint64_t* qempty = bars + 18;  // [2]
  uint64_t* accf = bars + 20;    // [8]
  uint64_t* acce = bars + 28;    // [8]
  int* bt_p = reinterpret_cast<int*>(misc + C::MISC_BTP);  // producer's block-table slice
  int* bt_e = reinterpret_cast<int*>(misc + C::MISC_BTE);  // epilogue's block-table slice
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + C::MISC_SLOT);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(misc + C::MISC_SLOT + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int P = gridDim.x;
  const int cta = blockIdx.x;
  int* pfx = reinterpret_cast<int*>(misc + C::MISC_PFX);
  if constexpr (kPaged) {
    // The work list: every non-empty chunk of every request, request-major.
    // Each CTA derives it from the context lengths (no global state).
    if (warp == 0) {
      const int B = p.R / p.next_n;
      const int cap = p.max_blocks * p.block_size;
      int carry = 0;
      if (lane == 0) pfx[0] = 0;
      for (int base = 0; base < B; base += 32) {
        const int b = base + lane;
        int cnt = 0;
        if (b < B) {
          const int Lraw = p.context_lens[b];
          if ((Lraw < 0 || Lraw > cap) && cta == 0) record_error(p.err, kErrBadIndex);
          const int L = Lraw < 0 ? 0 : (Lraw > cap ? cap : Lraw);
          cnt = (L + p.chunk_keys - 1) / p.chunk_keys;
        }
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        if (b < B) pfx[b + 1] = carry + incl;
        carry += __shfl_sync(0xffffffffu, incl, 31);
      }
    }
    __syncthreads();
  }
  int nslots;
  if constexpr (kPaged) {
    nslots = pfx[p.R / p.next_n];
  } else {
    nslots = (p.R + C::TOK - 1) / C::TOK;
  }
  const int rounds = (nslots + P - 1) / P;

  // -------------------------------------------------------------------- setup
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&qfull[i], 1);
      mbar_init(&qempty[i], 1);
    }
    for (int i = 0; i < C::NBUF; ++i) {
      mbar_init(&accf[i], 1);
      mbar_init(&acce[i], 128 * C::EPI_WG);  // one epilogue set
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------- producer
    int kiter = 0, ngroups = 0, qissued = 0;
    bool ok = true;
    if (lane == 0) {
      tma_prefetch_desc(&p.tmap_q);
      tma_prefetch_desc(&p.tmap_k);
    }
    for (int r = 0; r < rounds && ok; ++r) {
      const int slot = snake_slot(r, P, cta);
      if (slot >= nslots) continue;
      const ScoreGroup g = score_group<C::TOK, kPaged>(p, slot, lane, pfx);
      if (g.kt_end <= g.kt_begin) continue;
      if constexpr (kPaged) {
        // The group's physical block ids, read once with coalesced loads
        // (validated: an id outside the cache is recorded and replaced by 0).
        const int bs = p.block_size;
        const int nblk = (g.L + bs - 1) / bs;
        const int lb0 = g.kt_begin * (C::TILE / bs);
        const int cnt = (g.kt_end - g.kt_begin) * (C::TILE / bs);
        __syncwarp();
        for (int i = lane; i < cnt; i += 32) {
          int lb = lb0 + i;
          if (lb > nblk - 1) lb = nblk - 1;
          int pb = p.block_table[static_cast<int64_t>(g.b) * p.max_blocks + lb];
          if (pb < 0 || pb >= p.num_blocks) {
            record_error(p.err, kErrBadIndex);
            pb = 0;
          }
          bt_p[i] = pb;
        }
        __syncwarp();
      }
      if (lane == 0) {
        const int qb = ngroups % C::QBUF;
        if (!mbar_wait_bounded(&qempty[qb], (static_cast<uint32_t>(ngroups / C::QBUF) & 1u) ^ 1u,
                               abort_flag)) {
          ok = false;
        } else {
          mbar_arrive_expect_tx(&qfull[qb], C::Q_BYTES);
#pragma unroll
          for (int a = 0; a < C::ATOMS; ++a)
            tma_load_2d(q_s + qb * C::Q_BYTES + a * N * 128, &p.tmap_q, &qfull[qb],
                        a * C::ATOM_ELEMS, g.row0 * H);
          ++qissued;
          for (int kt = g.kt_begin; kt < g.kt_end; ++kt) {
            const int stage = kiter % C::NST;
            const uint32_t phase = static_cast<uint32_t>(kiter / C::NST) & 1u;
            if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
            uint8_t* dst = k_s + stage * C::STAGE_BYTES;
            if constexpr (!kPaged) {
#pragma unroll
              for (int a = 0; a < C::ATOMS; ++a)
                tma_load_2d(dst + a * C::TILE * 128, &p.tmap_k, &full[stage],
                            a * C::ATOM_ELEMS, kt * C::TILE);
            } else {
              const int bs = p.block_size;
              const int per_tile = C::TILE / bs;
              for (int i = 0; i < per_tile; ++i) {
                const int pb = bt_p[(kt - g.kt_begin) * per_tile + i];
#pragma unroll
                for (int a = 0; a < C::ATOMS; ++a)
                  tma_load_3d(dst + a * C::TILE * 128 + i * bs * 128, &p.tmap_k, &full[stage],
                              a * C::ATOM_ELEMS, 0, pb);
              }
            }
            ++kiter;
          }
        }
        ++ngroups;
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    }
    if (lane == 0 && !ok) {
      *abort_flag = 1;
      record_error(p.err, kErrTimeout);
      // Let the copies already in flight land before the CTA retires.
      const int first = kiter > C::NST ? kiter - C::NST : 0;
      for (int i = first; i < kiter; ++i)
        mbar_wait_bounded(&full[i % C::NST], static_cast<uint32_t>(i / C::NST) & 1u, nullptr,
                          100000000ull);
      for (int j = qissued > C::QBUF ? qissued - C::QBUF : 0; j < qissued; ++j)
        mbar_wait_bounded(&qfull[j % C::QBUF], static_cast<uint32_t>(j / C::QBUF) & 1u, nullptr,
                          100000000ull);
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issuer
    int kiter = 0, ngroups = 0, tcount = 0;
    bool ok = true;
    for (int r = 0; r < rounds && ok; ++r) {
      const int slot = snake_slot(r, P, cta);
      if (slot >= nslots) continue;
      const ScoreGroup g = score_group<C::TOK, kPaged>(p, slot, lane, pfx);
      if (g.kt_end <= g.kt_begin) continue;
      if (lane == 0) {
        const int qb = ngroups % C::QBUF;
        ok = mbar_wait_bounded(&qfull[qb], static_cast<uint32_t>(ngroups / C::QBUF) & 1u,
                               abort_flag);
        const uint32_t q_addr = smem_u32(q_s + qb * C::Q_BYTES);
        for (int kt = g.kt_begin; ok && kt < g.kt_end; ++kt) {
          const int stage = kiter % C::NST;
          const uint32_t phase = static_cast<uint32_t>(kiter / C::NST) & 1u;
          const int buf = tcount % C::NBUF;
          const uint32_t aphase = static_cast<uint32_t>(tcount / C::NBUF) & 1u;
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
            const uint64_t adesc =
                sw128_kmajor_desc(k_addr + atom * C::TILE * 128 + within * 32);
            const uint64_t bdesc = sw128_kmajor_desc(q_addr + atom * N * 128 + within * 32);
            mma_ss<kFp8>(d_tmem, adesc, bdesc, C::IDESC, ks > 0 ? 1u : 0u);
          }
          mma_commit(&empty[stage]);
          mma_commit(&accf[buf]);
          ++kiter;
          ++tcount;
        }
        if (ok) mma_commit(&qempty[qb]);  // q buffer free once this group's MMAs are done
        ++ngroups;
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    }
    if (lane == 0 && !ok) {
      *abort_flag = 1;
      record_error(p.err, kErrTimeout);
      if (tcount > 0) {
        // The last commit covers every MMA issued before it.
        const int last = tcount - 1;
        mbar_wait_bounded(&accf[last % C::NBUF], static_cast<uint32_t>(last / C::NBUF) & 1u,
                          nullptr, 100000000ull);
      }
    }
  } else {
    // ------------------------------------------------------------- epilogue
    const int ew = warp - 2;
    const int set = ew / (4 * C::EPI_WG);  // tiles i with i % EPI_SETS == set
    const int wg = (ew >> 2) % C::EPI_WG;  // column group of this warpgroup
    const int quarter = warp & 3;  // the TMEM lane quarter this warp may access
    const int key_in_tile = quarter * 32 + lane;
    // 64 heads, one token per warpgroup (prefill and paged, bf16 and e4m3):
    // the accumulator is read in the 16x256b shape: each thread sums 16
    // heads of 4 keys, a quad of threads shares those keys, and after the
    // exchange each thread owns one of them.
    constexpr bool kQuad = H == 64 && C::EPI_COLS == 64;
    const int my_key = kQuad ? quarter * 32 + (lane >> 2) + 8 * (lane & 3) : key_in_tile;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const int etid = threadIdx.x - 64;  // 0 .. EPI_THREADS-1
    int tcount = 0;
    bool ok = true;
    // No early exit from this loop: every epilogue warp must reach the same
    // named barriers.  After an abort the tile waits fail at once instead.
    for (int r = 0; r < rounds; ++r) {
      const int slot = snake_slot(r, P, cta);
      if (slot >= nslots) continue;
      const ScoreGroup g = score_group<C::TOK, kPaged>(p, slot, lane, pfx);
      if (g.kt_end <= g.kt_begin) continue;
      // Stage this group's weights and row ranges (every epilogue thread has
      // finished the previous group when the named barrier opens).
      asm volatile("bar.sync 1, %0;" ::"r"(C::EPI_THREADS) : "memory");
      for (int i = etid; i < N; i += C::EPI_THREADS) {
        const int tok = i / H, h = i % H;
        float wv = 0.f;
        if (tok < g.ntok) {
          const int64_t row = g.row0 + tok;
          wv = p.weights[row * H + h];
          if (p.q_scale) wv *= p.q_scale[row * H + h];
        }
        // Heads that take their ReLU as x + |x| (= 2 relu(x)) get a halved
        // weight: (w/2)(x + |x|) = w relu(x) exactly.
        w_s[i] = (kQuad || relu_by_add<kFp8>(h)) ? 0.5f * wv : wv;
      }
      if constexpr (kPaged && kFp8) {
        const int bs = p.block_size;
        const int nblk = (g.L + bs - 1) / bs;
        const int lb0 = g.kt_begin * (C::TILE / bs);
        const int cnt = (g.kt_end - g.kt_begin) * (C::TILE / bs);
        for (int i = etid; i < cnt; i += C::EPI_THREADS) {
          int lb = lb0 + i;
          if (lb > nblk - 1) lb = nblk - 1;
          int pb = p.block_table[static_cast<int64_t>(g.b) * p.max_blocks + lb];
          if (pb < 0 || pb >= p.num_blocks) pb = 0;
          bt_e[i] = pb;
        }
      }
      for (int i = etid; i < C::TOK; i += C::EPI_THREADS) {
        int lo = 0, hi = 0;
        if (i < g.ntok) {
          if constexpr (kPaged) {
            const int end = g.L - p.next_n + i + 1;
            hi = end < 0 ? 0 : end;
          } else {
            lo = min(max(p.row_starts[g.row0 + i], 0), p.S);
            hi = min(max(p.row_ends[g.row0 + i], 0), p.S);
            if (hi < lo) hi = lo;
          }
        }
        rs_s[i] = lo;
        re_s[i] = hi;
      }
      asm volatile("bar.sync 1, %0;" ::"r"(C::EPI_THREADS) : "memory");
      // This thread's row ranges, kept in registers for the whole group.
      int rlo[C::EPI_TOK], rhi[C::EPI_TOK];
#pragma unroll
      for (int j = 0; j < C::EPI_TOK; ++j) {
        rlo[j] = rs_s[wg * C::EPI_TOK + j];
        rhi[j] = re_s[wg * C::EPI_TOK + j];
      }
      // e4m3, H >= 16: this thread's EPI_COLS weights live in registers for
      // the whole group, and the accumulator is read 8 columns at a time, so
      // that the epilogue leaves shared-memory bandwidth to the MMA operand
      // reads (an e4m3 tile takes half the MMA time of a bf16 one).
      constexpr bool kRegW = kFp8 && H >= 16 && C::NPART == 8 && !kQuad;
      // kQuad: this thread's 16 heads 8b + 2(lane%4) + {0,1}, b = 0..7, as pairs.
      float2 wq[kQuad ? 8 : 1];
      if constexpr (kQuad) {
#pragma unroll
        for (int b = 0; b < 8; ++b)
          wq[b] = *reinterpret_cast<const float2*>(w_s + wg * C::EPI_COLS + 8 * b + 2 * (lane & 3));
      }
      float wr[kRegW ? C::EPI_COLS : 1];
      if constexpr (kRegW) {
#pragma unroll
        for (int i = 0; i < C::EPI_COLS / 4; ++i) {
          const float4 w4 = reinterpret_cast<const float4*>(w_s + wg * C::EPI_COLS)[i];
          wr[4 * i] = w4.x;
          wr[4 * i + 1] = w4.y;
          wr[4 * i + 2] = w4.z;
          wr[4 * i + 3] = w4.w;
        }
      }

      // fp8: this thread's key scale, loaded one tile ahead of its use.
      auto key_scale = [&](int kt) -> float {
        const int s = kt * C::TILE + my_key;
        if constexpr (kPaged) {
          const int bs = p.block_size;
          const int nblk = (g.L + bs - 1) / bs;
          int lb = s / bs;
          if (lb > nblk - 1) lb = nblk - 1;
          const int pb = bt_e[lb - g.kt_begin * (C::TILE / bs)];
          return p.k_scale[static_cast<int64_t>(pb) * bs + (s % bs)];
        } else {
          return s < p.S ? p.k_scale[s] : 0.f;
        }
      };
      // This set's first tile of the group (tiles alternate between sets);
      // tcount keeps counting every tile of the CTA.
      const int skip = ((set - tcount) % C::EPI_SETS + C::EPI_SETS) % C::EPI_SETS;
      const int kt0 = g.kt_begin + skip;
      const int ntile = g.kt_end - g.kt_begin;
      float ks_next = 1.f;
      if constexpr (kFp8) {
        if (kt0 < g.kt_end) ks_next = key_scale(kt0);
      }
      int tc = tcount + skip;
      tcount += ntile;
      for (int kt = kt0; ok && kt < g.kt_end; kt += C::EPI_SETS, tc += C::EPI_SETS) {
        const int buf = tc % C::NBUF;
        const uint32_t aphase = static_cast<uint32_t>(tc / C::NBUF) & 1u;
        // Warp-uniform outcome: tcgen05.ld below needs every lane.
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&accf[buf], aphase, abort_flag) ? 1 : 0);
        if (!ok) break;
        tc_fence_after_sync();
        const uint32_t tcol =
            tmem_base + lane_addr + static_cast<uint32_t>(buf * N + wg * C::EPI_COLS);
        const int s = kt * C::TILE + my_key;
        const float kscale = ks_next;
        if constexpr (kFp8) {
          if (kt + C::EPI_SETS < g.kt_end) ks_next = key_scale(kt + C::EPI_SETS);
        }
        const bool col_ok = s < p.S;
        if constexpr (kQuad) {
          // Four chunks, each one 16x256b.x4 load (16 lanes x 32 columns:
          // lanes +16(c & 1), heads 32(c >> 1) ..); the next chunk's load is
          // in flight while this one is summed.  Per key the heads still
          // alternate between two accumulators in ascending 8-head blocks.
          // ReLU as x + |x| (one packed add, the weights staged halved).
          const uint32_t cb = tmem_base + static_cast<uint32_t>(buf * N + wg * C::EPI_COLS);
          const uint32_t l0 = static_cast<uint32_t>(quarter * 32) << 16;
          const uint32_t l1 = static_cast<uint32_t>(quarter * 32 + 16) << 16;
          float2 acc4[4], acc4b[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) acc4[i] = acc4b[i] = make_float2(0.f, 0.f);
          uint32_t cur[16], nxt[16];
          tmem_ld16x256_x4_async(cb + l0, cur);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            tmem_wait_ld16(cur);
            if (c == 3) {
              // Every column of this tile is in registers: release it.
              tc_fence_before_sync();
              mbar_arrive(&acce[buf]);
            } else {
              const int cn = c + 1;
              tmem_ld16x256_x4_async(
                  cb + ((cn & 1) ? l1 : l0) + static_cast<uint32_t>(32 * (cn >> 1)), nxt);
            }
            {
              const int hf = c & 1;
#pragma unroll
              for (int jj = 0; jj < 4; ++jj) {
                const int rep = jj & 1;
                const int r0 = 4 * jj;
                const float2 w2 = wq[4 * (c >> 1) + jj];
                const float2 xa = make_float2(__uint_as_float(cur[r0]), __uint_as_float(cur[r0 + 1]));
                const float2 xb =
                    make_float2(__uint_as_float(cur[r0 + 2]), __uint_as_float(cur[r0 + 3]));
                const float2 ya = __fadd2_rn(xa, make_float2(fabsf(xa.x), fabsf(xa.y)));
                const float2 yb = __fadd2_rn(xb, make_float2(fabsf(xb.x), fabsf(xb.y)));
                if (rep == 0) {
                  acc4[2 * hf] = __ffma2_rn(w2, ya, acc4[2 * hf]);
                  acc4[2 * hf + 1] = __ffma2_rn(w2, yb, acc4[2 * hf + 1]);
                } else {
                  acc4b[2 * hf] = __ffma2_rn(w2, ya, acc4b[2 * hf]);
                  acc4b[2 * hf + 1] = __ffma2_rn(w2, yb, acc4b[2 * hf + 1]);
                }
              }
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) cur[i] = nxt[i];
          }
          // This thread's 16-head sums of keys +0, +8, +16, +24 (from lane/4);
          // the quad exchanges halves twice and thread m keeps key +8m.
          float tot[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 t2 = __fadd2_rn(acc4[i], acc4b[i]);
            tot[i] = t2.x + t2.y;
          }
          const bool b0 = (lane & 1) != 0, b1 = (lane & 2) != 0;
          float k0 = b0 ? tot[1] : tot[0], k1 = b0 ? tot[3] : tot[2];
          const float s0 = b0 ? tot[0] : tot[1], s1 = b0 ? tot[2] : tot[3];
          k0 += __shfl_xor_sync(0xffffffffu, s0, 1);
          k1 += __shfl_xor_sync(0xffffffffu, s1, 1);
          float acc = b1 ? k1 : k0;
          acc += __shfl_xor_sync(0xffffffffu, b1 ? k0 : k1, 2);
          acc *= kscale;
          const int tok = wg;
          if (tok < g.ntok && col_ok) {
            const float val = (s >= rlo[0] && s < rhi[0]) ? acc : -INFINITY;
            p.logits[static_cast<int64_t>(g.row0 + tok) * p.ld + s] = val;
          }
          continue;
        }
        if constexpr (kRegW) {
#pragma unroll
          for (int j = 0; j < C::EPI_TOK; ++j) {
            const int tok = wg * C::EPI_TOK + j;
            // Heads in pairs: one packed FMA per pair, partial h % 8 taking its
            // heads in ascending order (the same sums as the path below).
            float2 part2[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) part2[i] = make_float2(0.f, 0.f);
#pragma unroll
            for (int c = 0; c < H / 8; ++c) {
              float v[8];
              tmem_load8(tcol + static_cast<uint32_t>(j * H + c * 8), v);
              if (j == C::EPI_TOK - 1 && c == H / 8 - 1) {
                // Every column of this tile is in registers: release it.
                tc_fence_before_sync();
                mbar_arrive(&acce[buf]);
              }
#pragma unroll
              for (int hh = 0; hh < 8; hh += 2) {
                const int h = c * 8 + hh;
                const float2 y2 =
                    make_float2(relu_term<kFp8>(h, v[hh]), relu_term<kFp8>(h + 1, v[hh + 1]));
                const float2 w2 = make_float2(wr[j * H + h], wr[j * H + h + 1]);
                part2[(h % 8) / 2] = __ffma2_rn(w2, y2, part2[(h % 8) / 2]);
              }
            }
            float part[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              part[2 * i] = part2[i].x;
              part[2 * i + 1] = part2[i].y;
            }
#pragma unroll
            for (int w = 4; w > 0; w >>= 1) {
#pragma unroll
              for (int i = 0; i < w; ++i) part[i] = part[i] + part[i + w];
            }
            float acc = part[0];
            if constexpr (kFp8) acc *= kscale;
            if (tok < g.ntok && col_ok) {
              const float val = (s >= rlo[j] && s < rhi[j]) ? acc : -INFINITY;
              p.logits[static_cast<int64_t>(g.row0 + tok) * p.ld + s] = val;
            }
          }
          continue;
        }
        float v[C::EPI_COLS];
        tmem_load_cols<C::EPI_COLS>(tcol, v);
        tc_fence_before_sync();
        mbar_arrive(&acce[buf]);
#pragma unroll
        for (int j = 0; j < C::EPI_TOK; ++j) {
          const int tok = wg * C::EPI_TOK + j;
          const float* wt = w_s + tok * H;
          float part[C::NPART];
#pragma unroll
          for (int i = 0; i < C::NPART; ++i) part[i] = 0.f;
          if constexpr (C::NPART == 8) {
            // Heads in pairs: one packed FMA per pair, same partials and order.
            // Weights come four at a time (one 16-byte shared load), which
            // halves the epilogue's share of the shared-memory bandwidth the
            // MMAs read their operands through.
            float2 part2[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) part2[i] = make_float2(0.f, 0.f);
#pragma unroll
            for (int h = 0; h < H; h += 4) {
              const float4 w4 = *reinterpret_cast<const float4*>(wt + h);
              const float2 y2a = make_float2(relu_term<kFp8>(h, v[j * H + h]),
                                             relu_term<kFp8>(h + 1, v[j * H + h + 1]));
              const float2 y2b = make_float2(relu_term<kFp8>(h + 2, v[j * H + h + 2]),
                                             relu_term<kFp8>(h + 3, v[j * H + h + 3]));
              part2[(h % 8) / 2] = __ffma2_rn(make_float2(w4.x, w4.y), y2a, part2[(h % 8) / 2]);
              part2[(h % 8) / 2 + 1] =
                  __ffma2_rn(make_float2(w4.z, w4.w), y2b, part2[(h % 8) / 2 + 1]);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              part[2 * i] = part2[i].x;
              part[2 * i + 1] = part2[i].y;
            }
          } else {
#pragma unroll
            for (int h = 0; h < H; ++h)
              part[h % C::NPART] =
                  fmaf(wt[h], relu_term<kFp8>(h, v[j * H + h]), part[h % C::NPART]);
          }
#pragma unroll
          for (int w = C::NPART / 2; w > 0; w >>= 1) {
#pragma unroll
            for (int i = 0; i < w; ++i) part[i] = part[i] + part[i + w];
          }
          float acc = part[0];
          if constexpr (kFp8) acc *= kscale;
          if (tok < g.ntok && col_ok) {
            const float val = (s >= rlo[j] && s < rhi[j]) ? acc : -INFINITY;
            p.logits[static_cast<int64_t>(g.row0 + tok) * p.ld + s] = val;
          }
        }
      }
    }
    if (!ok) {
      *abort_flag = 1;
      record_error(p.err, kErrTimeout);
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

int device_sm_count();

// Persistent CTAs: one per SM, at most one per work item (paged decode: the
// number of (request, chunk) slots bounds the non-empty items).
template <int H, int N, int D, bool kFp8, bool kPaged>
cudaError_t launch_score_instance(const ScoreParams& p, int work_items, cudaStream_t st) {
  using C = ScoreCfg<H, N, D, kFp8, kPaged>;
  auto kern = score_kernel<H, N, D, kFp8, kPaged>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  if (work_items <= 0) return cudaSuccess;
  const int sms = device_sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const int grid = work_items < sms ? work_items : sms;
  kern<<<grid, C::THREADS, C::SMEM, st>>>(p);
  return cudaGetLastError();
}

}  // namespace dsa
