// dsa_score_mx.cuh -- lightning-indexer scoring with MXFP4 queries and keys
// (sm_103a, tcgen05.mma kind::mxf4 with block scales).
//
// The vLLM page ("vllm.models.kimi_k3.nvidia.dsa") scores MXFP4 keys against
// MXFP4 queries on request (KimiK3DSAIndexer.__init__: use_fp4_cache;
// KimiK3DSAIndexer.score: mxfp4_q_quant returns the queries, their block
// scales and the weights).  Elements are OCP E2M1 codes packed two per byte
// (the even element in the low nibble); every 32 consecutive elements of a
// row share one E8M0 scale 2^(e-127).  The block-scaled MMA applies both
// operands' scales inside the contraction, so
//     logit[t,s] = sum_h w[t,h] * max(0, sum_d q[t,h,d] k[s,d])
// needs no scale in the epilogue.
//
// Layout of the contraction as in dsa_score.cuh: keys on M (128 TMEM lanes),
// a group of TOK = 3 query rows x 64 heads on N = 192 (four rows would need
// two 256-column accumulators, all of tensor memory, with no room left for
// the scales).  Tensor memory holds two 192-column accumulators and the scale
// factors of the MMAs in flight:
//   A (keys)     a row's four scale bytes, copied to 4 columns of its lane
//   B (queries)  lane 32q + i, column j holds row 32j + i's four scale bytes
//                for every lane quarter q (columns 0-5: two copies of 4)
// (the layouts the block-scaled MMA reads; the copies come from shared-memory
// rows that the producer warp fills with tcgen05.cp.128x128b).
//
// Roles (448 threads: 14 warps, so 128 registers a thread):
//   warp 0      producer: scale rows (plain loads + shared stores) and TMA
//               boxes of packed E2M1 rows (64-byte swizzle) for q and K
//   warp 1      TMEM allocator; one thread copies the scale factors and
//               issues two K=64 block-scaled MMAs per 128-key tile
//   warps 2-13  three epilogue warpgroups (one per token) on the same tile,
//               the MMA of the next tile filling the other accumulator
#pragma once

#include "dsa_score.cuh"

namespace dsa {

struct MxCfg {
  static constexpr int H = 64;
  static constexpr int D = 128;
  static constexpr int TOK = 3;
  static constexpr int N = TOK * H;            // 128 MMA columns
  static constexpr int TILE = 128;             // keys per tile (MMA M)
  static constexpr int ROW_BYTES = D / 2;      // packed E2M1
  static constexpr int KSTEPS = D / 64;        // K = 64 elements per MMA
  static constexpr int SETS = 1;               // epilogue sets (alternate tiles)
  static constexpr int EPI_WARPS = 4 * TOK * SETS;
  static constexpr int THREADS = 64 + 32 * EPI_WARPS;
  static constexpr int Q_BYTES = N * ROW_BYTES;          // 8 KB
  static constexpr int STAGE_BYTES = TILE * ROW_BYTES;   // 8 KB
  static constexpr int SF_BYTES = 128 * 16;              // one 128-row scale block
  // tensor memory columns
  static constexpr uint32_t COL_ACC = 0;                 // two accumulators of N
  static constexpr uint32_t COL_SFA = 2 * N;             // two 4-column blocks
  static constexpr int NSFB = (N + 127) / 128;           // B-scale copies per q buffer
  static constexpr uint32_t COL_SFB = COL_SFA + 8;       // two blocks of NSFB x 4 columns
  static constexpr uint32_t TMEM_COLS = 512;
  // shared memory: q[2] | K stages | sfb[2] | sfa stages | misc
  static constexpr int NST = 8;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + 2 * Q_BYTES;
  static constexpr int OFF_SFB = OFF_K + NST * STAGE_BYTES;
  static constexpr int OFF_SFA = OFF_SFB + 2 * NSFB * SF_BYTES;
  static constexpr int OFF_W = OFF_SFA + NST * SF_BYTES;     // N floats
  static constexpr int OFF_RANGE = OFF_W + N * 4;            // TOK lo, TOK hi
  static constexpr int OFF_BARS = OFF_RANGE + 64;
  static constexpr int NBARS = 8 + 8 + 2 + 2 + 2 + 2 + 1;
  static constexpr int OFF_SLOT = OFF_BARS + NBARS * 8;
  static constexpr int SMEM = 1024 + OFF_SLOT + 16;

  static_assert(Q_BYTES % 1024 == 0 && STAGE_BYTES % 1024 == 0, "swizzle atoms");
  static_assert(SMEM <= 232448, "shared memory");
  static_assert(COL_SFB + 8 * NSFB <= TMEM_COLS, "tensor memory");
};

// Orders uses of r after the preceding tcgen05.wait::ld (emits nothing).
__device__ __forceinline__ void tmem_tie16(uint32_t (&r)[16]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}

// Shared-memory matrix descriptor of a K-major operand in the 64-byte
// swizzled layout TMA writes with CU_TENSOR_MAP_SWIZZLE_64B: rows of 64 bytes,
// 8-row (512-byte) swizzle atoms along M/N (stride-dimension offset 512,
// leading offset unused, layout type 4 = 64-byte swizzle).
__device__ __forceinline__ uint64_t sw64_kmajor_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1u) << 16;
  d |= static_cast<uint64_t>(512u >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(4u) << 61;
  return d;
}

// Descriptor of a 128-row x 16-byte block in shared memory (rows contiguous,
// no swizzle: 8-row core matrices 128 bytes apart), the source of
// tcgen05.cp.128x128b.
__device__ __forceinline__ uint64_t rows16_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(128u >> 4) << 16;
  d |= static_cast<uint64_t>(128u >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  return d;
}

// Instruction descriptor of tcgen05.mma kind::mxf4: E2M1 A and B (format 1),
// K-major, UE8M0 scales (bit 23), N >> 3 at bits 17-22, M >> 4 at 24-28, and
// the byte of the 32-bit scale column each operand's two scales start at
// (B: bits 4-5, A: bits 29-30; 0 or 2 with scale_vec::2X).
__host__ __device__ constexpr uint32_t mxf4_idesc(int M, int N, uint32_t sf_id) {
  return (sf_id << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (1u << 23) | (static_cast<uint32_t>(M >> 4) << 24) | (sf_id << 29);
}

__device__ __forceinline__ void mma_mxf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], "
      "[%5], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Shared memory (128 rows x 16 bytes) -> 128 TMEM lanes x 4 columns.
__device__ __forceinline__ void tmem_cp_128x128b(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.128x128b [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

__global__ void __launch_bounds__(MxCfg::THREADS, 1)
    score_mx_kernel(const __grid_constant__ ScoreParams p, const uint32_t* __restrict__ q_sf,
                    const uint32_t* __restrict__ k_sf) {
  using C = MxCfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* q_s = smem + C::OFF_Q;
  uint8_t* k_s = smem + C::OFF_K;
  uint8_t* sfb_s = smem + C::OFF_SFB;
  uint8_t* sfa_s = smem + C::OFF_SFA;
  float* w_s = reinterpret_cast<float*>(smem + C::OFF_W);
  int* range_s = reinterpret_cast<int*>(smem + C::OFF_RANGE);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BARS);
  uint64_t* full = bars;          // [8]
  uint64_t* empty = bars + 8;     // [8]
  uint64_t* qfull = bars + 16;    // [2]
  uint64_t* qempty = bars + 18;   // [2]
  uint64_t* accf = bars + 20;     // [2]
  uint64_t* acce = bars + 22;     // [2]
  uint64_t* drain = bars + 24;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_SLOT);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_SLOT + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int P = gridDim.x;
  const int cta = blockIdx.x;
  const int nslots = (p.R + C::TOK - 1) / C::TOK;
  const int rounds = (nslots + P - 1) / P;
  const int64_t qrows = static_cast<int64_t>(p.R) * C::H;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&qfull[i], 1);
      mbar_init(&qempty[i], 1);
      mbar_init(&accf[i], 1);
      mbar_init(&acce[i], C::EPI_WARPS / C::SETS);
    }
    mbar_init(drain, 1);
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
      const ScoreGroup g = score_group<C::TOK, false>(p, slot, lane, nullptr);
      if (g.kt_end <= g.kt_begin) continue;
      const int qb = ngroups & 1;
      if (lane == 0)
        ok = mbar_wait_bounded(&qempty[qb], (static_cast<uint32_t>(ngroups >> 1) & 1u) ^ 1u,
                               abort_flag);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      {
        // Query scales: lane 32q + i, column j <- q row 32j + i, for every q.
        const int64_t r0 = static_cast<int64_t>(g.row0) * C::H;
#pragma unroll
        for (int cc = 0; cc < C::NSFB; ++cc) {
          uint32_t wv[4];
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const int n = 128 * cc + 32 * jj + lane;
            const int64_t row = r0 + n;
            wv[jj] = (n < C::N && row < qrows) ? __ldg(q_sf + row) : 0x7F7F7F7Fu;
          }
          uint4* dst = reinterpret_cast<uint4*>(sfb_s + (qb * C::NSFB + cc) * C::SF_BYTES);
#pragma unroll
          for (int qq = 0; qq < 4; ++qq)
            dst[32 * qq + lane] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
        }
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_expect_tx(&qfull[qb], C::Q_BYTES);
        tma_load_2d(q_s + qb * C::Q_BYTES, &p.tmap_q, &qfull[qb], 0, g.row0 * C::H);
        ++qissued;
      }
      // Key scale words of a tile (one per key), loaded a tile ahead of use
      // so that their latency stays off the producer's per-tile path.
      auto load_kv = [&](int kt, uint32_t (&kv)[4]) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int key = kt * C::TILE + 32 * j + lane;
          kv[j] = (kt < g.kt_end && key < p.S) ? __ldg(k_sf + key) : 0x7F7F7F7Fu;
        }
      };
      uint32_t kv_next[4];
      load_kv(g.kt_begin, kv_next);
      for (int kt = g.kt_begin; kt < g.kt_end; ++kt) {
        const int stage = kiter % C::NST;
        const uint32_t phase = static_cast<uint32_t>(kiter / C::NST) & 1u;
        uint32_t kv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) kv[j] = kv_next[j];
        load_kv(kt + 1, kv_next);
        if (lane == 0) ok = mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        // Key scales: a key's four bytes in all 4 columns of its own lane.
        uint4* dst = reinterpret_cast<uint4*>(sfa_s + stage * C::SF_BYTES);
#pragma unroll
        for (int j = 0; j < 4; ++j) dst[32 * j + lane] = make_uint4(kv[j], kv[j], kv[j], kv[j]);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
          tma_load_2d(k_s + stage * C::STAGE_BYTES, &p.tmap_k, &full[stage], 0, kt * C::TILE);
        }
        ++kiter;
      }
      ++ngroups;
    }
    if (lane == 0 && !ok) {
      *abort_flag = 1;
      record_error(p.err, kErrTimeout);
      const int first = kiter > C::NST ? kiter - C::NST : 0;
      for (int i = first; i < kiter; ++i)
        mbar_wait_bounded(&full[i % C::NST], static_cast<uint32_t>(i / C::NST) & 1u, nullptr,
                          100000000ull);
      for (int j = qissued > 2 ? qissued - 2 : 0; j < qissued; ++j)
        mbar_wait_bounded(&qfull[j & 1], static_cast<uint32_t>(j >> 1) & 1u, nullptr,
                          100000000ull);
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issuer
    int kiter = 0, ngroups = 0, tc = 0;
    bool ok = true;
    for (int r = 0; r < rounds && ok; ++r) {
      const int slot = snake_slot(r, P, cta);
      if (slot >= nslots) continue;
      const ScoreGroup g = score_group<C::TOK, false>(p, slot, lane, nullptr);
      if (g.kt_end <= g.kt_begin) continue;
      if (lane == 0) {
        const int qb = ngroups & 1;
        ok = mbar_wait_bounded(&qfull[qb], static_cast<uint32_t>(ngroups >> 1) & 1u, abort_flag);
        const uint32_t q_addr = smem_u32(q_s + qb * C::Q_BYTES);
        const uint32_t sfb_t = tmem_base + C::COL_SFB + static_cast<uint32_t>(4 * C::NSFB * qb);
        bool first = true;
        for (int kt = g.kt_begin; ok && kt < g.kt_end; ++kt) {
          const int stage = kiter % C::NST;
          const uint32_t phase = static_cast<uint32_t>(kiter / C::NST) & 1u;
          const int buf = tc & 1;
          if (!mbar_wait_bounded(&acce[buf], (static_cast<uint32_t>(tc >> 1) & 1u) ^ 1u,
                                 abort_flag) ||
              !mbar_wait_bounded(&full[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t sfa_t = tmem_base + C::COL_SFA + static_cast<uint32_t>(4 * buf);
          tmem_cp_128x128b(sfa_t, rows16_desc(smem_u32(sfa_s + stage * C::SF_BYTES)));
          if (first) {
#pragma unroll
            for (int cc = 0; cc < C::NSFB; ++cc)
              tmem_cp_128x128b(sfb_t + 4u * cc,
                               rows16_desc(smem_u32(sfb_s + (qb * C::NSFB + cc) * C::SF_BYTES)));
            first = false;
          }
          const uint32_t d_tmem = tmem_base + C::COL_ACC + static_cast<uint32_t>(buf * C::N);
          const uint32_t k_addr = smem_u32(k_s + stage * C::STAGE_BYTES);
#pragma unroll
          for (int ks = 0; ks < C::KSTEPS; ++ks)
            mma_mxf4(d_tmem, sw64_kmajor_desc(k_addr + ks * 32), sw64_kmajor_desc(q_addr + ks * 32),
                     mxf4_idesc(C::TILE, C::N, 2u * ks), sfa_t, sfb_t, ks > 0 ? 1u : 0u);
          mma_commit(&empty[stage]);
          mma_commit(&accf[buf]);
          ++kiter;
          ++tc;
        }
        if (ok) mma_commit(&qempty[qb]);
        ++ngroups;
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    }
    if (lane == 0) {
      if (!ok) {
        *abort_flag = 1;
        record_error(p.err, kErrTimeout);
      }
      // TMEM is freed only after every copy and MMA of this thread completed.
      mma_commit(drain);
      mbar_wait_bounded(drain, 0u, nullptr, 100000000ull);
    }
  } else {
    // ------------------------------------------------------------- epilogue
    const int ew = warp - 2;
    const int set = ew / (4 * C::TOK);          // tiles with tc % SETS == set
    const int tok = (ew >> 2) % C::TOK;         // this warpgroup's token
    const int quarter = warp & 3;
    const int etid = threadIdx.x - 64;
    const int my_key = quarter * 32 + (lane >> 2) + 8 * (lane & 3);
    const uint32_t l0 = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t l1 = static_cast<uint32_t>(quarter * 32 + 16) << 16;
    int tcount = 0;
    bool ok = true;
    for (int r = 0; r < rounds; ++r) {
      const int slot = snake_slot(r, P, cta);
      if (slot >= nslots) continue;
      const ScoreGroup g = score_group<C::TOK, false>(p, slot, lane, nullptr);
      if (g.kt_end <= g.kt_begin) continue;
      // Stage the group's weights (halved: the ReLU is taken as x + |x|) and
      // row ranges once every epilogue thread is done with the previous group.
      asm volatile("bar.sync 1, %0;" ::"r"(32 * C::EPI_WARPS) : "memory");
      for (int i = etid; i < C::N; i += 32 * C::EPI_WARPS) {
        const int t = i / C::H, h = i % C::H;
        w_s[i] = t < g.ntok ? 0.5f * p.weights[static_cast<int64_t>(g.row0 + t) * C::H + h] : 0.f;
      }
      if (etid < C::TOK) {
        int lo = 0, hi = 0;
        if (etid < g.ntok) {
          lo = min(max(p.row_starts[g.row0 + etid], 0), p.S);
          hi = min(max(p.row_ends[g.row0 + etid], 0), p.S);
        }
        range_s[etid] = lo;
        range_s[C::TOK + etid] = hi;
      }
      asm volatile("bar.sync 1, %0;" ::"r"(32 * C::EPI_WARPS) : "memory");
      float2 wq[8];
#pragma unroll
      for (int b = 0; b < 8; ++b)
        wq[b] = *reinterpret_cast<const float2*>(w_s + tok * C::H + 8 * b + 2 * (lane & 3));
      const int rlo = range_s[tok], rhi = range_s[C::TOK + tok];
      const bool tok_ok = tok < g.ntok;
      const int ntile = g.kt_end - g.kt_begin;
      const int skip = ((set - tcount) % C::SETS + C::SETS) % C::SETS;
      int tc = tcount + skip;
      tcount += ntile;
      for (int kt = g.kt_begin + skip; ok && kt < g.kt_end; kt += C::SETS, tc += C::SETS) {
        const int buf = tc & 1;  // the accumulator of this tile
        ok = __all_sync(0xffffffffu,
                        mbar_wait_bounded(&accf[buf], static_cast<uint32_t>(tc >> 1) & 1u,
                                          abort_flag)
                            ? 1
                            : 0);
        if (!ok) break;
        tc_fence_after_sync();
        // The quad layout of dsa_score.cuh's e4m3 epilogue: 16x256b loads,
        // 16 heads of 4 keys per thread, ReLU as one packed add with |x|,
        // eight accumulators, then a shuffle exchange across the quad.
        const uint32_t cb = tmem_base + C::COL_ACC + static_cast<uint32_t>(buf * C::N + tok * C::H);
        float2 acc4[4], acc4b[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) acc4[i] = acc4b[i] = make_float2(0.f, 0.f);
        auto sum_chunk = [&](const uint32_t* v, int c) {
          const int hf = c & 1;
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const int rep = jj & 1;
            const int r0 = 4 * jj;
            const float2 w2 = wq[4 * (c >> 1) + jj];
            const float2 xa = make_float2(__uint_as_float(v[r0]), __uint_as_float(v[r0 + 1]));
            const float2 xb = make_float2(__uint_as_float(v[r0 + 2]), __uint_as_float(v[r0 + 3]));
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
        };
        // Chunk c: one 16x256b.x4 load, lanes +16(c & 1), heads 32(c >> 1) ..;
        // two chunks a batch: chunks 2-3 load while 0-1 are summed.
        uint32_t va[16], vb[16], vc[16], vd[16];
        tmem_ld16x256_x4_async(cb + l0, va);
        tmem_ld16x256_x4_async(cb + l1, vb);
        tmem_wait_ld16(va);
        tmem_tie16(vb);
        tmem_ld16x256_x4_async(cb + l0 + 32u, vc);
        tmem_ld16x256_x4_async(cb + l1 + 32u, vd);
        sum_chunk(va, 0);
        sum_chunk(vb, 1);
        tmem_wait_ld16(vc);
        tmem_tie16(vd);
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acce[buf]);
        sum_chunk(vc, 2);
        sum_chunk(vd, 3);
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
        const int s = kt * C::TILE + my_key;
        if (tok_ok && s < p.S)
          p.logits[static_cast<int64_t>(g.row0 + tok) * p.ld + s] =
              (s >= rlo && s < rhi) ? acc : -INFINITY;
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

}  // namespace dsa
