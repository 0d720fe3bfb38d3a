// dsa_topk.cu -- masked per-row top-k of fp32 index logits (sm_103a).
//
// Semantics of torch_dsa_topk as corrected in GitHub "vllm-project/vime" pull
// request #502 (third review comment): only columns inside the row's range
// [row_start, row_end) count, a -inf score is never selected, and the row is
// padded with -1 when fewer than k valid columns exist.  Readings where the
// page is silent: ties go to the lower column (-0.0 equals +0.0), NaN is never
// selected, and the selected columns are written in ascending column order.
//
// Every logit becomes an order-preserving 32-bit key (larger float -> larger
// key; -0.0 folded onto +0.0; -inf and NaN -> 0, which no valid score maps
// to).  The exact k-th largest key tau is found by a radix select over the key
// bits (11 + 11 + 10), after which every key > tau and the first need_eq keys
// == tau (in column order) are taken.  The output order comes from warp-ballot
// bitmaps of (key > tau) and (key == tau) and one prefix count over their
// words, so selected columns are written in ascending order directly.
//
// Two kernels:
//   topk_reg_kernel<THREADS, ITEMS, CL>  a row of up to CL*THREADS*ITEMS keys
//       is read once from memory into registers (ITEMS per thread, striped so
//       that each warp's loads are contiguous); the radix passes and the
//       ordered writes work on registers.  CL > 1 spreads a row over a
//       thread-block cluster whose CTAs merge their histograms and counts
//       through distributed shared memory (few, very long rows).
//   topk_stream_kernel  256 threads per row, several rows per SM: the first
//       pass streams the row with 16-byte loads, later passes re-read it
//       (from L2).
// A row whose columns are all valid and that has at most k of them is
// written directly as lo, lo+1, ..., hi-1.
#include "dsa_common.cuh"
#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr int kHistBins = 2048;

__device__ __forceinline__ uint32_t order_key(float x) {
  // fmaxf returns the other operand for a NaN (NaN -> -inf); adding +0.0
  // turns -0.0 into +0.0 (round to nearest).
  const float y = fmaxf(x, -INFINITY) + 0.0f;
  const uint32_t u = __float_as_uint(y);
  // Negative: all bits flipped; positive: the sign bit set.
  const uint32_t key = u ^ (static_cast<uint32_t>(static_cast<int32_t>(u) >> 31) | 0x80000000u);
  return key > 0x007FFFFFu ? key : 0u;  // -inf (0x007FFFFF) -> 0
}

// ---------------------------------------------------------------- clusters

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Every thread of every CTA of the cluster arrives and waits (release/acquire
// ordering of shared memory across the cluster).
__device__ __forceinline__ void cluster_barrier() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of `p` (this CTA's shared memory) in the shared memory of CTA `rank`.
__device__ __forceinline__ uint32_t cluster_map(const void* p, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(smem_u32(p)), "r"(rank));
  return out;
}

__device__ __forceinline__ void cluster_add(uint32_t addr, uint32_t v) {
  asm volatile("red.shared::cluster.add.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t cluster_load(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

// ------------------------------------------------------------- block scans

// Exclusive prefix sums of two counters per thread over the block; *total
// gets the block sums.  Contains barriers: every thread must call it.
template <int THREADS>
__device__ __forceinline__ uint2 block_scan2(uint2 v, uint2* warp_sums, uint2* total) {
  constexpr int NW = THREADS / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint2 x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t a = __shfl_up_sync(0xffffffffu, x.x, o);
    const uint32_t b = __shfl_up_sync(0xffffffffu, x.y, o);
    if (lane >= o) {
      x.x += a;
      x.y += b;
    }
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  uint2 before = make_uint2(0u, 0u), all = make_uint2(0u, 0u);
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    const uint2 s = warp_sums[w];
    if (w < warp) {
      before.x += s.x;
      before.y += s.y;
    }
    all.x += s.x;
    all.y += s.y;
  }
  *total = all;
  __syncthreads();
  return make_uint2(before.x + x.x - v.x, before.y + x.y - v.y);
}

// Over hist[0..nbins), the bin b holding the r-th largest element: above =
// sum of bins > b satisfies above < r <= above + hist[b].  Returns the sum of
// all bins; (b, above) are valid when r <= that sum.  Every thread gets the
// same values.
template <int THREADS>
__device__ __forceinline__ uint32_t find_bin(const uint32_t* hist, int nbins, uint32_t r,
                                             uint2* warp_sums, uint32_t* sel, uint32_t* bin,
                                             uint32_t* above) {
  const int per = nbins / THREADS;  // bins per thread, highest bins first
  const int top = nbins - 1 - static_cast<int>(threadIdx.x) * per;
  uint32_t local = 0;
  for (int i = 0; i < per; ++i) local += hist[top - i];
  uint2 total;
  const uint32_t excl = block_scan2<THREADS>(make_uint2(local, 0u), warp_sums, &total).x;
  if (excl < r && r <= excl + local) {
    uint32_t acc = excl;
    for (int i = 0; i < per; ++i) {
      const uint32_t h = hist[top - i];
      if (acc + h >= r) {
        sel[0] = static_cast<uint32_t>(top - i);
        sel[1] = acc;
        break;
      }
      acc += h;
    }
  }
  __syncthreads();
  *bin = sel[0];
  *above = sel[1];
  return total.x;
}

__device__ __forceinline__ void row_range(const TopkParams& p, int row, int* lo, int* hi) {
  if (p.context_lens) {
    const int b = row / p.next_n, j = row % p.next_n;
    const int end = p.context_lens[b] - p.next_n + j + 1;
    *lo = 0;
    *hi = min(max(end, 0), p.S);
  } else {
    *lo = min(max(p.row_starts[row], 0), p.S);
    *hi = min(max(p.row_ends[row], 0), p.S);
    if (*hi < *lo) *hi = *lo;
  }
}

// ------------------------------------------------------ register-resident

// Histogram slots are padded by one word every 32 bins, so that a thread
// reading a run of consecutive bins never shares a bank with its neighbours.
__device__ __forceinline__ int hpad(int bin) { return bin + (bin >> 5); }
constexpr int kHistSlots = kHistBins + kHistBins / 32;

// find_bin over a padded histogram (see find_bin), also returning the
// count of the selected bin.  Three barriers.
template <int THREADS>
__device__ __forceinline__ uint32_t find_bin_padded(const uint32_t* hist, int nbins, uint32_t r,
                                                    uint2* warp_sums, uint32_t* sel, uint32_t* bin,
                                                    uint32_t* above, uint32_t* count) {
  const int per = nbins / THREADS;  // consecutive bins per thread, highest first
  const int top = nbins - 1 - static_cast<int>(threadIdx.x) * per;
  uint32_t local = 0;
  for (int i = 0; i < per; ++i) local += hist[hpad(top - i)];
  uint2 total;
  const uint32_t excl = block_scan2<THREADS>(make_uint2(local, 0u), warp_sums, &total).x;
  if (excl < r && r <= excl + local) {
    uint32_t acc = excl;
    for (int i = 0; i < per; ++i) {
      const uint32_t h = hist[hpad(top - i)];
      if (acc + h >= r) {
        sel[0] = static_cast<uint32_t>(top - i);
        sel[1] = acc;
        sel[2] = h;
        break;
      }
      acc += h;
    }
  }
  __syncthreads();
  *bin = sel[0];
  *above = sel[1];
  *count = sel[2];
  return total.x;
}

template <int THREADS, int ITEMS, int CL>
__global__ void __launch_bounds__(THREADS, 65536 / (THREADS * 64)) topk_reg_kernel(const TopkParams p) {
  constexpr int NW = THREADS / 32;
  constexpr int SEG = THREADS * ITEMS;  // keys per CTA
  constexpr int WORDS = SEG / 32;
  static_assert(kHistBins % THREADS == 0 || THREADS <= kHistBins, "bins per thread");
  __shared__ uint32_t hist[2][kHistSlots];   // double buffer: one pass fills, the next is cleared
  // Cluster merge targets (read on the leader), double-buffered like hist.
  __shared__ uint32_t merged[CL > 1 ? 2 : 1][CL > 1 ? kHistSlots : 1];
  __shared__ uint32_t gt_bits[WORDS];
  __shared__ uint32_t eq_bits[WORDS];
  __shared__ uint2 warp_sums[NW];
  __shared__ uint32_t sel[4];
  __shared__ uint32_t valid_count;
  __shared__ uint2 cta_total;
  __shared__ uint2 cta_base;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = CL > 1 ? cluster_rank() : 0u;
  const int row = CL > 1 ? static_cast<int>(blockIdx.x) / CL : static_cast<int>(blockIdx.x);
  int lo, hi;
  row_range(p, row, &lo, &hi);
  const int n = hi - lo;
  const int seg0 = static_cast<int>(rank) * SEG;
  const int mine_n = min(max(n - seg0, 0), SEG);  // keys of this CTA's segment
  const float* src = p.logits + static_cast<int64_t>(row) * p.ld + lo + seg0;
  int32_t* dst = p.out + static_cast<int64_t>(row) * p.k;

  // hist[1] is cleared at the end of pass 0, before its first use.
  for (int i = tid; i < kHistSlots; i += THREADS) {
    hist[0][i] = 0u;
    if (CL > 1) merged[0][i] = 0u;
  }
  if (tid == 0) {
    valid_count = 0u;
    sel[3] = 0u;
  }

  // One read of the segment: element u*THREADS + tid; slots past the row end
  // are skipped a whole item at a time.
  uint32_t key[ITEMS];
#pragma unroll
  for (int u = 0; u < ITEMS; ++u) {
    const int e = u * THREADS + tid;
    key[u] = 0u;
    if (u * THREADS < mine_n && e < mine_n) key[u] = order_key(src[e]);
  }
  uint32_t nv = 0;
#pragma unroll
  for (int u = 0; u < ITEMS; ++u) nv += key[u] != 0u ? 1u : 0u;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) nv += __shfl_xor_sync(0xffffffffu, nv, o);
  // Histograms cleared (in every CTA of the cluster, before any merge).
  if constexpr (CL > 1) cluster_barrier(); else __syncthreads();
  if (lane == 0 && nv) atomicAdd(&valid_count, nv);

  // Pass 0 histogram of the top 11 bits (invalid keys are left out).  A row
  // of at most k columns takes every valid key: only the count is needed.
  if (n > p.k) {
#pragma unroll
    for (int u = 0; u < ITEMS; ++u) {
      if (u * THREADS < mine_n) {
        const uint32_t kk = key[u];
        if (kk != 0u) atomicAdd(&hist[0][hpad(static_cast<int>(kk >> 21))], 1u);
      }
    }
  }

  uint32_t prefix = 0u, rem = static_cast<uint32_t>(p.k);
  uint32_t tau = 0u, need_eq = 0u;  // take every key > tau, then the first need_eq == tau
  uint32_t nvalid = 0u;
#pragma unroll 1
  for (int d = 0; d < 3; ++d) {
    uint32_t* hcur = hist[d & 1];
    const int nbins = d == 2 ? 1024 : 2048;
    if (d > 0) {
      const int shift = d == 1 ? 10 : 0;
      const int pshift = d == 1 ? 21 : 10;
#pragma unroll
      for (int u = 0; u < ITEMS; ++u) {
        if (u * THREADS < mine_n) {
          // prefix >= 4 here (the smallest valid key is 0x00800000), so an
          // invalid key (0) never matches.
          const uint32_t kk = key[u];
          if ((kk >> pshift) == prefix)
            atomicAdd(&hcur[hpad(static_cast<int>((kk >> shift) & static_cast<uint32_t>(nbins - 1)))], 1u);
        }
      }
    }
    __syncthreads();
    if constexpr (CL > 1) {
      // Merge into the leader's histogram, then every CTA takes a copy.  The
      // leader zeroes the other merge buffer for the next pass meanwhile; the
      // second barrier orders that before anyone adds into it.
      const uint32_t leader = cluster_map(merged[d & 1], 0);
      for (int i = tid; i < kHistSlots; i += THREADS) {
        const uint32_t v = hcur[i];
        if (v) cluster_add(leader + 4u * i, v);
      }
      if (d == 0 && tid == 0 && valid_count) cluster_add(cluster_map(&sel[3], 0), valid_count);
      cluster_barrier();
      for (int i = tid; i < kHistSlots; i += THREADS) hcur[i] = cluster_load(leader + 4u * i);
      if (d == 0 && tid == 0) valid_count = cluster_load(cluster_map(&sel[3], 0));
      if (rank == 0)
        for (int i = tid; i < kHistSlots; i += THREADS) merged[(d + 1) & 1][i] = 0u;
      cluster_barrier();
    }
    if (d == 0) {
      nvalid = valid_count;
      if (nvalid <= static_cast<uint32_t>(p.k)) break;  // every valid key is taken
    }
    uint32_t b, above, cnt;
    find_bin_padded<THREADS>(hcur, nbins, rem, warp_sums, sel, &b, &above, &cnt);
    rem -= above;
    prefix = d == 0 ? b : ((prefix << (d == 1 ? 11 : 10)) | b);
    if (rem == cnt || d == 2) {
      // Either the whole bin is taken (every key whose top bits are >= prefix)
      // or the key is complete.
      const int used = d == 0 ? 11 : (d == 1 ? 22 : 32);
      if (d == 2) {
        tau = prefix;
        need_eq = rem;
      } else {
        tau = (prefix << (32 - used)) - 1u;
        need_eq = 0u;
      }
      break;
    }
    // Clear the other buffer for the next pass (it held pass d-1).
    uint32_t* hnext = hist[(d + 1) & 1];
    for (int i = tid; i < kHistSlots; i += THREADS) hnext[i] = 0u;
    __syncthreads();
  }

  const int nsel = nvalid < static_cast<uint32_t>(p.k) ? static_cast<int>(nvalid) : p.k;
  if (nvalid <= static_cast<uint32_t>(p.k) && nvalid == static_cast<uint32_t>(n)) {
    // Every column of the row is valid and taken: indices lo .. hi-1, in order.
    for (int i = tid; i < mine_n; i += THREADS) dst[seg0 + i] = lo + seg0 + i;
  } else {
    // Ballot words: word u*NW + warp holds columns seg0 + (u*NW + warp)*32 + lane.
#pragma unroll
    for (int u = 0; u < ITEMS; ++u) {
      if (u * THREADS < mine_n) {
        const uint32_t g = __ballot_sync(0xffffffffu, key[u] > tau);
        const uint32_t e = __ballot_sync(0xffffffffu, need_eq > 0u && key[u] == tau);
        if (lane == 0) {
          gt_bits[u * NW + warp] = g;
          eq_bits[u * NW + warp] = e;
        }
      }
    }
    __syncthreads();
    // Prefix counts over the words, in column order (each thread a run of words).
    const int nwords = (mine_n + 31) >> 5;
    const int per = (nwords + THREADS - 1) / THREADS;
    const int w0 = min(tid * per, nwords), w1 = min(w0 + per, nwords);
    uint2 mine = make_uint2(0u, 0u);
    for (int w = w0; w < w1; ++w) {
      mine.x += __popc(gt_bits[w]);
      mine.y += __popc(eq_bits[w]);
    }
    uint2 total;
    const uint2 before = block_scan2<THREADS>(mine, warp_sums, &total);
    uint2 base = make_uint2(0u, 0u);
    if constexpr (CL > 1) {
      // Counts of the lower-ranked CTAs of the cluster come first.
      if (tid == 0) cta_total = total;
      cluster_barrier();
      if (tid == 0) {
        uint2 acc = make_uint2(0u, 0u);
        for (uint32_t r = 0; r < rank; ++r) {
          const uint32_t a = cluster_map(&cta_total, r);
          acc.x += cluster_load(a);
          acc.y += cluster_load(a + 4u);
        }
        cta_base = acc;
      }
      __syncthreads();
      base = cta_base;
      cluster_barrier();  // no CTA leaves while another may still read its shared memory
    }
    // Word prefixes (gt count, eq count) replace the ballot words in place.
    uint32_t gp = base.x + before.x, ep = base.y + before.y;
    for (int w = w0; w < w1; ++w) {
      const uint32_t g = gt_bits[w], e = eq_bits[w];
      gt_bits[w] = gp;
      eq_bits[w] = ep;
      gp += __popc(g);
      ep += __popc(e);
    }
    __syncthreads();
    // Every lane writes its own column: position = selected columns before it.
    const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
    for (int u = 0; u < ITEMS; ++u) {
      if (u * THREADS < mine_n) {
        const int w = u * NW + warp;
        const uint32_t kk = key[u];
        const bool g = kk > tau;
        const bool e = need_eq > 0u && kk == tau;
        const uint32_t gm = __ballot_sync(0xffffffffu, g);
        const uint32_t em = __ballot_sync(0xffffffffu, e);
        const uint32_t gb = gt_bits[w] + __popc(gm & lt);
        const uint32_t eb = eq_bits[w] + __popc(em & lt);
        const int col = lo + seg0 + u * THREADS + tid;
        if (g) dst[gb + min(eb, need_eq)] = col;
        else if (e && eb < need_eq) dst[gb + eb] = col;
      }
    }
  }
  if (rank == 0)
    for (int i = nsel + tid; i < p.k; i += THREADS) dst[i] = -1;
}

// ------------------------------------------------------------- short rows

// One CTA per row of up to THREADS*ITEMS keys, held in registers.  Warp w
// owns columns [w*32*ITEMS, (w+1)*32*ITEMS) of the row, item u of lane l
// being column w*32*ITEMS + u*32 + l: every load is warp-contiguous, and a
// warp meets its columns in order, so each selected column's output position
// is a running per-warp count plus the selected columns of earlier warps.
template <int THREADS, int ITEMS, int MINB>
__global__ void __launch_bounds__(THREADS, MINB) topk_row_kernel(const TopkParams p) {
  constexpr int NW = THREADS / 32;
  constexpr int WSPAN = 32 * ITEMS;
  __shared__ __align__(16) uint32_t hist[2][kHistSlots];
  __shared__ uint2 warp_sums[NW];
  __shared__ uint2 warp_cnt[NW];
  __shared__ uint32_t sel[4];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = blockIdx.x;
  int lo, hi;
  row_range(p, row, &lo, &hi);
  const int n = hi - lo;
  const float* src = p.logits + static_cast<int64_t>(row) * p.ld + lo;
  int32_t* dst = p.out + static_cast<int64_t>(row) * p.k;
  const int wbase = warp * WSPAN;
  // Items of this warp holding at least one column of the row (warp-uniform).
  const int nit = min(max((n - wbase + 31) >> 5, 0), ITEMS);

  float x[ITEMS];
#pragma unroll
  for (int u = 0; u < ITEMS; ++u) {
    const int c = wbase + u * 32 + lane;
    x[u] = c < n ? __ldg(src + c) : -INFINITY;
  }

  uint32_t tau = 0u, need_eq = 0u;  // take every key > tau, then the first need_eq == tau
  int nsel;
  uint32_t key[ITEMS];
  if (n <= p.k) {
    // Every valid key is taken: tau = 0.  All of them valid: lo, lo+1, ...
    // (x > -inf is false for -inf and NaN alone.)
    uint32_t nv = 0u;
#pragma unroll
    for (int u = 0; u < ITEMS; ++u) nv += x[u] > -INFINITY ? 1u : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) nv += __shfl_xor_sync(0xffffffffu, nv, o);
    if (lane == 0) warp_cnt[warp].x = nv;
    __syncthreads();
    uint32_t all = 0u;
#pragma unroll
    for (int w = 0; w < NW; ++w) all += warp_cnt[w].x;
    if (all == static_cast<uint32_t>(n)) {
      for (int i = tid; i < p.k; i += THREADS) dst[i] = i < n ? lo + i : -1;
      return;
    }
    nsel = static_cast<int>(all);
#pragma unroll
    for (int u = 0; u < ITEMS; ++u) key[u] = order_key(x[u]);
    __syncthreads();  // warp_cnt is rewritten below
  } else {
#pragma unroll
    for (int u = 0; u < ITEMS; ++u) key[u] = order_key(x[u]);
    for (int i = tid; i < kHistSlots / 4; i += THREADS) {
      reinterpret_cast<uint4*>(hist[0])[i] = make_uint4(0u, 0u, 0u, 0u);
      reinterpret_cast<uint4*>(hist[1])[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    __syncthreads();
    // Digit 1: the top 11 key bits (invalid keys are left out).
#pragma unroll
    for (int u = 0; u < ITEMS; ++u) {
      if (u < nit) {
        const uint32_t kk = key[u];
        if (kk != 0u) atomicAdd(&hist[0][hpad(static_cast<int>(kk >> 21))], 1u);
      }
    }
    __syncthreads();
    uint32_t b, above, cnt;
    const uint32_t nvalid =
        find_bin_padded<THREADS>(hist[0], kHistBins, static_cast<uint32_t>(p.k), warp_sums, sel,
                                 &b, &above, &cnt);
    if (nvalid <= static_cast<uint32_t>(p.k)) {
      nsel = static_cast<int>(nvalid);  // every valid key is taken
    } else {
      nsel = p.k;
      uint32_t rem = static_cast<uint32_t>(p.k) - above;
      uint32_t prefix = b;
      if (rem == cnt) {
        tau = (prefix << 21) - 1u;  // the whole bin is taken
      } else {
        // Digit 2: bits 20..10 of the keys in bin `prefix`; hist[0] is
        // cleared meanwhile for digit 3.
#pragma unroll
        for (int u = 0; u < ITEMS; ++u) {
          if (u < nit) {
            const uint32_t kk = key[u];
            if ((kk >> 21) == prefix)
              atomicAdd(&hist[1][hpad(static_cast<int>((kk >> 10) & 2047u))], 1u);
          }
        }
        for (int i = tid; i < kHistSlots / 4; i += THREADS)
          reinterpret_cast<uint4*>(hist[0])[i] = make_uint4(0u, 0u, 0u, 0u);
        __syncthreads();
        find_bin_padded<THREADS>(hist[1], kHistBins, rem, warp_sums, sel, &b, &above, &cnt);
        rem -= above;
        prefix = (prefix << 11) | b;
        if (rem == cnt) {
          tau = (prefix << 10) - 1u;
        } else {
          // Digit 3: bits 9..0 of the keys with the 22-bit prefix.
#pragma unroll
          for (int u = 0; u < ITEMS; ++u) {
            if (u < nit) {
              const uint32_t kk = key[u];
              if ((kk >> 10) == prefix) atomicAdd(&hist[0][hpad(static_cast<int>(kk & 1023u))], 1u);
            }
          }
          __syncthreads();
          find_bin_padded<THREADS>(hist[0], 1024, rem, warp_sums, sel, &b, &above, &cnt);
          tau = (prefix << 10) | b;
          need_eq = rem - above;
        }
      }
    }
  }

  // Per-warp counts of keys > tau (and == tau), then the ordered writes.
  uint32_t cg = 0u, ce = 0u;
#pragma unroll
  for (int u = 0; u < ITEMS; ++u) cg += key[u] > tau ? 1u : 0u;
  if (need_eq != 0u) {
#pragma unroll
    for (int u = 0; u < ITEMS; ++u) ce += key[u] == tau ? 1u : 0u;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    cg += __shfl_xor_sync(0xffffffffu, cg, o);
    ce += __shfl_xor_sync(0xffffffffu, ce, o);
  }
  if (lane == 0) warp_cnt[warp] = make_uint2(cg, ce);
  __syncthreads();
  uint32_t grun = 0u, erun = 0u;
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    if (w < warp) {
      grun += warp_cnt[w].x;
      erun += warp_cnt[w].y;
    }
  }
  const uint32_t lt = (1u << lane) - 1u;
  if (need_eq == 0u) {
#pragma unroll
    for (int u = 0; u < ITEMS; ++u) {
      if (u < nit) {
        const bool g = key[u] > tau;
        const uint32_t m = __ballot_sync(0xffffffffu, g);
        if (g) dst[grun + __popc(m & lt)] = lo + wbase + u * 32 + lane;
        grun += __popc(m);
      }
    }
  } else {
#pragma unroll
    for (int u = 0; u < ITEMS; ++u) {
      if (u < nit) {
        const bool g = key[u] > tau, e = key[u] == tau;
        const uint32_t mg = __ballot_sync(0xffffffffu, g);
        const uint32_t me = __ballot_sync(0xffffffffu, e);
        const uint32_t gb = grun + __popc(mg & lt), eb = erun + __popc(me & lt);
        const int col = lo + wbase + u * 32 + lane;
        if (g) dst[gb + min(eb, need_eq)] = col;
        else if (e && eb < need_eq) dst[gb + eb] = col;
        grun += __popc(mg);
        erun += __popc(me);
      }
    }
  }
  for (int i = nsel + tid; i < p.k; i += THREADS) dst[i] = -1;
}

// --------------------------------------------------------------- streaming

// Visit slots i in [0, n_iter) with THREADS threads, i = base + u*THREADS for
// u < U: U independent read-only loads are issued before any is used, so
// that each thread keeps U requests in flight.  Only src[0..n_load) is read;
// x = -inf for every other slot.  fn(i, x) is called for every slot of a
// batch, also for i >= n_iter, so that warp-collective code inside fn runs on
// full warps; fn must not touch memory indexed by such an i.  Lanes of a warp
// see consecutive i for each u.
template <int THREADS, int U, class Fn>
__device__ __forceinline__ void stream_row(const float* __restrict__ src, int n_iter, int n_load,
                                           Fn&& fn) {
  for (int base = static_cast<int>(threadIdx.x); base < n_iter; base += THREADS * U) {
    float x[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * THREADS;
      x[u] = i < n_load ? __ldg(src + i) : -INFINITY;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) fn(base + u * THREADS, x[u]);
  }
}


template <int kStreamThreads>
__global__ void __launch_bounds__(kStreamThreads, kStreamThreads >= 1024 ? 1 : 8)
    topk_stream_kernel(const TopkParams p) {
  // Loads in flight per thread in the streaming passes.
  constexpr int U = kStreamThreads >= 1024 ? 16 : 4;
  // Keys of the threshold bin gathered after pass 0 (when they fit).
  constexpr int kCand = kStreamThreads >= 1024 ? 8192 : 2048;
  extern __shared__ uint32_t sm[];
  uint32_t* hist = sm;                   // kHistBins
  uint32_t* cand = sm + kHistBins;       // kCand keys
  uint32_t* gt_bits = cand + kCand;      // ceil(S/32) words
  uint32_t* eq_bits = gt_bits + p.bitmap_words;
  __shared__ uint2 warp_sums[kStreamThreads / 32];
  __shared__ uint32_t sel[4];
  __shared__ uint32_t valid_count;
  __shared__ uint32_t ncand;

  const int row = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31;
  int lo, hi;
  row_range(p, row, &lo, &hi);
  const int n = hi - lo;
  const float* src = p.logits + static_cast<int64_t>(row) * p.ld + lo;
  int32_t* dst = p.out + static_cast<int64_t>(row) * p.k;

  // Pass 0: histogram of the top 11 key bits, 16-byte loads from memory.
  {
  for (int i = tid; i < kHistBins; i += kStreamThreads) hist[i] = 0u;
  if (tid == 0) valid_count = 0u;
  __syncthreads();
  {
    uint32_t nv = 0;
    const uintptr_t addr = reinterpret_cast<uintptr_t>(src);
    const int head = min(static_cast<int>(((16u - (addr & 15u)) & 15u) >> 2), n);
    const int body = (n - head) >> 2;
    // A row of at most k columns takes every valid key: only the count is needed.
    const bool need_hist = n > p.k;
    auto add = [&](float x) {
      const uint32_t kk = order_key(x);
      if (kk != 0u) {
        if (need_hist) atomicAdd(&hist[kk >> 21], 1u);
        ++nv;
      }
    };
    for (int i = tid; i < head; i += kStreamThreads) add(src[i]);
    const float4* src4 = reinterpret_cast<const float4*>(src + head);
    for (int i0 = tid; i0 < body; i0 += 4 * kStreamThreads) {
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + u * kStreamThreads;
        v[u] = i < body ? __ldg(src4 + i) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        add(v[u].x);
        add(v[u].y);
        add(v[u].z);
        add(v[u].w);
      }
    }
    for (int i = head + 4 * body + tid; i < n; i += kStreamThreads) add(src[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) nv += __shfl_xor_sync(0xffffffffu, nv, o);
    if (lane == 0 && nv) atomicAdd(&valid_count, nv);
  }
  }
  __syncthreads();
  const uint32_t nvalid = valid_count;
  const int nsel = nvalid < static_cast<uint32_t>(p.k) ? static_cast<int>(nvalid) : p.k;

  uint32_t prefix = 0u, rem = static_cast<uint32_t>(p.k), tau = 0u, need_eq = 0u;
  if (nvalid > static_cast<uint32_t>(p.k)) {
    bool gathered = false;  // the keys still in play sit in cand[0..ncand)
#pragma unroll 1
    for (int d = 0; d < 3; ++d) {
      const int nbins = d == 2 ? 1024 : 2048;
      if (d > 0) {
        const int shift = d == 1 ? 10 : 0;
        const int pshift = d == 1 ? 21 : 10;
        for (int i = tid; i < nbins; i += kStreamThreads) hist[i] = 0u;
        __syncthreads();
        if (gathered) {
          const int nc = min(static_cast<int>(ncand), kCand);
          for (int i = tid; i < nc; i += kStreamThreads) {
            const uint32_t kk = cand[i];
            if ((kk >> pshift) == prefix)
              atomicAdd(&hist[(kk >> shift) & static_cast<uint32_t>(nbins - 1)], 1u);
          }
        } else {
          stream_row<kStreamThreads, U>(src, n, n, [&](int, float x) {
            const uint32_t kk = order_key(x);
            if ((kk >> pshift) == prefix)
              atomicAdd(&hist[(kk >> shift) & static_cast<uint32_t>(nbins - 1)], 1u);
          });
        }
        __syncthreads();
      }
      uint32_t b, above;
      find_bin<kStreamThreads>(hist, nbins, rem, warp_sums, sel, &b, &above);
      const uint32_t cnt = hist[b];
      rem -= above;
      prefix = d == 0 ? b : ((prefix << (d == 1 ? 11 : 10)) | b);
      __syncthreads();
      if (rem == cnt || d == 2) {
        const int used = d == 0 ? 11 : (d == 1 ? 22 : 32);
        tau = d == 2 ? prefix : (prefix << (32 - used)) - 1u;
        need_eq = d == 2 ? rem : 0u;
        break;
      }
      if (d == 0 && cnt <= static_cast<uint32_t>(kCand)) {
        // One pass gathers the keys of the threshold bin; the later passes
        // read them from shared memory instead of the row.
        if (tid == 0) ncand = 0u;
        __syncthreads();
        // Warp-collective body: iterate over whole warps (loads stay < n).
        stream_row<kStreamThreads, U>(src, (n + 31) & ~31, n, [&](int, float x) {
          const uint32_t kk = order_key(x);
          const bool hit = (kk >> 21) == prefix;
          const uint32_t m = __ballot_sync(0xffffffffu, hit);
          if (m) {
            uint32_t slot = 0u;
            if (lane == 0) slot = atomicAdd(&ncand, static_cast<uint32_t>(__popc(m)));
            slot = __shfl_sync(0xffffffffu, slot, 0);
            const uint32_t idx = slot + __popc(m & ((1u << lane) - 1u));
            if (hit && idx < static_cast<uint32_t>(kCand)) cand[idx] = kk;
          }
        });
        __syncthreads();
        gathered = true;
      }
    }
  }

  if (nvalid <= static_cast<uint32_t>(p.k) && nvalid == static_cast<uint32_t>(n)) {
    for (int i = tid; i < n; i += kStreamThreads) dst[i] = lo + i;
  } else {
    const int nwords = (n + 31) >> 5;
    // Every warp-load covers one 32-column word (n rounded up to whole words).
    stream_row<kStreamThreads, U>(src, nwords << 5, n, [&](int i, float x) {
      const uint32_t kk = i < n ? order_key(x) : 0u;
      const uint32_t g = __ballot_sync(0xffffffffu, kk > tau);
      const uint32_t e = __ballot_sync(0xffffffffu, need_eq > 0u && kk == tau);
      if (lane == 0 && (i >> 5) < nwords) {
        gt_bits[i >> 5] = g;
        eq_bits[i >> 5] = e;
      }
    });
    __syncthreads();
    const int per = (nwords + kStreamThreads - 1) / kStreamThreads;
    const int w0 = min(tid * per, nwords), w1 = min(w0 + per, nwords);
    uint2 mine = make_uint2(0u, 0u);
    for (int w = w0; w < w1; ++w) {
      mine.x += __popc(gt_bits[w]);
      mine.y += __popc(eq_bits[w]);
    }
    uint2 total;
    const uint2 before = block_scan2<kStreamThreads>(mine, warp_sums, &total);
    uint32_t gb = before.x, eb = before.y;
    for (int w = w0; w < w1; ++w) {
      const uint32_t g = gt_bits[w], e = eq_bits[w];
      uint32_t m = g | e;
      while (m) {
        const int bit = __ffs(m) - 1;
        m &= m - 1;
        const int col = lo + (w << 5) + bit;
        if ((g >> bit) & 1u) {
          dst[gb + min(eb, need_eq)] = col;
          ++gb;
        } else {
          if (eb < need_eq) dst[gb + eb] = col;
          ++eb;
        }
      }
    }
  }
  for (int i = nsel + tid; i < p.k; i += kStreamThreads) dst[i] = -1;
}

// ----------------------------------------------------------- split path
//
// Few long rows (decode): every phase runs on a grid of (16384-key segment,
// row) CTAs, and the phases talk through per-row scratch:
//   hist[2048]        first-digit (top 11 bits) histogram of the row's valid keys
//   state[16]         mode, tau, need_eq, nvalid, b1, rem, completion counters, ncand
//   cand[kSplitCand]  keys of the threshold bin b1: their low 21 bits, and the
//                     segment they came from in the bits above
//   seg[3*kSplitSegs] per segment: keys above the first threshold, then the
//                     numbers of selected keys > tau and == tau in earlier segments
// Only hist and state are zeroed before the first phase.  Phases (one launch
// each):
//   hist    segments add their histograms; the last segment CTA of a row to
//           finish (a completion counter after a fence; nobody waits) picks
//           the threshold bin b1 and the row's mode;
//   gather  segments count their keys above bin b1 and append the keys of
//           bin b1; the last one of a row refines them to the exact tau and
//           need_eq (streaming the row when the bin holds more than
//           kSplitCand keys) and turns the per-segment counts into the output
//           offsets of every segment;
//   write   each segment places its selected columns at its offsets, in
//           column order; segment 0 writes the -1 tail.
constexpr int kSegKeys = 16384;
constexpr int kSegThreads = 1024;
constexpr int kSegItems = kSegKeys / kSegThreads;  // 16
constexpr int kSplitCand = 16384;
constexpr int kSplitSegs = 64;  // rows of up to 64 * 16384 keys
constexpr int kStateWords = 16;
constexpr int kStHist = 0, kStState = kHistBins, kStCand = kHistBins + kStateWords,
              kStSeg = kHistBins + kStateWords + kSplitCand,
              kStBase = kStSeg + kSplitSegs,  // (gt, eq) offset pairs
              kStWords = kStBase + 2 * kSplitSegs;
constexpr int kStZeroWords = kHistBins + kStateWords;  // zeroed before the first phase
// state words
constexpr int kSMode = 0, kSTau = 1, kSNeed = 2, kSValid = 3, kSB1 = 4, kSRem = 5,
              kSDoneHist = 6, kSDoneGather = 7, kSNcand = 8;
// Rows after the first phase: every valid key taken in place (iota); the
// exact tau known (select); the keys of bin b1 to be gathered and refined
// (gather), or, too many of them, the row to be streamed (stream).
enum : uint32_t { kModeSelect = 1u, kModeIota = 2u, kModeGather = 3u, kModeStream = 4u };
constexpr uint32_t kLow21 = (1u << 21) - 1u;

__device__ __forceinline__ uint32_t* split_row(const TopkParams& p, int row) {
  return p.split + static_cast<int64_t>(row) * p.split_words;
}

// True in every thread of the CTA that is the last of `total` CTAs to pass
// here for this counter: each CTA fences its earlier global writes, then
// counts itself in.  No CTA ever waits for another.
__device__ __forceinline__ bool last_to_arrive(uint32_t* counter, uint32_t total,
                                               uint32_t* flag_smem) {
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) *flag_smem = (atomicAdd(counter, 1u) == total - 1u) ? 1u : 0u;
  __syncthreads();
  const bool last = *flag_smem != 0u;
  if (last) __threadfence();
  return last;
}

__global__ void __launch_bounds__(kSegThreads, 2) topk_hist_kernel(const TopkParams p) {
  __shared__ uint32_t hist[kHistBins];
  __shared__ uint2 warp_sums[kSegThreads / 32];
  __shared__ uint32_t sel[2];
  __shared__ uint32_t flag;
  const int row = blockIdx.x;
  const int tid = threadIdx.x;
  int lo, hi;
  row_range(p, row, &lo, &hi);
  const int n = hi - lo;
  const int s0 = static_cast<int>(blockIdx.y) * kSegKeys;
  const int cnt = min(n - s0, kSegKeys);
  uint32_t* w = split_row(p, row);
  if (cnt <= 0) {
    if (blockIdx.y == 0 && tid == 0) {  // empty row: nothing to select
      w[kStState + kSMode] = kModeIota;
      w[kStState + kSValid] = 0u;
    }
    return;
  }
  for (int i = tid; i < kHistBins; i += kSegThreads) hist[i] = 0u;
  __syncthreads();
  const float* src = p.logits + static_cast<int64_t>(row) * p.ld + lo + s0;
  stream_row<kSegThreads, kSegItems>(src, cnt, cnt, [&](int, float x) {
    const uint32_t kk = order_key(x);
    if (kk != 0u) atomicAdd(&hist[kk >> 21], 1u);
  });
  __syncthreads();
  uint32_t* g = w + kStHist;
  for (int i = tid; i < kHistBins; i += kSegThreads) {
    const uint32_t v = hist[i];
    if (v) atomicAdd(&g[i], v);
  }
  const uint32_t nseg = static_cast<uint32_t>((n + kSegKeys - 1) / kSegKeys);
  if (!last_to_arrive(&w[kStState + kSDoneHist], nseg, &flag)) return;
  // The row's histogram is complete: find the threshold bin once.
  for (int i = tid; i < kHistBins; i += kSegThreads) hist[i] = __ldcg(&g[i]);
  __syncthreads();
  uint32_t b1, above;
  const uint32_t nvalid =
      find_bin<kSegThreads>(hist, kHistBins, static_cast<uint32_t>(p.k), warp_sums, sel, &b1, &above);
  if (tid == 0) {
    w[kStState + kSValid] = nvalid;
    if (nvalid <= static_cast<uint32_t>(p.k)) {
      // Every valid key is taken: tau = 0 (invalid keys are 0).
      w[kStState + kSMode] = nvalid == static_cast<uint32_t>(n) ? kModeIota : kModeSelect;
      w[kStState + kSTau] = 0u;
      w[kStState + kSNeed] = 0u;
    } else {
      const uint32_t rem = static_cast<uint32_t>(p.k) - above;
      const uint32_t bcnt = hist[b1];
      w[kStState + kSB1] = b1;
      w[kStState + kSRem] = rem;
      if (rem == bcnt) {  // the whole bin is taken
        w[kStState + kSMode] = kModeSelect;
        w[kStState + kSTau] = (b1 << 21) - 1u;
        w[kStState + kSNeed] = 0u;
      } else {
        w[kStState + kSMode] = bcnt <= static_cast<uint32_t>(kSplitCand) ? kModeGather : kModeStream;
      }
    }
  }
}

// Digits two and three of the radix select inside bin b1, over the keys
// key_at(i) for i < n (a key outside bin b1 is skipped).  rem is the rank
// still wanted inside bin b1.  Returns tau; *need_eq = keys == tau to take.
// Contains barriers: every thread must call it.
template <class KeyAt>
__device__ __forceinline__ uint32_t refine_in_bin(uint32_t b1, uint32_t rem, uint32_t* hist,
                                                  uint2* warp_sums, uint32_t* sel,
                                                  uint32_t* need_eq, KeyAt&& visit) {
  const int tid = threadIdx.x;
  uint32_t prefix = b1;
#pragma unroll 1
  for (int d = 1; d < 3; ++d) {
    const int nbins = d == 2 ? 1024 : 2048;
    const int shift = d == 1 ? 10 : 0;
    const int pshift = d == 1 ? 21 : 10;
    __syncthreads();
    for (int i = tid; i < nbins; i += kSegThreads) hist[i] = 0u;
    __syncthreads();
    visit([&](uint32_t kk) {
      if ((kk >> pshift) == prefix)
        atomicAdd(&hist[(kk >> shift) & static_cast<uint32_t>(nbins - 1)], 1u);
    });
    __syncthreads();
    uint32_t b, ab;
    find_bin<kSegThreads>(hist, nbins, rem, warp_sums, sel, &b, &ab);
    const uint32_t c = hist[b];
    rem -= ab;
    prefix = (prefix << (d == 1 ? 11 : 10)) | b;
    if (d == 1 && rem == c) {  // the whole sub-bin is taken
      *need_eq = 0u;
      return (prefix << 10) - 1u;
    }
  }
  *need_eq = rem;
  return prefix;
}

__global__ void __launch_bounds__(kSegThreads, 2) topk_gather_kernel(const TopkParams p) {
  constexpr int NW = kSegThreads / 32;
  __shared__ uint32_t hist[kHistBins];
  __shared__ uint2 warp_sums[NW];
  __shared__ uint32_t sel[2];
  __shared__ uint32_t flag;
  __shared__ uint32_t cta_hits, cta_base;
  __shared__ uint32_t seg_gt[kSplitSegs], seg_eq[kSplitSegs];
  extern __shared__ uint32_t cand_s[];  // kSplitCand keys: staging, then the refine's copy
  const int row = blockIdx.x;
  const int seg = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int lo, hi;
  row_range(p, row, &lo, &hi);
  const int n = hi - lo;
  const int s0 = seg * kSegKeys;
  const int cnt = min(n - s0, kSegKeys);
  if (cnt <= 0) return;
  uint32_t* w = split_row(p, row);
  const float* src = p.logits + static_cast<int64_t>(row) * p.ld + lo + s0;
  float x[kSegItems];
#pragma unroll
  for (int u = 0; u < kSegItems; ++u) {
    const int e = u * kSegThreads + tid;
    x[u] = e < cnt ? __ldg(src + e) : -INFINITY;
  }
  const uint32_t mode = w[kStState + kSMode];
  if (mode == kModeIota) return;
  const uint32_t b1 = w[kStState + kSB1];
  // Keys above `thr` are taken whatever the refinement finds; keys of bin
  // `want` (none unless gathering) are the candidates.
  const uint32_t thr = mode == kModeSelect ? w[kStState + kSTau] : ((b1 + 1u) << 21) - 1u;
  const uint32_t want = mode == kModeGather ? b1 : 0xFFFFFFFFu;
  if (tid == 0) cta_hits = 0u;
  __syncthreads();
  // This segment's candidates are staged in shared memory (any order), then
  // copied to one slot range of the row's candidate list.
  const uint32_t lt = (1u << lane) - 1u;
  uint32_t above = 0u;
#pragma unroll
  for (int u = 0; u < kSegItems; ++u) {
    const uint32_t kk = order_key(x[u]);
    above += kk > thr ? 1u : 0u;
    const bool hit = (kk >> 21) == want;
    const uint32_t m = __ballot_sync(0xffffffffu, hit);
    if (m) {
      uint32_t slot = 0u;
      if (lane == 0) slot = atomicAdd(&cta_hits, static_cast<uint32_t>(__popc(m)));
      slot = __shfl_sync(0xffffffffu, slot, 0) + __popc(m & lt);
      if (hit) cand_s[slot] = (static_cast<uint32_t>(seg) << 21) | (kk & kLow21);
    }
  }
  // Keys above the threshold in this segment (block reduction).
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) above += __shfl_xor_sync(0xffffffffu, above, o);
  if (lane == 0) warp_sums[warp] = make_uint2(above, 0u);
  __syncthreads();
  if (tid == 0) {
    uint32_t a = 0u;
    for (int i = 0; i < NW; ++i) a += warp_sums[i].x;
    w[kStSeg + seg] = a;
    cta_base = cta_hits ? atomicAdd(&w[kStState + kSNcand], cta_hits) : 0u;
  }
  __syncthreads();
  {
    const uint32_t nh = cta_hits, base = cta_base;
    uint32_t* cand = w + kStCand;
    for (uint32_t i = tid; i < nh; i += kSegThreads)
      if (base + i < static_cast<uint32_t>(kSplitCand)) cand[base + i] = cand_s[i];
  }
  const uint32_t nseg = static_cast<uint32_t>((n + kSegKeys - 1) / kSegKeys);
  if (!last_to_arrive(&w[kStState + kSDoneGather], nseg, &flag)) return;

  // Last gather CTA of the row: the exact tau / need_eq, then the offsets of
  // every segment's selected columns.
  for (int i = tid; i < kSplitSegs; i += kSegThreads) {
    seg_gt[i] = 0u;
    seg_eq[i] = 0u;
  }
  uint32_t tau = thr, need_eq = 0u;
  if (mode == kModeGather) {
    const int nc = min(static_cast<int>(__ldcg(&w[kStState + kSNcand])), kSplitCand);
    const uint32_t* cand = w + kStCand;
    for (int i = tid; i < nc; i += kSegThreads) cand_s[i] = __ldcg(&cand[i]);
    const uint32_t hi_bits = b1 << 21;
    tau = refine_in_bin(b1, w[kStState + kSRem], hist, warp_sums, sel, &need_eq, [&](auto&& fn) {
      for (int i = tid; i < nc; i += kSegThreads) fn(hi_bits | (cand_s[i] & kLow21));
    });
    for (int i = tid; i < nc; i += kSegThreads) {
      const uint32_t c = cand_s[i];
      const uint32_t kk = hi_bits | (c & kLow21);
      if (kk > tau) atomicAdd(&seg_gt[c >> 21], 1u);
      else if (kk == tau && need_eq) atomicAdd(&seg_eq[c >> 21], 1u);
    }
  } else if (mode == kModeStream) {
    const float* row_src = p.logits + static_cast<int64_t>(row) * p.ld + lo;
    tau = refine_in_bin(b1, w[kStState + kSRem], hist, warp_sums, sel, &need_eq, [&](auto&& fn) {
      stream_row<kSegThreads, kSegItems>(row_src, n, n, [&](int, float x) { fn(order_key(x)); });
    });
    stream_row<kSegThreads, kSegItems>(row_src, n, n, [&](int i, float x) {
      const uint32_t kk = order_key(x);
      if ((kk >> 21) == b1) {
        if (kk > tau) atomicAdd(&seg_gt[i / kSegKeys], 1u);
        else if (kk == tau && need_eq) atomicAdd(&seg_eq[i / kSegKeys], 1u);
      }
    });
  }
  __syncthreads();
  if (warp == 0) {
    // Exclusive prefix sums over the (at most 64) segments, two per lane.
    uint32_t g[2], e[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int s = h * 32 + lane;
      g[h] = s < static_cast<int>(nseg) ? __ldcg(&w[kStSeg + s]) + seg_gt[s] : 0u;
      e[h] = s < static_cast<int>(nseg) ? seg_eq[s] : 0u;
    }
    uint32_t carry_g = 0u, carry_e = 0u;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t ig = g[h], ie = e[h];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t a = __shfl_up_sync(0xffffffffu, ig, o);
        const uint32_t b = __shfl_up_sync(0xffffffffu, ie, o);
        if (lane >= o) {
          ig += a;
          ie += b;
        }
      }
      const int s = h * 32 + lane;
      if (s < static_cast<int>(nseg)) {
        w[kStBase + 2 * s] = carry_g + ig - g[h];
        w[kStBase + 2 * s + 1] = carry_e + ie - e[h];
      }
      carry_g += __shfl_sync(0xffffffffu, ig, 31);
      carry_e += __shfl_sync(0xffffffffu, ie, 31);
    }
    if (lane == 0) {
      w[kStState + kSTau] = tau;
      w[kStState + kSNeed] = need_eq;
      w[kStState + kSMode] = kModeSelect;
    }
  }
}

__global__ void __launch_bounds__(kSegThreads, 2) topk_write_kernel(const TopkParams p) {
  constexpr int NW = kSegThreads / 32;
  constexpr int WORDS = kSegKeys / 32;  // 512
  // Word u*NW + warp covers segment columns (u*NW + warp)*32 + lane: the
  // ballots of (key > tau) and (key == tau), then the number of selected
  // columns before the word (this segment's offsets included).
  __shared__ uint32_t gt_bits[WORDS], eq_bits[WORDS];
  __shared__ uint32_t gt_pre[WORDS], eq_pre[WORDS];
  __shared__ uint2 warp_sums[NW];
  const int row = blockIdx.x;
  const int seg = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int lo, hi;
  row_range(p, row, &lo, &hi);
  const uint32_t* w = split_row(p, row);
  int32_t* dst = p.out + static_cast<int64_t>(row) * p.k;
  if (seg == 0) {
    const uint32_t nvalid = w[kStState + kSValid];
    const int nsel = nvalid < static_cast<uint32_t>(p.k) ? static_cast<int>(nvalid) : p.k;
    for (int i = nsel + tid; i < p.k; i += kSegThreads) dst[i] = -1;
  }
  const int s0 = seg * kSegKeys;
  const int cnt = min(hi - lo - s0, kSegKeys);
  if (cnt <= 0) return;
  const float* src = p.logits + static_cast<int64_t>(row) * p.ld + lo + s0;
  float x[kSegItems];
#pragma unroll
  for (int u = 0; u < kSegItems; ++u) {
    const int e = u * kSegThreads + tid;
    x[u] = e < cnt ? __ldg(src + e) : -INFINITY;
  }
  const uint32_t mode = w[kStState + kSMode];
  if (mode == kModeIota) {
    for (int i = tid; i < cnt; i += kSegThreads) dst[s0 + i] = lo + s0 + i;
    return;
  }
  const uint32_t tau = w[kStState + kSTau], need_eq = w[kStState + kSNeed];
#pragma unroll
  for (int u = 0; u < kSegItems; ++u) {
    const uint32_t kk = order_key(x[u]);
    const uint32_t g = __ballot_sync(0xffffffffu, kk > tau);
    const uint32_t e = need_eq ? __ballot_sync(0xffffffffu, kk == tau) : 0u;
    if (lane == 0) {
      gt_bits[u * NW + warp] = g;
      eq_bits[u * NW + warp] = e;
    }
  }
  __syncthreads();
  uint2 mine = make_uint2(0u, 0u);
  if (tid < WORDS) mine = make_uint2(__popc(gt_bits[tid]), __popc(eq_bits[tid]));
  uint2 total;
  const uint2 before = block_scan2<kSegThreads>(mine, warp_sums, &total);
  if (tid < WORDS) {
    gt_pre[tid] = w[kStBase + 2 * seg] + before.x;
    eq_pre[tid] = w[kStBase + 2 * seg + 1] + before.y;
  }
  __syncthreads();
  const uint32_t bit = 1u << lane, lt = bit - 1u;
#pragma unroll 4
  for (int u = 0; u < kSegItems; ++u) {
    const int wd = u * NW + warp;
    const uint32_t gm = gt_bits[wd], em = eq_bits[wd];
    if ((gm | em) == 0u) continue;  // nothing selected in these 32 columns
    const uint32_t gb = gt_pre[wd] + __popc(gm & lt);
    const uint32_t eb = eq_pre[wd] + __popc(em & lt);
    const int col = lo + s0 + u * kSegThreads + tid;
    if (gm & bit) dst[gb + min(eb, need_eq)] = col;
    else if ((em & bit) && eb < need_eq) dst[gb + eb] = col;
  }
}

template <int THREADS, int ITEMS, int MINB>
cudaError_t launch_row(const TopkParams& p, cudaStream_t s) {
  topk_row_kernel<THREADS, ITEMS, MINB><<<p.R, THREADS, 0, s>>>(p);
  return cudaGetLastError();
}

template <int THREADS, int ITEMS, int CL>
cudaError_t launch_reg(const TopkParams& p, cudaStream_t s) {
  auto kern = topk_reg_kernel<THREADS, ITEMS, CL>;
  if constexpr (CL == 1) {
    kern<<<p.R, THREADS, 0, s>>>(p);
    return cudaGetLastError();
  } else {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.R) * CL);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
  }
}

}  // namespace

int topk_bitmap_words(int max_row) { return (max_row + 31) / 32; }

bool topk_supported(int max_row) {
  const size_t stream_smem = sizeof(uint32_t) * (static_cast<size_t>(kHistBins) + 8192 +
                                                 2 * static_cast<size_t>(topk_bitmap_words(max_row)));
  return max_row >= 0 && stream_smem <= 232448;
}

// Longest row (in keys) the register-resident kernel takes.
constexpr int kTopkRegMaxRow = 1024 * 32 * 8;

bool topk_split_rows(int64_t rows, int64_t max_row) {
  return max_row > kSegKeys && max_row <= static_cast<int64_t>(kSplitSegs) * kSegKeys &&
         rows <= 512;
}

int topk_split_words(int64_t) {
  return (kStWords + 63) / 64 * 64;  // rows stay 256-byte aligned
}

template <int THREADS>
cudaError_t launch_stream(const TopkParams& p, cudaStream_t s) {
  const size_t cand = THREADS >= 1024 ? 8192 : 2048;
  const size_t smem = sizeof(uint32_t) * (static_cast<size_t>(kHistBins) + cand +
                                          2 * static_cast<size_t>(p.bitmap_words));
  if (smem > 232448) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(topk_stream_kernel<THREADS>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  topk_stream_kernel<THREADS><<<p.R, THREADS, smem, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_topk(const TopkParams& p, cudaStream_t s) {
  if (p.R <= 0) return cudaSuccess;
  const int S = p.S;
  if (p.split) {
    // Few long rows: every phase on (segment, row) grids, see the split path.
    // Only each row's histogram and state words start at zero.
    cudaError_t e = cudaMemset2DAsync(p.split, static_cast<size_t>(p.split_words) * sizeof(uint32_t),
                                      0, kStZeroWords * sizeof(uint32_t),
                                      static_cast<size_t>(p.R), s);
    if (e != cudaSuccess) return e;
    const int gather_smem = kSplitCand * static_cast<int>(sizeof(uint32_t));
    e = cudaFuncSetAttribute(topk_gather_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             gather_smem);
    if (e != cudaSuccess) return e;
    // Rows vary fastest: every row's first segment is scheduled before any
    // second one, and the empty tail segments of short rows come last.
    const dim3 grid(static_cast<unsigned>(p.R), (S + kSegKeys - 1) / kSegKeys);
    topk_hist_kernel<<<grid, kSegThreads, 0, s>>>(p);
    topk_gather_kernel<<<grid, kSegThreads, gather_smem, s>>>(p);
    topk_write_kernel<<<grid, kSegThreads, 0, s>>>(p);
    return cudaGetLastError();
  }
  // Short rows: keys in registers, one CTA per row, several rows per SM.
  if (S <= 4096) return launch_row<256, 16, 6>(p, s);
  if (S <= 8192) return launch_row<512, 16, 3>(p, s);
  if (S <= 16384) return launch_row<1024, 16, 1>(p, s);
  // Very long rows without split scratch: a cluster of register-resident CTAs per row.
  if (S > 65536 && S <= 131072) return launch_reg<1024, 32, 4>(p, s);
  if (S > 131072 && S <= kTopkRegMaxRow) return launch_reg<1024, 32, 8>(p, s);
  // Otherwise: 256-thread CTAs that stream the row (8 rows in flight per SM).
  return launch_stream<256>(p, s);
}

}  // namespace dsa
