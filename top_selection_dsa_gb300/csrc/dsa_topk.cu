// dsa_topk.cu -- masked per-row top-k of fp32 index logits (sm_103a).
//
// Semantics of torch_dsa_topk as corrected in GitHub "vllm-project/vime" pull
// request #502 (third review comment): only columns inside the row's range
// [row_start, row_end) count, a -inf score is never selected, and the row is
// padded with -1 when fewer than k valid columns exist.  Readings where the
// page is silent: ties go to the lower column (-0.0 equals +0.0), NaN is never
// selected, and the selected columns are written in ascending column order.
//
// One 256-thread CTA per row; several rows share an SM, so the per-row
// barriers of one CTA overlap with the memory traffic of the others.
//   1. every logit becomes an order-preserving 32-bit key (larger float ->
//      larger key; -0.0 folded onto +0.0; -inf and NaN -> 0, which no valid
//      score maps to); pass 1 streams the row from HBM with 16-byte loads and
//      histograms the top 11 key bits;
//   2. if at most k keys are valid, every valid key is taken; otherwise two
//      more histogram passes (11 and 10 bits, re-reading the row, which is
//      now in L2) find the exact k-th largest key tau and how many keys equal
//      to tau to take (need_eq) after all keys greater than tau;
//   3. a last pass turns the row into two bitmaps (key > tau, key == tau) with
//      warp ballots; one prefix scan over the words gives every selected
//      column its output position, so indices come out in column order; the
//      first need_eq ties (in column order) are the ones kept; -1 fills the
//      tail of the output row.
#include "dsa_common.cuh"
#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kHistBins = 2048;

__device__ __forceinline__ uint32_t order_key(float x) {
  uint32_t u = __float_as_uint(x);
  if (u == 0x80000000u) u = 0u;                        // -0.0 -> +0.0
  const uint32_t key = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  const bool invalid = (x != x) || (u == 0xFF800000u);  // NaN or -inf
  return invalid ? 0u : key;
}

// Exclusive prefix sums of two counters per thread over the block.  Contains
// barriers: every thread must call it.
__device__ __forceinline__ uint2 block_exclusive_scan2(uint2 v, uint2* warp_sums, uint2* total) {
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
  for (int w = 0; w < kWarps; ++w) {
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

// Over hist[0..nbins), the bin b holding the r-th largest element (r >= 1):
// above = sum of bins > b satisfies above < r <= above + hist[b].  Every thread
// returns the same (b, above).
__device__ __forceinline__ void find_bin(const uint32_t* hist, int nbins, uint32_t r,
                                         uint2* warp_sums, uint32_t* sel, uint32_t* bin,
                                         uint32_t* above) {
  const int per = nbins / kThreads;  // bins per thread, highest bins first
  const int top = nbins - 1 - threadIdx.x * per;
  uint32_t local = 0;
  for (int i = 0; i < per; ++i) local += hist[top - i];
  uint2 total;
  const uint32_t excl = block_exclusive_scan2(make_uint2(local, 0u), warp_sums, &total).x;
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
}

__global__ void __launch_bounds__(kThreads) topk_kernel(const TopkParams p) {
  extern __shared__ uint32_t sm[];
  uint32_t* hist = sm;                   // kHistBins
  uint32_t* gt_bits = sm + kHistBins;    // ceil(S/32) words: key > tau
  uint32_t* eq_bits = gt_bits + p.bitmap_words;  // key == tau
  __shared__ uint2 warp_sums[kWarps];
  __shared__ uint32_t sel[2];

  const int row = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int lo, hi;
  if (p.context_lens) {
    const int b = row / p.next_n, j = row % p.next_n;
    const int end = p.context_lens[b] - p.next_n + j + 1;
    lo = 0;
    hi = min(max(end, 0), p.S);
  } else {
    lo = min(max(p.row_starts[row], 0), p.S);
    hi = min(max(p.row_ends[row], 0), p.S);
    if (hi < lo) hi = lo;
  }
  const int n = hi - lo;
  const float* src = p.logits + static_cast<int64_t>(row) * p.ld + lo;
  int32_t* dst = p.out + static_cast<int64_t>(row) * p.k;

  // ---- pass 1: histogram of the top 11 key bits, 16-byte loads from HBM.
  for (int i = tid; i < kHistBins; i += kThreads) hist[i] = 0u;
  __syncthreads();
  {
    const uintptr_t addr = reinterpret_cast<uintptr_t>(src);
    int head = (addr & 3u) ? n : static_cast<int>(((16u - (addr & 15u)) & 15u) >> 2);
    head = min(head, n);
    const int body = (n - head) >> 2;
    for (int i = tid; i < head; i += kThreads) atomicAdd(&hist[order_key(src[i]) >> 21], 1u);
    const float4* src4 = reinterpret_cast<const float4*>(src + head);
    for (int i = tid; i < body; i += kThreads) {
      const float4 v = __ldg(src4 + i);
      atomicAdd(&hist[order_key(v.x) >> 21], 1u);
      atomicAdd(&hist[order_key(v.y) >> 21], 1u);
      atomicAdd(&hist[order_key(v.z) >> 21], 1u);
      atomicAdd(&hist[order_key(v.w) >> 21], 1u);
    }
    for (int i = head + 4 * body + tid; i < n; i += kThreads)
      atomicAdd(&hist[order_key(src[i]) >> 21], 1u);
  }
  __syncthreads();
  // Bin 0 holds exactly the invalid keys: the smallest valid key is 0x00800000.
  const int nvalid = n - static_cast<int>(hist[0]);

  uint32_t tau = 0u;      // take every key > tau ...
  uint32_t need_eq = 0u;  // ... and the first need_eq keys == tau, in column order
  if (nvalid > p.k) {
    uint32_t rem = static_cast<uint32_t>(p.k);
    uint32_t b1, a1, b2, a2, b3, a3;
    find_bin(hist, kHistBins, rem, warp_sums, sel, &b1, &a1);
    rem -= a1;
    __syncthreads();
    for (int i = tid; i < kHistBins; i += kThreads) hist[i] = 0u;
    __syncthreads();
    for (int i = tid; i < n; i += kThreads) {
      const uint32_t key = order_key(src[i]);
      if ((key >> 21) == b1) atomicAdd(&hist[(key >> 10) & 0x7FFu], 1u);
    }
    __syncthreads();
    find_bin(hist, kHistBins, rem, warp_sums, sel, &b2, &a2);
    rem -= a2;
    const uint32_t prefix = (b1 << 11) | b2;
    __syncthreads();
    for (int i = tid; i < 1024; i += kThreads) hist[i] = 0u;
    __syncthreads();
    for (int i = tid; i < n; i += kThreads) {
      const uint32_t key = order_key(src[i]);
      if ((key >> 10) == prefix) atomicAdd(&hist[key & 0x3FFu], 1u);
    }
    __syncthreads();
    find_bin(hist, 1024, rem, warp_sums, sel, &b3, &a3);
    rem -= a3;
    tau = (prefix << 10) | b3;
    need_eq = rem;
  }

  // ---- last pass: bitmaps of (key > tau) and (key == tau), one word per
  // 32 consecutive columns, written by warp ballots.
  const int nwords = (n + 31) >> 5;
  for (int w = warp; w < nwords; w += kWarps) {
    const int i = (w << 5) + lane;
    const uint32_t key = i < n ? order_key(src[i]) : 0u;
    const uint32_t g = __ballot_sync(0xffffffffu, key > tau);
    const uint32_t e = __ballot_sync(0xffffffffu, need_eq > 0u && key == tau);
    if (lane == 0) {
      gt_bits[w] = g;
      eq_bits[w] = e;
    }
  }
  __syncthreads();

  // ---- positions: prefix counts over words (each thread owns a run of words).
  const int per = (nwords + kThreads - 1) / kThreads;
  const int w0 = min(tid * per, nwords), w1 = min(w0 + per, nwords);
  uint2 mine = make_uint2(0u, 0u);
  for (int w = w0; w < w1; ++w) {
    mine.x += __popc(gt_bits[w]);
    mine.y += __popc(eq_bits[w]);
  }
  uint2 total;
  const uint2 before = block_exclusive_scan2(mine, warp_sums, &total);
  uint32_t gb = before.x, eb = before.y;
  for (int w = w0; w < w1; ++w) {
    uint32_t g = gt_bits[w], e = eq_bits[w];
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
  const int nsel = nvalid < p.k ? nvalid : p.k;
  for (int i = nsel + tid; i < p.k; i += kThreads) dst[i] = -1;
}

}  // namespace

int topk_bitmap_words(int max_row) { return (max_row + 31) / 32; }

cudaError_t launch_topk(const TopkParams& p, cudaStream_t s) {
  if (p.R <= 0) return cudaSuccess;
  const size_t smem =
      sizeof(uint32_t) * (static_cast<size_t>(kHistBins) + 2 * static_cast<size_t>(p.bitmap_words));
  cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  topk_kernel<<<p.R, kThreads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace dsa
