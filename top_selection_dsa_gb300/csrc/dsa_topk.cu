// dsa_topk.cu -- masked per-row top-k of fp32 index logits (sm_103a).
//
// Semantics of torch_dsa_topk as corrected in GitHub "vllm-project/vime" pull
// request #502 (third review comment): only columns inside the row's range
// [row_start, row_end) count, a -inf score is never selected, and the row is
// padded with -1 when fewer than k valid columns exist.  Readings where the
// page is silent: ties go to the lower column (-0.0 equals +0.0), NaN is never
// selected, and the selected columns are written in ascending column order.
//
// One CTA per row:
//   1. every logit becomes an order-preserving 32-bit key (larger float ->
//      larger key; -0.0 folded onto +0.0; -inf and NaN -> 0, which no valid
//      score maps to) and, when the row fits, is cached in shared memory;
//   2. if at most k keys are valid, all of them are taken;
//   3. otherwise an exact radix select over the key bits (11 + 11 + 10) finds
//      the k-th largest key tau and how many keys equal to tau must be taken
//      (need_eq) after every key greater than tau;
//   4. one ordered pass over the row writes every key > tau and the first
//      need_eq keys == tau, at positions given by a block-wide prefix count,
//      which yields ascending column order directly; -1 fills the tail.
#include "dsa_common.cuh"
#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kItems = 4;  // consecutive columns per thread in the ordered pass
constexpr int kHistBins = 2048;

__device__ __forceinline__ uint32_t order_key(float x) {
  uint32_t u = __float_as_uint(x);
  if (u == 0x80000000u) u = 0u;                        // -0.0 -> +0.0
  const uint32_t key = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  const bool invalid = (x != x) || (u == 0xFF800000u);  // NaN or -inf
  return invalid ? 0u : key;
}

// Exclusive prefix sum of one value per thread over the block; *total gets
// the block sum.  Contains barriers: every thread must call it.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* warp_sums,
                                                         uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = lane < kWarps ? warp_sums[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kWarps) warp_sums[lane] = w;
  }
  __syncthreads();
  const uint32_t before = warp ? warp_sums[warp - 1] : 0u;
  *total = warp_sums[kWarps - 1];
  __syncthreads();
  return before + x - v;
}

// Over hist[0..nbins), find the bin b holding the r-th largest element
// (r >= 1): above = sum of bins > b satisfies above < r <= above + hist[b].
// Every thread returns the same (b, above).
__device__ __forceinline__ void find_bin(const uint32_t* hist, int nbins, uint32_t r,
                                         uint32_t* warp_sums, uint32_t* sel, uint32_t* bin,
                                         uint32_t* above) {
  const int per = nbins / kThreads;  // bins per thread, highest bins first
  const int top = nbins - 1 - threadIdx.x * per;
  uint32_t local = 0;
  for (int i = 0; i < per; ++i) local += hist[top - i];
  uint32_t total;
  const uint32_t excl = block_exclusive_scan(local, warp_sums, &total);
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
  __syncthreads();
}

__global__ void __launch_bounds__(kThreads) topk_kernel(const TopkParams p) {
  extern __shared__ uint32_t sm[];
  uint32_t* hist = sm;                 // kHistBins
  uint32_t* cache = sm + kHistBins;    // p.cache_cap keys
  __shared__ uint32_t warp_sums[32];
  __shared__ uint32_t sel[2];

  const int row = blockIdx.x;
  const int tid = threadIdx.x;
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
  const bool cached = n <= p.cache_cap;

  // Pass 1: keys (+ cache) and the histogram of their top 11 bits.
  for (int i = tid; i < kHistBins; i += kThreads) hist[i] = 0u;
  __syncthreads();
  for (int i = tid; i < n; i += kThreads) {
    const uint32_t key = order_key(src[i]);
    if (cached) cache[i] = key;
    atomicAdd(&hist[key >> 21], 1u);
  }
  __syncthreads();
  // Bin 0 holds exactly the invalid keys: the smallest valid key is 0x00800000.
  const int nvalid = n - static_cast<int>(hist[0]);
  __syncthreads();

  uint32_t tau = 0u;   // take every key > tau ...
  uint32_t need_eq = 0u;  // ... and the first need_eq keys == tau (column order)
  if (nvalid > p.k) {
    uint32_t rem = static_cast<uint32_t>(p.k);
    uint32_t b1, a1, b2, a2, b3, a3;
    find_bin(hist, kHistBins, rem, warp_sums, sel, &b1, &a1);
    rem -= a1;
    for (int i = tid; i < kHistBins; i += kThreads) hist[i] = 0u;
    __syncthreads();
    for (int i = tid; i < n; i += kThreads) {
      const uint32_t key = cached ? cache[i] : order_key(src[i]);
      if ((key >> 21) == b1) atomicAdd(&hist[(key >> 10) & 0x7FFu], 1u);
    }
    __syncthreads();
    find_bin(hist, kHistBins, rem, warp_sums, sel, &b2, &a2);
    rem -= a2;
    const uint32_t prefix = (b1 << 11) | b2;
    for (int i = tid; i < 1024; i += kThreads) hist[i] = 0u;
    __syncthreads();
    for (int i = tid; i < n; i += kThreads) {
      const uint32_t key = cached ? cache[i] : order_key(src[i]);
      if ((key >> 10) == prefix) atomicAdd(&hist[key & 0x3FFu], 1u);
    }
    __syncthreads();
    find_bin(hist, 1024, rem, warp_sums, sel, &b3, &a3);
    rem -= a3;
    tau = (prefix << 10) | b3;
    need_eq = rem;
  }

  // Ordered pass: ascending columns, positions from a block-wide prefix count.
  uint32_t base_gt = 0u, base_eq = 0u;
  for (int c0 = 0; c0 < n; c0 += kThreads * kItems) {
    const int i0 = c0 + tid * kItems;
    uint32_t keys[kItems];
    uint32_t n_gt = 0u, n_eq = 0u;
#pragma unroll
    for (int u = 0; u < kItems; ++u) {
      const int i = i0 + u;
      const uint32_t key = i < n ? (cached ? cache[i] : order_key(src[i])) : 0u;
      keys[u] = key;
      n_gt += key > tau ? 1u : 0u;
      n_eq += (need_eq > 0u && key == tau) ? 1u : 0u;
    }
    uint32_t total;
    const uint32_t excl = block_exclusive_scan(n_gt | (n_eq << 16), warp_sums, &total);
    uint32_t gb = base_gt + (excl & 0xFFFFu);
    uint32_t eb = base_eq + (excl >> 16);
#pragma unroll
    for (int u = 0; u < kItems; ++u) {
      const uint32_t key = keys[u];
      if (key > tau) {
        dst[gb + min(eb, need_eq)] = lo + i0 + u;
        ++gb;
      } else if (need_eq > 0u && key == tau) {
        if (eb < need_eq) dst[gb + eb] = lo + i0 + u;
        ++eb;
      }
    }
    base_gt += total & 0xFFFFu;
    base_eq += total >> 16;
  }
  const int nsel = nvalid < p.k ? nvalid : p.k;
  for (int i = nsel + tid; i < p.k; i += kThreads) dst[i] = -1;
}

}  // namespace

cudaError_t launch_topk(const TopkParams& p, cudaStream_t s) {
  if (p.R <= 0) return cudaSuccess;
  const size_t smem = sizeof(uint32_t) * (static_cast<size_t>(kHistBins) + p.cache_cap);
  cudaError_t e =
      cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  topk_kernel<<<p.R, kThreads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace dsa
