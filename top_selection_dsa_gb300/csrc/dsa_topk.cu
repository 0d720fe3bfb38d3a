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
// key; -0.0 folded onto +0.0; -inf and NaN below every valid score).  The
// exact k-th largest key tau is found by a radix select over the key bits
// (11 + 11 + 10), after which every key > tau and the first need_eq keys ==
// tau (in column order) are taken, in ascending column order.
//
// Kernels (dispatch in launch_topk):
//   topk_rows_kernel   one 256-thread CTA per row, rows of up to 262144
//       columns in 4096-key chunks.  A one-chunk row lives in registers:
//       radix passes over registers, then ballots and per-warp counts place
//       every selected column.  A longer row is read twice (histogram, then a
//       pass that marks the keys above the threshold bin in a shared-memory
//       bitmap and gathers the threshold bin's keys); the exact threshold
//       comes from the gathered keys, and a scan of the bitmap writes the
//       columns out.
//   split path         few long rows (decode): every phase on a grid of
//       (row, 4096-key unit) CTAs that talk through per-row scratch.
//   topk_stream_kernel rows longer than the others take: 256 threads per
//       row stream the row with 16-byte loads for each pass.
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

// Over hist[0..NBINS) (unpadded, 16-byte aligned), the bin b holding the r-th
// largest element, as find_bin; also that bin's count, and the sum of all bins
// is returned.  Thread t sums the PER bins [NBINS-(t+1)*PER, NBINS-t*PER)
// (lower threads hold higher bins); a warp scan and one exchange of warp
// totals give each thread its exclusive prefix.  Two barriers; wsum holds
// THREADS/32 words.
template <int THREADS, int NBINS>
__device__ __forceinline__ uint32_t find_bin_fast(const uint32_t* hist, uint32_t r, uint32_t* wsum,
                                                  uint32_t* sel, uint32_t* bin, uint32_t* above,
                                                  uint32_t* count) {
  constexpr int PER = NBINS / THREADS;
  constexpr int NW = THREADS / 32;
  static_assert(PER >= 1 && NBINS % THREADS == 0, "bins per thread");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int first = NBINS - (tid + 1) * PER;
  uint32_t v[PER];
  if constexpr (PER % 4 == 0) {
#pragma unroll
    for (int j = 0; j < PER / 4; ++j) {
      const uint4 q = reinterpret_cast<const uint4*>(hist + first)[j];
      v[4 * j] = q.x;
      v[4 * j + 1] = q.y;
      v[4 * j + 2] = q.z;
      v[4 * j + 3] = q.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < PER; ++j) v[j] = hist[first + j];
  }
  uint32_t local = 0u;
#pragma unroll
  for (int j = 0; j < PER; ++j) local += v[j];
  uint32_t incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  uint32_t before = 0u, total = 0u;
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    const uint32_t t = wsum[w];
    if (w < warp) before += t;
    total += t;
  }
  const uint32_t excl = before + incl - local;
  if (excl < r && r <= excl + local) {
    // One thread: walk its run again, highest bin first.
    uint32_t acc = excl;
    for (int j = PER - 1; j >= 0; --j) {
      const uint32_t h = hist[first + j];
      if (acc + h >= r) {
        sel[0] = static_cast<uint32_t>(first + j);
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
  return total;
}

// Programmatic dependent launch: the next kernel of the stream may start
// once every CTA of this one has run launch_dependents; it runs
// grid_dependency_wait (which returns once this grid has completed and its
// writes are visible) before reading anything this grid writes.  Both are
// no-ops for a kernel launched without the attribute.
__device__ __forceinline__ void launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ------------------------------------------------------------ bitmap rows

// One CTA of THREADS threads per row, the row taken in chunks of THREADS*16
// keys.  In chunk q, lane l of warp w holds the columns
// q*CH + w*512 + g*128 + j*32 + l (g, j = 0..3): every load is a
// warp-contiguous 128-byte line, and the ballot of the 32 lanes for (g, j)
// is exactly the selection-bitmap word of those columns.  A row of one chunk
// stays in registers; longer rows are read again for every pass (from L2).
//
//   pass 1   histogram of the top 11 key bits -> the bin b1 holding rank k;
//   pass 2   keys above bin b1 are selected (bitmap words written by
//            ballot of float compares against the bin's bounds); the keys
//            of bin b1 are marked in a second bitmap, whose columns a scan
//            then lists, and their keys are read again by column;
//   refine   bits 20..10, then 9..0, of the gathered keys -> tau and the
//            number need_eq of keys == tau to take; the selected candidates
//            are added to the bitmap (keys == tau to a second bitmap);
//   emit     a scan over the bitmap words gives each word its output offset
//            (keys == tau are taken in column order up to need_eq), and each
//            word's set bits are written out in order.
// When bin b1 holds more keys than the candidate list, digits 2 and 3 are
// found by two more passes over the row and one pass marks the bitmaps.
//
// Keys map -inf, NaN and the padding slots to one value, kNoKey (0x007FFFFF,
// the key of -inf), below every valid key (>= 0x00800000); in the first
// digit they all land in bin 3, which is left out.
constexpr uint32_t kNoKey = 0x007FFFFFu;
constexpr int kChunkMax = 64;  // chunks per row: rows of up to 64 * 4096 keys

__device__ __forceinline__ uint32_t chunk_key(float x) {
  const float y = fmaxf(x, -INFINITY) + 0.0f;  // NaN -> -inf, -0 -> +0
  const uint32_t u = __float_as_uint(y);
  return u ^ (static_cast<uint32_t>(static_cast<int32_t>(u) >> 31) | 0x80000000u);
}

// The float whose chunk_key is `key`.  For x not NaN, x > key_float(t) holds
// exactly when chunk_key(x) > t, for any t but 0x7FFFFFFF (the key -0.0
// would have: no key takes that value, so 0x7FFFFFFE stands in for it), and
// x == key_float(t) exactly when chunk_key(x) == t, for t the key of some
// value.  A NaN compares false, as its key, kNoKey, is below every bound.
// Past the key of +inf the result is a NaN, which no x exceeds.  Subnormal
// bounds and values compare exactly because this file is built without
// flush-to-zero (no -ftz / --use_fast_math).
__device__ __forceinline__ float key_float(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}
__device__ __forceinline__ float key_float_gt(uint32_t key) {
  return key_float(key == 0x7FFFFFFFu ? 0x7FFFFFFEu : key);
}

// Keys of chunk q for this thread: key[4g + j].
template <int THREADS>
__device__ __forceinline__ void load_chunk(const float* src, int n, int q, int warp, int lane,
                                           uint32_t (&key)[16]) {
  constexpr int CH = THREADS * 16;
  const int c0 = q * CH + warp * 512 + lane;
  if ((q + 1) * CH <= n) {
#pragma unroll
    for (int i = 0; i < 16; ++i) key[i] = chunk_key(__ldg(src + c0 + i * 32));
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int c = c0 + i * 32;
      key[i] = c < n ? chunk_key(__ldg(src + c)) : kNoKey;
    }
  }
}

// The raw values of chunk q for this thread (-inf past the row): loads only,
// so that they can be issued a chunk ahead of their use.
template <int THREADS>
__device__ __forceinline__ void load_chunk_raw(const float* src, int n, int q, int warp, int lane,
                                               float (&x)[16]) {
  constexpr int CH = THREADS * 16;
  const int c0 = q * CH + warp * 512 + lane;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int c = c0 + i * 32;
    x[i] = c < n ? __ldg(src + c) : -INFINITY;
  }
}

// Lines of this warp's share of chunk q into L1 (lanes 0-15, one 128-byte
// line each), ahead of its loads.
template <int THREADS>
__device__ __forceinline__ void prefetch_chunk_l1(const float* src, int n, int q, int warp, int lane) {
  constexpr int CH = THREADS * 16;
  const int c = q * CH + warp * 512 + lane * 32;
  if (lane < 16 && c < n)
    asm volatile("prefetch.global.L1 [%0];" ::"l"(reinterpret_cast<uint64_t>(src + c)));
}

// As load_chunk_raw, without per-element checks on whole chunks.
template <int THREADS>
__device__ __forceinline__ void load_chunk_f(const float* src, int n, int q, int warp, int lane,
                                             float (&x)[16]) {
  constexpr int CH = THREADS * 16;
  const int c0 = q * CH + warp * 512 + lane;
  if ((q + 1) * CH <= n) {
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = __ldg(src + c0 + i * 32);
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int c = c0 + i * 32;
      x[i] = c < n ? __ldg(src + c) : -INFINITY;
    }
  }
}

// Groups of this warp in chunk q that hold a column of the row (warp-uniform).
template <int THREADS>
__device__ __forceinline__ int chunk_groups(int n, int q, int warp) {
  const int first = q * THREADS * 16 + warp * 512;
  return min(max((n - first + 127) >> 7, 0), 4);
}

// Bitmap word of (chunk q, warp, item i = 4g + j).
template <int THREADS>
__device__ __forceinline__ int chunk_word(int q, int warp, int i) {
  return q * (THREADS / 2) + warp * 16 + i;
}

// Shared-memory words the kernel needs for rows of up to max_row columns and
// a candidate list of `cand` keys.
template <int THREADS>
__host__ __device__ constexpr int bitmap_row_words(int max_row) {
  return (max_row + THREADS * 16 - 1) / (THREADS * 16) * (THREADS / 2);
}

template <int THREADS, int MINB>
__global__ void __launch_bounds__(THREADS, MINB) topk_rows_kernel(const TopkParams p, int cand_cap,
                                                                    int words) {
  constexpr int NW = THREADS / 32;
  constexpr int CH = THREADS * 16;
  extern __shared__ __align__(16) uint32_t smem[];
  uint32_t* hist = smem;                        // kHistBins
  // cand_key and cand_col are contiguous: with cand_cap >= 1024 their
  // 2 * cand_cap words also hold a 2048-bin histogram, or the staged output.
  uint32_t* cand_key = hist + kHistBins;        // cand_cap: low 21 key bits (or a 2nd histogram)
  uint32_t* cand_col = cand_key + cand_cap;     // cand_cap: columns
  uint32_t* sel_bits = cand_col + cand_cap;     // words
  uint32_t* eq_bits = sel_bits + words;         // words
  __shared__ __align__(16) uint32_t wsum[NW];
  __shared__ uint2 warp_sums[NW];
  __shared__ uint32_t sel[4];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // Last row first: under a causal mask the rows grow with their index, so
  // the longest rows are scheduled first and the short ones fill the tail
  // (causal T=4096 prefill: 0.031 -> 0.029 ms).
  const int row = p.R - 1 - static_cast<int>(blockIdx.x);
  int lo, hi;
  row_range(p, row, &lo, &hi);
  const int n = hi - lo;
  const float* src = p.logits + static_cast<int64_t>(row) * p.ld + lo;
  int32_t* dst = p.out + static_cast<int64_t>(row) * p.k;
  const int nch = (n + CH - 1) / CH;
  const uint32_t lt = (1u << lane) - 1u;
  // Launched as a programmatic dependent of the kernel that wrote the logits
  // (when there is one): everything above overlaps its tail.
  grid_dependency_wait();

  if (n <= p.k) {
    // Every valid key is taken; all of them valid (x > -inf is false for
    // -inf and NaN alone): lo, lo+1, ...
    uint32_t nv = 0u;
    for (int c = tid; c < n; c += THREADS * 2) {
      nv += __ldg(src + c) > -INFINITY ? 1u : 0u;
      if (c + THREADS < n) nv += __ldg(src + c + THREADS) > -INFINITY ? 1u : 0u;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) nv += __shfl_xor_sync(0xffffffffu, nv, o);
    if (lane == 0) wsum[warp] = nv;
    __syncthreads();
    uint32_t all = 0u;
#pragma unroll
    for (int w = 0; w < NW; ++w) all += wsum[w];
    if (all == static_cast<uint32_t>(n)) {
      for (int i = tid; i < p.k; i += THREADS) dst[i] = i < n ? lo + i : -1;
      return;
    }
  }

  uint32_t key[16];
  if (nch == 1) load_chunk<THREADS>(src, n, 0, warp, lane, key);

  uint32_t tau = kNoKey, need_eq = 0u;  // keys > tau, then need_eq keys == tau
  int nsel;
  bool marked = false;                  // bitmaps already complete (gather path)
  if (n <= p.k) {
    uint32_t all = 0u;
#pragma unroll
    for (int w = 0; w < NW; ++w) all += wsum[w];
    nsel = static_cast<int>(all);  // every valid key
  } else {
    for (int i = tid; i < kHistBins / 4; i += THREADS)
      reinterpret_cast<uint4*>(hist)[i] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    // Pass 1: the top 11 key bits (bin 3 collects the invalid slots).  A row
    // of several chunks is read from memory (HBM) here: the next chunk's
    // loads are issued before the current chunk's histogram adds.  (The later
    // passes re-read the row from L2, where prefetching did not pay.)
    if (nch == 1) {
      const int ng = chunk_groups<THREADS>(n, 0, warp);
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (i / 4 < ng) atomicAdd(&hist[key[i] >> 21], 1u);
    } else {
      float nx[16];
      load_chunk_raw<THREADS>(src, n, 0, warp, lane, nx);
      for (int q = 0; q < nch; ++q) {
#pragma unroll
        for (int i = 0; i < 16; ++i) key[i] = chunk_key(nx[i]);
        if (q + 1 < nch) load_chunk_raw<THREADS>(src, n, q + 1, warp, lane, nx);
        const int ng = chunk_groups<THREADS>(n, q, warp);
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (i / 4 < ng) atomicAdd(&hist[key[i] >> 21], 1u);
      }
    }
    __syncthreads();
    // Read before the barriers of find_bin_fast, hence before any clear.
    // Bin 3 lies below every valid bin, so rank k of a row with more than k
    // valid keys is found above it.
    const uint32_t invalid = hist[3];
    uint32_t b1, above, c1;
    const uint32_t nvalid =
        find_bin_fast<THREADS, kHistBins>(hist, static_cast<uint32_t>(p.k), wsum, sel, &b1,
                                          &above, &c1) - invalid;
    if (nvalid <= static_cast<uint32_t>(p.k)) {
      nsel = static_cast<int>(nvalid);  // every valid key
    } else {
      nsel = p.k;
      uint32_t rem = static_cast<uint32_t>(p.k) - above;
      if (rem == c1) {
        tau = (b1 << 21) - 1u;  // the whole bin is taken
      } else if (nch > 1 && c1 <= static_cast<uint32_t>(cand_cap)) {
        // Pass 2, by float compares against the bounds of bin b1 (no key
        // transform): keys above the bin go straight into the selection
        // bitmap, the bin's own keys into a second one (eq_bits for now).
        const uint32_t thr = ((b1 + 1u) << 21) - 1u;
        const float f_hi = key_float_gt(thr), f_lo = key_float(b1 << 21);
        for (int q = 0; q < nch; ++q) {
          float x[16];
          load_chunk_f<THREADS>(src, n, q, warp, lane, x);
          if (q + 1 < nch) prefetch_chunk_l1<THREADS>(src, n, q + 1, warp, lane);
          const int ng = chunk_groups<THREADS>(n, q, warp);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            if (i / 4 >= ng) continue;  // words of later groups lie past the row
            const bool up = x[i] > f_hi;
            const uint32_t g = __ballot_sync(0xffffffffu, up);
            const uint32_t e = __ballot_sync(0xffffffffu, !up && x[i] >= f_lo);
            if (lane == 0) {
              sel_bits[chunk_word<THREADS>(q, warp, i)] = g;
              eq_bits[chunk_word<THREADS>(q, warp, i)] = e;
            }
          }
        }
        __syncthreads();
        // The bin's columns to the candidate list in column order: thread t
        // takes a run of words (and clears them for the marks below), a scan
        // gives its first slot.  Then their keys, read again by column.
        const int nwords = (n + 31) >> 5;
        const int per = (nwords + THREADS - 1) / THREADS;
        const int w0 = min(tid * per, nwords), w1 = min(w0 + per, nwords);
        uint32_t mine = 0u;
        for (int w = w0; w < w1; ++w) mine += __popc(eq_bits[w]);
        uint2 gathered;
        uint32_t slot = block_scan2<THREADS>(make_uint2(mine, 0u), warp_sums, &gathered).x;
        for (int w = w0; w < w1; ++w) {
          uint32_t f = eq_bits[w];
          eq_bits[w] = 0u;
          while (f) {
            const int b = __ffs(static_cast<int>(f)) - 1;
            if (slot < static_cast<uint32_t>(cand_cap))
              cand_col[slot] = static_cast<uint32_t>(w * 32 + b);
            ++slot;
            f &= f - 1u;
          }
        }
        const int nc = min(static_cast<int>(gathered.x), cand_cap);
        __syncthreads();
#pragma unroll 4
        for (int i = tid; i < nc; i += THREADS)
          cand_key[i] = chunk_key(__ldg(src + cand_col[i])) & 0x1FFFFFu;
        // Refine over the c1 gathered keys: bits 20..10, then 9..0.
        for (int i = tid; i < kHistBins / 4; i += THREADS)
          reinterpret_cast<uint4*>(hist)[i] = make_uint4(0u, 0u, 0u, 0u);
        __syncthreads();
        for (int i = tid; i < nc; i += THREADS) atomicAdd(&hist[cand_key[i] >> 10], 1u);
        __syncthreads();
        uint32_t b2, a2, c2;
        find_bin_fast<THREADS, kHistBins>(hist, rem, wsum, sel, &b2, &a2, &c2);
        rem -= a2;
        uint32_t low;  // low 21 bits of tau
        if (rem == c2) {
          low = (b2 << 10) - 1u;  // b2 > 0 here, since rem < c1
        } else {
          for (int i = tid; i < 1024 / 4; i += THREADS)
            reinterpret_cast<uint4*>(hist)[i] = make_uint4(0u, 0u, 0u, 0u);
          __syncthreads();
          for (int i = tid; i < nc; i += THREADS) {
            const uint32_t ck = cand_key[i];
            if ((ck >> 10) == b2) atomicAdd(&hist[ck & 1023u], 1u);
          }
          __syncthreads();
          uint32_t b3, a3, c3;
          find_bin_fast<THREADS, 1024>(hist, rem, wsum, sel, &b3, &a3, &c3);
          low = (b2 << 10) | b3;
          need_eq = rem - a3;
        }
        tau = (b1 << 21) | low;
        for (int i = tid; i < nc; i += THREADS) {
          const uint32_t kk = (b1 << 21) | cand_key[i];
          const uint32_t col = cand_col[i];
          if (kk > tau) atomicOr(&sel_bits[col >> 5], 1u << (col & 31u));
          else if (kk == tau && need_eq) atomicOr(&eq_bits[col >> 5], 1u << (col & 31u));
        }
        marked = true;
      } else {
        // Digits 2 and 3 from the keys (registers, or the row again).  The
        // second histogram lives in the candidate space (2 * cand_cap >= 2048 words).
        uint32_t* h2 = cand_key;
        for (int i = tid; i < kHistBins / 4; i += THREADS)
          reinterpret_cast<uint4*>(h2)[i] = make_uint4(0u, 0u, 0u, 0u);
        for (int q = 0; q < nch; ++q) {
          if (nch > 1) load_chunk<THREADS>(src, n, q, warp, lane, key);
          const int ng = chunk_groups<THREADS>(n, q, warp);
          __syncthreads();  // h2 cleared (first chunk)
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const uint32_t kk = key[i];
            if (i / 4 < ng && (kk >> 21) == b1) atomicAdd(&h2[(kk >> 10) & 2047u], 1u);
          }
        }
        // hist is free again: cleared for digit 3 meanwhile.
        for (int i = tid; i < 1024 / 4; i += THREADS)
          reinterpret_cast<uint4*>(hist)[i] = make_uint4(0u, 0u, 0u, 0u);
        __syncthreads();
        uint32_t b2, a2, c2;
        find_bin_fast<THREADS, kHistBins>(h2, rem, wsum, sel, &b2, &a2, &c2);
        rem -= a2;
        const uint32_t prefix = (b1 << 11) | b2;
        if (rem == c2) {
          tau = (prefix << 10) - 1u;
        } else {
          for (int q = 0; q < nch; ++q) {
            if (nch > 1) load_chunk<THREADS>(src, n, q, warp, lane, key);
            const int ng = chunk_groups<THREADS>(n, q, warp);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const uint32_t kk = key[i];
              if (i / 4 < ng && (kk >> 10) == prefix) atomicAdd(&hist[kk & 1023u], 1u);
            }
          }
          __syncthreads();
          uint32_t b3, a3, c3;
          find_bin_fast<THREADS, 1024>(hist, rem, wsum, sel, &b3, &a3, &c3);
          tau = (prefix << 10) | b3;
          need_eq = rem - a3;
        }
      }
    }
  }

  if (nch == 1) {
    // One chunk, in registers: warp w owns columns [w*512, (w+1)*512) in
    // item order; per-warp counts give each warp its output offset.
    const int ng = chunk_groups<THREADS>(n, 0, warp);
    uint32_t cg = 0u, ce = 0u;
#pragma unroll
    for (int i = 0; i < 16; ++i) cg += key[i] > tau ? 1u : 0u;
    if (need_eq) {
#pragma unroll
      for (int i = 0; i < 16; ++i) ce += key[i] == tau ? 1u : 0u;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      cg += __shfl_xor_sync(0xffffffffu, cg, o);
      ce += __shfl_xor_sync(0xffffffffu, ce, o);
    }
    __syncthreads();  // every reader of warp_sums / wsum is done
    if (lane == 0) warp_sums[warp] = make_uint2(cg, ce);
    __syncthreads();
    uint32_t grun = 0u, erun = 0u;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      if (w < warp) {
        grun += warp_sums[w].x;
        erun += warp_sums[w].y;
      }
    }
    const int col0 = lo + warp * 512 + lane;
    if (need_eq == 0u) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        if (i / 4 < ng) {
          const bool g = key[i] > tau;
          const uint32_t m = __ballot_sync(0xffffffffu, g);
          if (g) dst[grun + __popc(m & lt)] = col0 + i * 32;
          grun += __popc(m);
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        if (i / 4 < ng) {
          const bool g = key[i] > tau, e = key[i] == tau;
          const uint32_t mg = __ballot_sync(0xffffffffu, g);
          const uint32_t me = __ballot_sync(0xffffffffu, e);
          const uint32_t gb = grun + __popc(mg & lt), eb = erun + __popc(me & lt);
          if (g) dst[gb + min(eb, need_eq)] = col0 + i * 32;
          else if (e && eb < need_eq) dst[gb + eb] = col0 + i * 32;
          grun += __popc(mg);
          erun += __popc(me);
        }
      }
    }
    for (int i = nsel + tid; i < p.k; i += THREADS) dst[i] = -1;
    return;
  }

  // Several chunks: bitmaps (unless the gather path filled them), then the
  // emit.  Words of groups past the row are never read.
  if (!marked) {
    // Float compares against tau's value (tau is a key of the row whenever
    // need_eq > 0).
    const float f_gt = key_float_gt(tau), f_eq = key_float(tau);
    for (int q = 0; q < nch; ++q) {
      float x[16];
      load_chunk_f<THREADS>(src, n, q, warp, lane, x);
      if (q + 1 < nch) prefetch_chunk_l1<THREADS>(src, n, q + 1, warp, lane);
      const int ng = chunk_groups<THREADS>(n, q, warp);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        if (i / 4 < ng) {
          const uint32_t g = __ballot_sync(0xffffffffu, x[i] > f_gt);
          const uint32_t e = need_eq ? __ballot_sync(0xffffffffu, x[i] == f_eq) : 0u;
          if (lane == 0) {
            sel_bits[chunk_word<THREADS>(q, warp, i)] = g;
            eq_bits[chunk_word<THREADS>(q, warp, i)] = e;
          }
        }
      }
    }
  }
  __syncthreads();
  // Thread t walks the words [t*per, (t+1)*per) of the row.  The columns go
  // through shared memory (the candidate space is dead by now) when k fits,
  // so that the global stores are coalesced.
  uint32_t* stage = cand_key;
  const bool staged = p.k <= 2 * cand_cap;
  {
    const int nwords = (n + 31) >> 5;
    const int per = (nwords + THREADS - 1) / THREADS;
    const int w0 = min(tid * per, nwords), w1 = min(w0 + per, nwords);
    uint2 mine = make_uint2(0u, 0u);
    for (int w = w0; w < w1; ++w) {
      mine.x += __popc(sel_bits[w]);
      mine.y += __popc(eq_bits[w]);
    }
    uint2 total;
    uint2 before = block_scan2<THREADS>(mine, warp_sums, &total);
    for (int w = w0; w < w1; ++w) {
      const uint32_t s = sel_bits[w];
      uint32_t e = eq_bits[w];
      const uint32_t ecount = __popc(e);
      if (e) {
        // Keys == tau are taken in column order until need_eq of them.
        const uint32_t room = need_eq > before.y ? need_eq - before.y : 0u;
        uint32_t keep = 0u;
        for (uint32_t t = 0; t < room && e; ++t) {
          const uint32_t b = e & (0u - e);
          keep |= b;
          e ^= b;
        }
        e = keep;
      }
      uint32_t f = s | e;
      uint32_t pos = before.x + min(before.y, need_eq);
      while (f) {
        const int b = __ffs(static_cast<int>(f)) - 1;
        const int col = lo + w * 32 + b;
        if (staged) stage[pos] = static_cast<uint32_t>(col);
        else dst[pos] = col;
        ++pos;
        f &= f - 1u;
      }
      before.x += __popc(s);
      before.y += ecount;
    }
  }
  if (staged) {
    __syncthreads();
    if ((p.k & 3) == 0 && (reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {
      // Four columns a store (the output row is 16-byte aligned).
      for (int i = 4 * tid; i < p.k; i += 4 * THREADS) {
        uint4 v = *reinterpret_cast<const uint4*>(stage + i);
        if (i + 3 >= nsel) {
          v.x = i < nsel ? v.x : 0xFFFFFFFFu;
          v.y = i + 1 < nsel ? v.y : 0xFFFFFFFFu;
          v.z = i + 2 < nsel ? v.z : 0xFFFFFFFFu;
          v.w = i + 3 < nsel ? v.w : 0xFFFFFFFFu;
        }
        *reinterpret_cast<uint4*>(dst + i) = v;
      }
    } else {
      for (int i = tid; i < p.k; i += THREADS) dst[i] = i < nsel ? static_cast<int>(stage[i]) : -1;
    }
  } else {
    for (int i = nsel + tid; i < p.k; i += THREADS) dst[i] = -1;
  }
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
// Few long rows (decode): every phase runs on a grid of (row, 4096-key unit)
// CTAs of 256 threads, each holding its unit in registers in the chunk
// layout of topk_rows_kernel.  The phases talk through per-row scratch:
//   hist[2048]          first-digit histogram of the row's valid keys
//   state[16]           mode, tau, need_eq, nvalid, b1, rem, completion
//                       counters, ncand
//   above[kSplitUnits]  per unit: keys above the threshold (bin b1, or tau)
//   base[2*kSplitUnits] per unit: selected keys > tau and == tau before it
//   cand[kSplitCand]    keys of bin b1: low 21 key bits, the unit above them
// Only hist and state are zeroed before the first phase.  Phases (one launch
// each, no CTA ever waits for another):
//   hist    units add their histograms; the last unit CTA of a row to finish
//           (a completion counter after a fence) finds bin b1 and the row's
//           mode;
//   gather  units count their keys above bin b1 and append the keys of bin
//           b1; the last one of a row refines those to tau and need_eq
//           (streaming the row when bin b1 holds more than kSplitCand keys)
//           and turns the per-unit counts into every unit's output offsets;
//   write   each unit places its selected columns at its offsets, in column
//           order; unit 0 writes the -1 tail.
constexpr int kUnitThreads = 256;
constexpr int kUnitKeys = kUnitThreads * 16;  // 4096
constexpr int kSplitUnits = 256;              // rows of up to 256 * 4096 keys
constexpr int kSplitMaxRows = 512;
constexpr int kSplitCand = 16384;
constexpr int kStateWords = 16;
constexpr int kStHist = 0, kStState = kHistBins, kStAbove = kStState + kStateWords,
              kStBase = kStAbove + kSplitUnits, kStCand = kStBase + 2 * kSplitUnits,
              kStWords = kStCand + kSplitCand;
constexpr int kStZeroWords = kHistBins + kStateWords;  // zeroed before the first phase
// state words
constexpr int kSMode = 0, kSTau = 1, kSNeed = 2, kSValid = 3, kSB1 = 4, kSRem = 5,
              kSDoneHist = 6, kSDoneGather = 7, kSNcand = 8;
// Rows after the first phase: every valid key taken in place (iota); tau
// known (select); the keys of bin b1 to be gathered and refined (gather), or,
// too many of them, the row to be streamed (stream).
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

// The split path's work items: every (row, unit) whose unit holds keys, and
// unit 0 of each empty row (whose state and -1 row still have to be
// written), row-major.  Each phase runs a grid of resident CTAs that take
// items blockIdx.x, blockIdx.x + gridDim.x, ... so that no CTA is spent on
// the empty tail units of short rows.  pre[r] (shared, R + 1 entries) = the
// items of rows before r; returns their total.  Every thread must call it.
__device__ __forceinline__ int split_items(const TopkParams& p, int* pre, uint2* warp_sums) {
  const int tid = threadIdx.x;
  int cnt[2] = {0, 0};
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int row = 2 * tid + j;
    if (row < p.R) {
      int lo, hi;
      row_range(p, row, &lo, &hi);
      cnt[j] = hi > lo ? (hi - lo + kUnitKeys - 1) / kUnitKeys : 1;
    }
  }
  uint2 total;
  const uint32_t before =
      block_scan2<kUnitThreads>(make_uint2(static_cast<uint32_t>(cnt[0] + cnt[1]), 0u),
                                warp_sums, &total).x;
  if (2 * tid < p.R) pre[2 * tid] = static_cast<int>(before);
  if (2 * tid + 1 < p.R) pre[2 * tid + 1] = static_cast<int>(before) + cnt[0];
  if (tid == 0) pre[p.R] = static_cast<int>(total.x);
  __syncthreads();
  return static_cast<int>(total.x);
}

// Item -> (row, unit): the largest row with pre[row] <= item.
__device__ __forceinline__ void split_item(const int* pre, int R, int item, int* row, int* unit) {
  int lo_r = 0, hi_r = R;
  while (hi_r - lo_r > 1) {
    const int mid = (lo_r + hi_r) >> 1;
    if (pre[mid] <= item) lo_r = mid; else hi_r = mid;
  }
  *row = lo_r;
  *unit = item - pre[lo_r];
}

__global__ void __launch_bounds__(kUnitThreads, 5) topk_unit_hist_kernel(const TopkParams p) {
  constexpr int NW = kUnitThreads / 32;
  __shared__ __align__(16) uint32_t hist[kHistBins];
  __shared__ __align__(16) uint32_t wsum[NW];
  __shared__ uint32_t sel[4];
  __shared__ uint32_t flag;
  __shared__ int pre[kSplitMaxRows + 1];
  __shared__ uint2 scan_sums[NW];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int items = split_items(p, pre, scan_sums);
  // After the library's scoring kernel this phase is its programmatic
  // dependent: the logits (and the scratch cleared before it) are read only
  // once it has completed (a no-op for a plain launch).  The gather phase,
  // which loads logits before its own wait, may start only after that.
  grid_dependency_wait();
  launch_dependents();
  for (int item = blockIdx.x; item < items; item += gridDim.x) {
  int row, unit;
  split_item(pre, p.R, item, &row, &unit);
  __syncthreads();  // the previous item's readers of shared memory are done
  int lo, hi;
  row_range(p, row, &lo, &hi);
  const int n = hi - lo;
  const int c0 = unit * kUnitKeys;
  const int cnt = min(n - c0, kUnitKeys);
  uint32_t* w = split_row(p, row);
  if (cnt <= 0) {
    if (tid == 0) {  // empty row: nothing to select
      w[kStState + kSMode] = kModeIota;
      w[kStState + kSValid] = 0u;
    }
    continue;
  }
  uint32_t key[16];
  load_chunk<kUnitThreads>(p.logits + static_cast<int64_t>(row) * p.ld + lo + c0, cnt, 0, warp,
                           lane, key);
  for (int i = tid; i < kHistBins / 4; i += kUnitThreads)
    reinterpret_cast<uint4*>(hist)[i] = make_uint4(0u, 0u, 0u, 0u);
  __syncthreads();
  const int ng = chunk_groups<kUnitThreads>(cnt, 0, warp);
#pragma unroll
  for (int i = 0; i < 16; ++i)
    if (i / 4 < ng) atomicAdd(&hist[key[i] >> 21], 1u);
  __syncthreads();
  uint32_t* g = w + kStHist;
  // Bin 3 holds the invalid slots (kNoKey) alone: it is left out.
  for (int i = tid; i < kHistBins; i += kUnitThreads) {
    const uint32_t v = hist[i];
    if (v && i != 3) atomicAdd(&g[i], v);
  }
  const uint32_t nunits = static_cast<uint32_t>((n + kUnitKeys - 1) / kUnitKeys);
  if (!last_to_arrive(&w[kStState + kSDoneHist], nunits, &flag)) continue;
  // The row's histogram is complete: find the threshold bin once.
  for (int i = tid; i < kHistBins; i += kUnitThreads) hist[i] = __ldcg(&g[i]);
  __syncthreads();
  uint32_t b1, above, c1;
  const uint32_t nvalid = find_bin_fast<kUnitThreads, kHistBins>(
      hist, static_cast<uint32_t>(p.k), wsum, sel, &b1, &above, &c1);
  if (tid == 0) {
    w[kStState + kSValid] = nvalid;
    if (nvalid <= static_cast<uint32_t>(p.k)) {
      // Every valid key is taken: tau = kNoKey.
      w[kStState + kSMode] = nvalid == static_cast<uint32_t>(n) ? kModeIota : kModeSelect;
      w[kStState + kSTau] = kNoKey;
    } else {
      const uint32_t rem = static_cast<uint32_t>(p.k) - above;
      w[kStState + kSB1] = b1;
      w[kStState + kSRem] = rem;
      if (rem == c1) {  // the whole bin is taken
        w[kStState + kSMode] = kModeSelect;
        w[kStState + kSTau] = (b1 << 21) - 1u;
      } else {
        w[kStState + kSMode] = c1 <= static_cast<uint32_t>(kSplitCand) ? kModeGather : kModeStream;
      }
    }
  }
  }
}

__global__ void __launch_bounds__(kUnitThreads, 4) topk_unit_gather_kernel(const TopkParams p) {
  constexpr int NW = kUnitThreads / 32;
  __shared__ __align__(16) uint32_t hist[kHistBins];
  __shared__ __align__(16) uint32_t wsum[NW];
  __shared__ uint2 warp_sums[NW];
  __shared__ uint32_t sel[4];
  __shared__ uint32_t flag, cta_hits, cta_base;
  __shared__ uint32_t stage[kUnitKeys];  // this unit's candidates
  __shared__ uint32_t unit_gt[kSplitUnits], unit_eq[kSplitUnits];
  __shared__ int pre[kSplitMaxRows + 1];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  launch_dependents();
  const int items = split_items(p, pre, warp_sums);
  for (int item = blockIdx.x; item < items; item += gridDim.x) {
  int row, unit;
  split_item(pre, p.R, item, &row, &unit);
  __syncthreads();  // the previous item's readers of shared memory are done
  int lo, hi;
  row_range(p, row, &lo, &hi);
  const int n = hi - lo;
  const int c0 = unit * kUnitKeys;
  const int cnt = min(n - c0, kUnitKeys);
  if (cnt <= 0) continue;
  uint32_t* w = split_row(p, row);
  const float* row_src = p.logits + static_cast<int64_t>(row) * p.ld + lo;
  uint32_t key[16];
  load_chunk<kUnitThreads>(row_src + c0, cnt, 0, warp, lane, key);
  grid_dependency_wait();  // the histogram phase is complete
  const uint32_t mode = w[kStState + kSMode];
  if (mode == kModeIota) continue;
  const uint32_t b1 = w[kStState + kSB1];
  // Keys above `thr` are taken whatever the refinement finds; keys of bin
  // `want` (none unless gathering) are the candidates.
  const uint32_t thr = mode == kModeSelect ? w[kStState + kSTau] : ((b1 + 1u) << 21) - 1u;
  const uint32_t want = mode == kModeGather ? b1 : 0xFFFFFFFFu;
  if (tid == 0) cta_hits = 0u;
  __syncthreads();
  const int ng = chunk_groups<kUnitThreads>(cnt, 0, warp);
  const uint32_t lt = (1u << lane) - 1u;
  uint32_t nab = 0u;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    if (i / 4 >= ng) continue;
    const uint32_t kk = key[i];
    nab += kk > thr ? 1u : 0u;  // kNoKey is never above thr (>= kNoKey)
    const bool hit = (kk >> 21) == want;
    const uint32_t m = __ballot_sync(0xffffffffu, hit);
    if (m) {
      uint32_t slot = 0u;
      if (lane == 0) slot = atomicAdd(&cta_hits, static_cast<uint32_t>(__popc(m)));
      slot = __shfl_sync(0xffffffffu, slot, 0) + __popc(m & lt);
      if (hit) stage[slot] = (static_cast<uint32_t>(unit) << 21) | (kk & kLow21);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) nab += __shfl_xor_sync(0xffffffffu, nab, o);
  if (lane == 0) wsum[warp] = nab;
  __syncthreads();
  if (tid == 0) {
    uint32_t a = 0u;
#pragma unroll
    for (int i = 0; i < NW; ++i) a += wsum[i];
    w[kStAbove + unit] = a;
    cta_base = cta_hits ? atomicAdd(&w[kStState + kSNcand], cta_hits) : 0u;
  }
  __syncthreads();
  {
    const uint32_t nh = cta_hits, base = cta_base;
    uint32_t* cand = w + kStCand;
    for (uint32_t i = tid; i < nh; i += kUnitThreads)
      if (base + i < static_cast<uint32_t>(kSplitCand)) cand[base + i] = stage[i];
  }
  const uint32_t nunits = static_cast<uint32_t>((n + kUnitKeys - 1) / kUnitKeys);
  if (!last_to_arrive(&w[kStState + kSDoneGather], nunits, &flag)) continue;

  // Last gather CTA of the row: tau / need_eq, then the offsets of every
  // unit's selected columns.
  for (int i = tid; i < kSplitUnits; i += kUnitThreads) {
    unit_gt[i] = 0u;
    unit_eq[i] = 0u;
  }
  uint32_t tau = thr, need_eq = 0u;
  if (mode == kModeGather || mode == kModeStream) {
    const bool gathered = mode == kModeGather;
    const uint32_t* cand = w + kStCand;
    const int nc = gathered ? min(static_cast<int>(__ldcg(&w[kStState + kSNcand])), kSplitCand) : 0;
    const int nq = (n + kUnitKeys - 1) / kUnitKeys;
    uint32_t rem = w[kStState + kSRem];
    // Calls fn(low 21 bits, unit) for every key of bin b1.  Gathered keys
    // pass through shared memory (`stage`) kUnitKeys at a time, loaded once
    // when they all fit.
    const bool resident = nc <= kUnitKeys;
    auto stage_from = [&](int base) {
      const int m = min(nc - base, kUnitKeys);
      __syncthreads();  // earlier readers of stage are done
      uint32_t v[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int i = tid + j * kUnitThreads;
        v[j] = i < m ? __ldcg(&cand[base + i]) : 0u;
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int i = tid + j * kUnitThreads;
        if (i < m) stage[i] = v[j];
      }
      __syncthreads();
    };
    if (gathered && resident) stage_from(0);
    auto for_each_in_bin = [&](auto&& fn) {
      if (gathered) {
        for (int base = 0; base < nc; base += kUnitKeys) {
          if (!resident) stage_from(base);
          const int m = min(nc - base, kUnitKeys);
          for (int i = tid; i < m; i += kUnitThreads) {
            const uint32_t c = stage[i];
            fn(c & kLow21, c >> 21);
          }
        }
      } else {
        for (int q = 0; q < nq; ++q) {
          load_chunk<kUnitThreads>(row_src, n, q, warp, lane, key);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if ((key[i] >> 21) == b1) fn(key[i] & kLow21, static_cast<uint32_t>(q));
        }
      }
    };
    __syncthreads();
    for (int i = tid; i < kHistBins / 4; i += kUnitThreads)
      reinterpret_cast<uint4*>(hist)[i] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    for_each_in_bin([&](uint32_t low, uint32_t) { atomicAdd(&hist[low >> 10], 1u); });
    __syncthreads();
    uint32_t b2, a2, c2;
    find_bin_fast<kUnitThreads, kHistBins>(hist, rem, wsum, sel, &b2, &a2, &c2);
    rem -= a2;
    uint32_t low;
    if (rem == c2) {
      low = (b2 << 10) - 1u;  // b2 > 0 here, since rem < c1
    } else {
      for (int i = tid; i < 1024 / 4; i += kUnitThreads)
        reinterpret_cast<uint4*>(hist)[i] = make_uint4(0u, 0u, 0u, 0u);
      __syncthreads();
      for_each_in_bin([&](uint32_t lw, uint32_t) {
        if ((lw >> 10) == b2) atomicAdd(&hist[lw & 1023u], 1u);
      });
      __syncthreads();
      uint32_t b3, a3, c3;
      find_bin_fast<kUnitThreads, 1024>(hist, rem, wsum, sel, &b3, &a3, &c3);
      low = (b2 << 10) | b3;
      need_eq = rem - a3;
    }
    tau = (b1 << 21) | low;
    for_each_in_bin([&](uint32_t lw, uint32_t u) {
      const uint32_t kk = (b1 << 21) | lw;
      if (kk > tau) atomicAdd(&unit_gt[u], 1u);
      else if (kk == tau && need_eq) atomicAdd(&unit_eq[u], 1u);
    });
  }
  __syncthreads();
  // Exclusive prefix over the units (at most kSplitUnits = kUnitThreads).
  uint2 mine = make_uint2(0u, 0u);
  if (tid < static_cast<int>(nunits))
    mine = make_uint2(__ldcg(&w[kStAbove + tid]) + unit_gt[tid], unit_eq[tid]);
  uint2 total;
  const uint2 before = block_scan2<kUnitThreads>(mine, warp_sums, &total);
  if (tid < static_cast<int>(nunits)) {
    w[kStBase + 2 * tid] = before.x;
    w[kStBase + 2 * tid + 1] = before.y;
  }
  if (tid == 0) {
    w[kStState + kSTau] = tau;
    w[kStState + kSNeed] = need_eq;
    w[kStState + kSMode] = kModeSelect;
  }
  }
}

__global__ void __launch_bounds__(kUnitThreads, 5) topk_unit_write_kernel(const TopkParams p) {
  constexpr int NW = kUnitThreads / 32;
  __shared__ uint2 warp_cnt[NW];
  __shared__ uint2 scan_sums[NW];
  __shared__ int pre[kSplitMaxRows + 1];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int items = split_items(p, pre, scan_sums);
  for (int item = blockIdx.x; item < items; item += gridDim.x) {
  int row, unit;
  split_item(pre, p.R, item, &row, &unit);
  __syncthreads();  // the previous item's readers of warp_cnt are done
  int lo, hi;
  row_range(p, row, &lo, &hi);
  const int n = hi - lo;
  const uint32_t* w = split_row(p, row);
  int32_t* dst = p.out + static_cast<int64_t>(row) * p.k;
  const int c0 = unit * kUnitKeys;
  const int cnt = min(n - c0, kUnitKeys);
  uint32_t key[16];
  if (cnt > 0)
    load_chunk<kUnitThreads>(p.logits + static_cast<int64_t>(row) * p.ld + lo + c0, cnt, 0, warp,
                             lane, key);
  grid_dependency_wait();  // the gather phase is complete
  if (unit == 0) {
    const uint32_t nvalid = w[kStState + kSValid];
    const int nsel = nvalid < static_cast<uint32_t>(p.k) ? static_cast<int>(nvalid) : p.k;
    for (int i = nsel + tid; i < p.k; i += kUnitThreads) dst[i] = -1;
  }
  if (cnt <= 0) continue;
  const uint32_t mode = w[kStState + kSMode];
  if (mode == kModeIota) {
    for (int i = tid; i < cnt; i += kUnitThreads) dst[c0 + i] = lo + c0 + i;
    continue;
  }
  const uint32_t tau = w[kStState + kSTau], need_eq = w[kStState + kSNeed];
  const int ng = chunk_groups<kUnitThreads>(cnt, 0, warp);
  uint32_t cg = 0u, ce = 0u;
#pragma unroll
  for (int i = 0; i < 16; ++i) cg += key[i] > tau ? 1u : 0u;
  if (need_eq) {
#pragma unroll
    for (int i = 0; i < 16; ++i) ce += key[i] == tau ? 1u : 0u;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    cg += __shfl_xor_sync(0xffffffffu, cg, o);
    ce += __shfl_xor_sync(0xffffffffu, ce, o);
  }
  if (lane == 0) warp_cnt[warp] = make_uint2(cg, ce);
  __syncthreads();
  // Selected columns of earlier units, then of earlier warps, come first.
  uint32_t grun = w[kStBase + 2 * unit], erun = w[kStBase + 2 * unit + 1];
#pragma unroll
  for (int i = 0; i < NW; ++i) {
    if (i < warp) {
      grun += warp_cnt[i].x;
      erun += warp_cnt[i].y;
    }
  }
  const uint32_t lt = (1u << lane) - 1u;
  const int col0 = lo + c0 + warp * 512 + lane;
  if (need_eq == 0u) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i / 4 < ng) {
        const bool g = key[i] > tau;
        const uint32_t m = __ballot_sync(0xffffffffu, g);
        if (g) dst[grun + __popc(m & lt)] = col0 + i * 32;
        grun += __popc(m);
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i / 4 < ng) {
        const bool g = key[i] > tau, e = key[i] == tau;
        const uint32_t mg = __ballot_sync(0xffffffffu, g);
        const uint32_t me = __ballot_sync(0xffffffffu, e);
        const uint32_t gb = grun + __popc(mg & lt), eb = erun + __popc(me & lt);
        if (g) dst[gb + min(eb, need_eq)] = col0 + i * 32;
        else if (e && eb < need_eq) dst[gb + eb] = col0 + i * 32;
        grun += __popc(mg);
        erun += __popc(me);
      }
    }
  }
  }
}

// ------------------------------------------------------------- score order
//
// torch_dsa_topk takes torch.topk, whose indices come in descending order of
// score; the canonical output here is ascending column order.  This pass
// puts each row back into score order: one CTA per row sorts 64-bit
// composites (score key << 32 | ~column) descending with a bitonic network in
// shared memory, so that equal scores keep the lower column first and the
// -1 padding (composite 0) stays at the tail.
constexpr int kSortThreads = 256;

__global__ void __launch_bounds__(kSortThreads) topk_sort_kernel(const float* __restrict__ logits,
                                                                 int64_t ld, int32_t* topk, int k,
                                                                 int n, uint32_t* err) {
  extern __shared__ __align__(16) unsigned long long sk[];  // n = k rounded up to a power of two
  const int row = blockIdx.x, tid = threadIdx.x;
  int32_t* r = topk + static_cast<int64_t>(row) * k;
  const float* lg = logits + static_cast<int64_t>(row) * ld;
  bool bad = false;
  for (int i = tid; i < n; i += kSortThreads) {
    unsigned long long v = 0ull;
    if (i < k) {
      const int c = r[i];
      if (c >= 0 && c < ld) {
        // Invalid scores (-inf, NaN) get key 0: after every valid one.
        const uint32_t key = order_key(__ldg(lg + c));
        v = (static_cast<unsigned long long>(key) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(c));
      } else if (c >= 0) {
        bad = true;  // past the row: treated as padding, never read
      }
    }
    sk[i] = v;
  }
  if (bad) record_error(err, kErrBadIndex);
  __syncthreads();
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = tid; i < n / 2; i += kSortThreads) {
        const int a = 2 * i - (i & (stride - 1));
        const int b = a + stride;
        const bool desc = (a & size) == 0;
        const unsigned long long x = sk[a], y = sk[b];
        if ((x < y) == desc) {
          sk[a] = y;
          sk[b] = x;
        }
      }
      __syncthreads();
    }
  }
  for (int i = tid; i < k; i += kSortThreads) {
    const unsigned long long v = sk[i];
    r[i] = v ? static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(v)) : -1;
  }
}

// ------------------------------------------------------------ rank merge
//
// Decode context parallelism (KimiK3DSAIndexer.__init__ on the vLLM page:
// each rank scores its interleaved share of the key cache, takes a local
// top-k, and the op merges the ranks' local top-k into the global one): the
// merge of C candidates per row (score, global column; column < 0 = empty)
// into the k best by (score descending, column ascending), written in
// ascending column order with -1 padding.  One CTA per row: a bitonic sort of
// composites (key << 32 | ~column) puts the winners first, a second one puts
// their columns in ascending order.
constexpr int kMergeThreads = 512;

template <class K>
__device__ __forceinline__ void bitonic_desc(K* a, int n) {
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < n / 2; i += blockDim.x) {
        const int lo = 2 * i - (i & (stride - 1));
        const int hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const K x = a[lo], y = a[hi];
        if ((x < y) == desc) {
          a[lo] = y;
          a[hi] = x;
        }
      }
      __syncthreads();
    }
  }
}

// Candidates of row `row`: C = W * kr of them, candidate i at
// (i / kr) * rank_stride + row * kr + i % kr (W = 1, kr = C: a [T, C] array;
// rank_stride = T * kr: [W, T, kr] rank-major, as an all-gather leaves them).
__global__ void __launch_bounds__(kMergeThreads) topk_merge_kernel(
    const float* __restrict__ scores, const int32_t* __restrict__ cols, int C, int kr,
    int64_t rank_stride, int n, int k, int m, int32_t* __restrict__ out) {
  extern __shared__ __align__(16) unsigned long long mk[];  // n composites
  const int row = blockIdx.x;
  __shared__ uint32_t nvalid;
  if (threadIdx.x == 0) nvalid = 0u;
  __syncthreads();
  uint32_t mine = 0u;
  for (int i = threadIdx.x; i < n; i += kMergeThreads) {
    unsigned long long v = 0ull;
    if (i < C) {
      const int w = i / kr;
      const int64_t off = w * rank_stride + static_cast<int64_t>(row) * kr + (i - w * kr);
      const int c = __ldg(cols + off);
      const uint32_t key = c >= 0 ? order_key(__ldg(scores + off)) : 0u;  // -inf / NaN: never taken
      if (key != 0u) {
        v = (static_cast<unsigned long long>(key) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(c));
        ++mine;
      }
    }
    mk[i] = v;
  }
  if (mine) atomicAdd(&nvalid, mine);
  __syncthreads();
  bitonic_desc(mk, n);
  // The winners' columns (the first min(k, valid) composites), ascending.
  const int take = min(k, static_cast<int>(nvalid));
  uint32_t* col = reinterpret_cast<uint32_t*>(mk + n);  // m words after the composites
  for (int i = threadIdx.x; i < m; i += kMergeThreads)
    col[i] = i < take ? 0xFFFFFFFFu - static_cast<uint32_t>(mk[i]) : 0xFFFFFFFFu;
  __syncthreads();
  // Descending sort of the complements = ascending columns; padding (~0 -> 0) last.
  for (int i = threadIdx.x; i < m; i += kMergeThreads) col[i] = ~col[i];
  __syncthreads();
  bitonic_desc(col, m);
  int32_t* dst = out + static_cast<int64_t>(row) * k;
  for (int i = threadIdx.x; i < k; i += kMergeThreads)
    dst[i] = i < take ? static_cast<int32_t>(~col[i]) : -1;
}

}  // namespace

int topk_bitmap_words(int max_row) { return (max_row + 31) / 32; }

bool topk_supported(int max_row) {
  const size_t stream_smem = sizeof(uint32_t) * (static_cast<size_t>(kHistBins) + 8192 +
                                                 2 * static_cast<size_t>(topk_bitmap_words(max_row)));
  return max_row >= 0 && stream_smem <= 232448;
}

// Few long rows (at most 512, some longer than 16384 columns): from 32 rows
// on, one 1024-thread CTA per row (rows of up to kChunkMax * 4096 columns);
// fewer rows, or longer ones, take the split path, which spreads each row
// over many CTAs.
constexpr int kWideRowsMin = 32;

bool topk_wide_rows(int64_t rows, int64_t max_row) {
  return max_row > 16384 && max_row <= static_cast<int64_t>(kChunkMax) * 4096 &&
         rows >= kWideRowsMin && rows <= kSplitMaxRows;
}

bool topk_split_rows(int64_t rows, int64_t max_row) {
  return max_row > 16384 && max_row <= static_cast<int64_t>(kSplitUnits) * kUnitKeys &&
         rows <= kSplitMaxRows && !topk_wide_rows(rows, max_row);
}

int topk_split_words(int64_t) {
  return (kStWords + 63) / 64 * 64;  // rows stay 256-byte aligned
}

cudaError_t topk_split_clear(uint32_t* split, int split_words, int rows, cudaStream_t s) {
  return cudaMemset2DAsync(split, static_cast<size_t>(split_words) * sizeof(uint32_t), 0,
                           kStZeroWords * sizeof(uint32_t), static_cast<size_t>(rows), s);
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
    // Few long rows: every phase on (row, unit) grids, see the split path.
    // Only each row's histogram and state words start at zero: cleared here,
    // or, in the composed calls, before the scoring kernel, so that the first
    // phase can start as that kernel's programmatic dependent.
    cudaError_t e = cudaSuccess;
    if (!p.after_score) {
      e = topk_split_clear(p.split, p.split_words, p.R, s);
      if (e != cudaSuccess) return e;
    }
    // Each phase: at most as many CTAs as are resident at once (their launch
    // bounds), each walking the row-major list of units that hold keys.
    const int64_t units = static_cast<int64_t>(p.R) * ((S + kUnitKeys - 1) / kUnitKeys);
    const int sms = device_sm_count() > 0 ? device_sm_count() : 1;
    auto grid_of = [&](int per_sm) {
      return dim3(static_cast<unsigned>(std::min<int64_t>(units, static_cast<int64_t>(sms) * per_sm)));
    };
    // The later phases (and the first one after the library's own scoring
    // kernel) start early and wait for the previous kernel in hardware
    // before reading what it wrote.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid_of(5);
    cfg.blockDim = dim3(kUnitThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.after_score ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, topk_unit_hist_kernel, p);
    if (e != cudaSuccess) return e;
    cfg.gridDim = grid_of(4);
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, topk_unit_gather_kernel, p);
    if (e != cudaSuccess) return e;
    cfg.gridDim = grid_of(5);
    return cudaLaunchKernelEx(&cfg, topk_unit_write_kernel, p);
  }
  // Few long rows: one 1024-thread CTA per row, the row in 16384-key chunks
  // (16 loads in flight per thread), 4096 candidates.  On 128 paged-decode
  // rows of up to 131072 keys this takes 0.044 ms against 0.051 for the
  // split path, and 0.059 against 0.148 on 128 full 131072-key rows; below 32
  // rows the split path's many CTAs per row win (8 rows: 0.038 vs 0.058).
  if (topk_wide_rows(p.R, S)) {
    const int cand = 4096;
    const int words = bitmap_row_words<1024>(S);
    const int smem = (kHistBins + 2 * cand + 2 * words) * static_cast<int>(sizeof(uint32_t));
    cudaError_t e = cudaFuncSetAttribute(topk_rows_kernel<1024, 1>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.R));
    cfg.blockDim = dim3(1024);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = s;
    // A programmatic dependent of the scoring kernel only, as below.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.after_score ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, topk_rows_kernel<1024, 1>, p, cand, words);
  }
  // One 256-thread CTA per row, the row in 4096-key chunks.
  if (S <= kChunkMax * 4096) {
    // 2048 candidates (the threshold bin of a 32768-key row holds up to about
    // 2 K keys; a larger bin takes the digit passes): 32 KB of shared memory
    // per CTA up to 32768 columns, so the register limit of five CTAs per SM
    // is the binding one.
    const int cand = 2048;
    const int words = bitmap_row_words<256>(S);
    const int smem = (kHistBins + 2 * cand + 2 * words) * static_cast<int>(sizeof(uint32_t));
    cudaError_t e = cudaFuncSetAttribute(topk_rows_kernel<256, 5>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.R));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = s;
    // A programmatic dependent of the scoring kernel only: the kernel reads
    // its row range before griddepcontrol.wait.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.after_score ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, topk_rows_kernel<256, 5>, p, cand, words);
  }
  // Otherwise: 256-thread CTAs that stream the row (8 rows in flight per SM).
  return launch_stream<256>(p, s);
}

cudaError_t launch_topk_sort(const float* logits, int64_t ld, int32_t* topk, int T, int k,
                             uint32_t* err, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  int n = 1;
  while (n < k) n <<= 1;
  const int smem = n * static_cast<int>(sizeof(unsigned long long));
  cudaError_t e = cudaFuncSetAttribute(topk_sort_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       smem);
  if (e != cudaSuccess) return e;
  topk_sort_kernel<<<T, kSortThreads, smem, s>>>(logits, ld, topk, k, n, err);
  return cudaGetLastError();
}

cudaError_t launch_topk_merge(const float* scores, const int32_t* cols, int T, int W, int kr,
                              int k, int32_t* out, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  const int C = W * kr;
  int n = 1;
  while (n < C) n <<= 1;
  int m = 1;
  while (m < k) m <<= 1;
  const int smem = n * static_cast<int>(sizeof(unsigned long long)) +
                   m * static_cast<int>(sizeof(uint32_t));
  cudaError_t e = cudaFuncSetAttribute(topk_merge_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  topk_merge_kernel<<<T, kMergeThreads, smem, s>>>(scores, cols, C, kr,
                                                   static_cast<int64_t>(T) * kr, n, k, m, out);
  return cudaGetLastError();
}

// Decode context parallelism: a rank's top-k indices (local columns, in
// place in cols) become (local score, global position) pairs.  The rank owns
// the runs of `inter` positions p with (p / inter) % W == rank, in order, so
// local column j is global ((j / inter) * W + rank) * inter + j % inter.
__global__ void dcp_pairs_kernel(const float* __restrict__ logits, int64_t ld, int T, int k,
                                 int rank, int W, int inter, float* __restrict__ scores,
                                 int32_t* __restrict__ cols) {
  const int64_t total = static_cast<int64_t>(T) * k;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int j = cols[i];
    if (j >= 0) {
      const int64_t t = i / k;
      scores[i] = logits[t * ld + j];
      const int64_t run = j / inter;
      cols[i] = static_cast<int32_t>((run * W + rank) * inter + (j - run * inter));
    } else {
      scores[i] = -INFINITY;
      cols[i] = -1;
    }
  }
}

cudaError_t launch_dcp_pairs(const float* logits, int64_t ld, int T, int k, int rank, int W,
                             int inter, float* scores, int32_t* cols, cudaStream_t s) {
  const int64_t total = static_cast<int64_t>(T) * k;
  if (total <= 0) return cudaSuccess;
  const int sms = device_sm_count() > 0 ? device_sm_count() : 1;
  const int64_t blocks = std::min<int64_t>((total + 255) / 256, static_cast<int64_t>(sms) * 8);
  dcp_pairs_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(logits, ld, T, k, rank, W, inter,
                                                                 scores, cols);
  return cudaGetLastError();
}

}  // namespace dsa
