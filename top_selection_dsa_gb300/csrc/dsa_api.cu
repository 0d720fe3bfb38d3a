// dsa_api.cu -- the C ABI declared in include/dsa.h: argument validation,
// TMA descriptor encoding, launches on the caller's stream, and the per-device
// error word that the kernels' bounded waits report into.
//
// Nothing here allocates device memory: outputs and scratch space belong to
// the caller.  Host-detectable errors return before any CUDA call is made.
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "dsa.h"

#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <vector>
#include "dsa_common.cuh"
#include "dsa_internal.h"

namespace dsa {

// Sticky error word of each device (bits kErrTimeout / kErrBadIndex).
__device__ uint32_t g_error_word;

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

constexpr int kMaxDevices = 64;

// Device address of g_error_word on the current device (looked up once per
// device), or null.
uint32_t* error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  static std::mutex mu;
  static uint32_t* addr[kMaxDevices] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, g_error_word) != cudaSuccess) return nullptr;
    addr[dev] = static_cast<uint32_t*>(a);
  }
  return addr[dev];
}

}  // namespace

// SM count of the current device (queried once per device).
int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  static std::mutex mu;
  static int count[kMaxDevices] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (count[dev] == 0 &&
      cudaDeviceGetAttribute(&count[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    count[dev] = 0;
  return count[dev];
}

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
bool pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }
cudaStream_t as_stream(dsa_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

dsa_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA; }

// An NVTX range named after the entry point around each call, so that a
// profiler's timeline shows which library call queued which kernels.  (With
// no tool attached an NVTX call returns at once.)
struct CallRange {
  explicit CallRange(const char* name) { nvtxRangePushA(name); }
  ~CallRange() { nvtxRangePop(); }
  CallRange(const CallRange&) = delete;
  CallRange& operator=(const CallRange&) = delete;
};

// 128-byte-swizzled tiled map over a row-major [rows, D] matrix (2-D) or a
// [blocks, block_rows, D] cache (3-D), box = 128 bytes of D x box_rows rows.
bool encode_map(CUtensorMap* map, const void* base, dsa_dtype_t dtype, int D, int64_t rows,
                int box_rows, int64_t blocks) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const int esz = dtype == DSA_BF16 ? 2 : 1;
  const CUtensorMapDataType dt =
      dtype == DSA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const cuuint32_t box_inner = 128 / esz;
  CUresult r;
  if (blocks <= 0) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * esz};
    const cuuint32_t box[2] = {box_inner, static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows),
                                static_cast<cuuint64_t>(blocks)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * esz,
                                   static_cast<cuuint64_t>(D) * esz * rows};
    const cuuint32_t box[3] = {box_inner, static_cast<cuuint32_t>(box_rows), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    r = fn(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  return r == CUDA_SUCCESS;
}

// 64-byte-swizzled tiled map over packed E2M1 rows [rows, 64 bytes], box =
// 64 bytes x box_rows rows (the MXFP4 operands, D = 128).
bool encode_map_e2m1(CUtensorMap* map, const void* base, int64_t rows, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {64, static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {64};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

// Workspace of the composed calls: the fp32 logits [rows, round_up(cols, 4)],
// padded to 256 bytes, then (split top-k path only) the per-row histograms.
size_t logits_scratch_bytes(int64_t rows, int64_t cols) {
  return static_cast<size_t>(round_up(
      rows * round_up(cols > 0 ? cols : 1, 4) * static_cast<int64_t>(sizeof(float)), 256));
}

size_t split_scratch_bytes(int64_t rows, int64_t cols) {
  return static_cast<size_t>(rows) * static_cast<size_t>(topk_split_words(cols)) *
         sizeof(uint32_t);
}

uint32_t* split_scratch(void* workspace, int64_t rows, int64_t cols) {
  if (!topk_split_rows(rows, cols)) return nullptr;
  return reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) +
                                     logits_scratch_bytes(rows, cols));
}

// The composed calls clear the split path's scratch (when they use it)
// before their scoring kernel, so that the top-k's first phase can start as
// that kernel's programmatic dependent.
cudaError_t clear_split(uint32_t* split, int64_t rows, int64_t cols, cudaStream_t st) {
  if (!split || rows == 0) return cudaSuccess;
  return topk_split_clear(split, topk_split_words(cols), static_cast<int>(rows), st);
}

// ---------------------------------------------------------------- validation

dsa_status_t check_elems(dsa_dtype_t dtype, int H, int D, const void* k_scale) {
  if (dtype != DSA_BF16 && dtype != DSA_E4M3) return DSA_ERR_INVALID_ARG;
  if (!pow2(H) || H > 64) return DSA_ERR_UNSUPPORTED;
  if (dtype == DSA_BF16 && D != 64 && D != 128) return DSA_ERR_UNSUPPORTED;
  if (dtype == DSA_E4M3 && D != 128) return DSA_ERR_UNSUPPORTED;
  if ((dtype == DSA_E4M3) != (k_scale != nullptr)) return DSA_ERR_INVALID_ARG;
  return DSA_OK;
}

dsa_status_t check_logits_args(const void* q, const float* q_scale, const void* k,
                               const float* k_scale, dsa_dtype_t dtype, const float* weights,
                               const int32_t* row_starts, const int32_t* row_ends, int T, int S,
                               int H, int D) {
  if (!q || !k || !weights || !row_starts || !row_ends) return DSA_ERR_INVALID_ARG;
  if (T < 0 || S < 0 || H < 1 || D < 1) return DSA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(weights, 4) || !aligned(row_starts, 4) ||
      !aligned(row_ends, 4) || (q_scale && !aligned(q_scale, 4)) ||
      (k_scale && !aligned(k_scale, 4)))
    return DSA_ERR_INVALID_ARG;
  dsa_status_t st = check_elems(dtype, H, D, k_scale);
  if (st != DSA_OK) return st;
  if (static_cast<int64_t>(T) * H >= (int64_t(1) << 31)) return DSA_ERR_UNSUPPORTED;
  return DSA_OK;
}

// Validated, unchecked launch of the prefill scoring kernel.
dsa_status_t run_logits(const void* q, const float* q_scale, const void* k, const float* k_scale,
                        dsa_dtype_t dtype, const float* weights, const int32_t* row_starts,
                        const int32_t* row_ends, int T, int S, int H, int D, float* logits,
                        int64_t ld, cudaStream_t st) {
  if (T == 0 || S == 0) return DSA_OK;
  ScoreParams p = {};
  if (!encode_map(&p.tmap_q, q, dtype, D, static_cast<int64_t>(T) * H, 256, 0) ||
      !encode_map(&p.tmap_k, k, dtype, D, S, 128, 0))
    return DSA_ERR_CUDA;
  p.weights = weights;
  p.q_scale = q_scale;
  p.k_scale = k_scale;
  p.row_starts = row_starts;
  p.row_ends = row_ends;
  p.logits = logits;
  p.ld = ld;
  p.R = T;
  p.S = S;
  p.err = error_word();
  if (!p.err) return DSA_ERR_CUDA;
  cudaError_t e = dtype == DSA_BF16 ? launch_score_prefill_bf16(p, H, D, st)
                                    : launch_score_prefill_fp8(p, H, D, st);
  return from_cuda(e);
}

dsa_status_t check_mx_args(const void* q, const uint8_t* q_sf, const void* k, const uint8_t* k_sf,
                           const float* weights, const int32_t* row_starts,
                           const int32_t* row_ends, int T, int S, int H, int D) {
  if (!q || !q_sf || !k || !k_sf || !weights || !row_starts || !row_ends)
    return DSA_ERR_INVALID_ARG;
  if (T < 0 || S < 0 || H < 1 || D < 1) return DSA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(q_sf, 4) || !aligned(k_sf, 4) ||
      !aligned(weights, 4) || !aligned(row_starts, 4) || !aligned(row_ends, 4))
    return DSA_ERR_INVALID_ARG;
  if (!score_mx_supported(H, D)) return DSA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(T) * H >= (int64_t(1) << 31)) return DSA_ERR_UNSUPPORTED;
  return DSA_OK;
}

// Validated, unchecked launch of the MXFP4 prefill scoring kernel.
dsa_status_t run_logits_mx(const void* q, const uint8_t* q_sf, const void* k,
                           const uint8_t* k_sf, const float* weights, const int32_t* row_starts,
                           const int32_t* row_ends, int T, int S, int H, float* logits,
                           int64_t ld, cudaStream_t st) {
  if (T == 0 || S == 0) return DSA_OK;
  ScoreParams p = {};
  if (!encode_map_e2m1(&p.tmap_q, q, static_cast<int64_t>(T) * H, score_mx_q_rows()) ||
      !encode_map_e2m1(&p.tmap_k, k, S, 128))
    return DSA_ERR_CUDA;
  p.weights = weights;
  p.row_starts = row_starts;
  p.row_ends = row_ends;
  p.logits = logits;
  p.ld = ld;
  p.R = T;
  p.S = S;
  p.err = error_word();
  if (!p.err) return DSA_ERR_CUDA;
  return from_cuda(launch_score_mx(p, q_sf, k_sf, st));
}

dsa_status_t run_topk(const float* logits, int64_t ld, const int32_t* row_starts,
                      const int32_t* row_ends, const int32_t* context_lens, int next_n, int R,
                      int S, int k, int32_t* out, cudaStream_t st, uint32_t* split,
                      bool after_score) {
  if (R == 0) return DSA_OK;
  TopkParams p = {};
  p.after_score = after_score ? 1 : 0;
  p.logits = logits;
  p.ld = ld;
  p.row_starts = row_starts;
  p.row_ends = row_ends;
  p.context_lens = context_lens;
  p.next_n = next_n;
  p.R = R;
  p.S = S;
  p.k = k;
  p.bitmap_words = topk_bitmap_words(S);
  p.out = out;
  p.split = split;
  p.split_words = split ? topk_split_words(S) : 0;
  return from_cuda(launch_topk(p, st));
}

struct PagedShape {
  int B, next_n, block_size, max_blocks, num_blocks, H, D;
};

dsa_status_t check_paged_args(const void* q, const float* q_scale, const float* weights,
                              const void* k_cache, const float* k_scale, dsa_dtype_t dtype,
                              const int32_t* block_table, const int32_t* context_lens,
                              const PagedShape& s) {
  if (!q || !weights || !k_cache || !block_table || !context_lens) return DSA_ERR_INVALID_ARG;
  if (s.B < 0 || s.next_n < 1 || s.max_blocks < 1 || s.num_blocks < 1 || s.H < 1 || s.D < 1)
    return DSA_ERR_INVALID_ARG;
  if (!pow2(s.block_size) || s.block_size < 8 || s.block_size > 128) return DSA_ERR_UNSUPPORTED;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(weights, 4) ||
      !aligned(block_table, 4) || !aligned(context_lens, 4) || (q_scale && !aligned(q_scale, 4)) ||
      (k_scale && !aligned(k_scale, 4)))
    return DSA_ERR_INVALID_ARG;
  dsa_status_t st = check_elems(dtype, s.H, s.D, k_scale);
  if (st != DSA_OK) return st;
  if (!score_paged_supported(dtype == DSA_E4M3, s.H, s.D, s.next_n)) return DSA_ERR_UNSUPPORTED;
  if (s.B > kMaxPagedRequests) return DSA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(s.max_blocks) * s.block_size >= (int64_t(1) << 30) ||
      static_cast<int64_t>(s.B) * s.next_n * s.H >= (int64_t(1) << 31))
    return DSA_ERR_UNSUPPORTED;
  return DSA_OK;
}

constexpr int kPagedChunkKeys = 2048;

dsa_status_t run_logits_paged(const void* q, const float* q_scale, const float* weights,
                              const void* k_cache, const float* k_scale, dsa_dtype_t dtype,
                              const int32_t* block_table, const int32_t* context_lens,
                              const PagedShape& s, float* logits, int64_t ld, cudaStream_t st) {
  if (s.B == 0) return DSA_OK;
  const int64_t R = static_cast<int64_t>(s.B) * s.next_n;
  const int max_ctx = s.max_blocks * s.block_size;
  ScoreParams p = {};
  // The q box must be exactly the kernel's N rows: the stage accounting
  // (expect_tx) and the shared-memory q region are sized for N.
  const int ncols = score_paged_cols(s.H, s.next_n);
  if (!encode_map(&p.tmap_q, q, dtype, s.D, R * s.H, ncols, 0) ||
      !encode_map(&p.tmap_k, k_cache, dtype, s.D, s.block_size, s.block_size, s.num_blocks))
    return DSA_ERR_CUDA;
  p.weights = weights;
  p.q_scale = q_scale;
  p.k_scale = k_scale;
  p.block_table = block_table;
  p.context_lens = context_lens;
  p.logits = logits;
  p.ld = ld;
  p.R = static_cast<int>(R);
  p.S = max_ctx;
  p.max_blocks = s.max_blocks;
  p.next_n = s.next_n;
  p.block_size = s.block_size;
  p.num_blocks = s.num_blocks;
  p.chunk_keys = kPagedChunkKeys;
  p.chunks_per_req = (max_ctx + kPagedChunkKeys - 1) / kPagedChunkKeys;
  p.err = error_word();
  if (!p.err) return DSA_ERR_CUDA;
  return from_cuda(launch_score_paged(p, dtype == DSA_E4M3, s.H, s.D, st));
}

// ------------------------------------------------------------ small kernels

__global__ void fill_kernel(float* dst, int64_t rows, int64_t cols, int64_t ld, float v) {
  const int64_t total = rows * cols;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    dst[(i / cols) * ld + (i % cols)] = v;
}

__global__ void wait_timeout_selftest_kernel(uint32_t* err, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  // Nothing ever arrives on `bar`: the bounded wait must give up.
  if (threadIdx.x == 0 && !mbar_wait_bounded(&bar, 0u, nullptr, timeout_ns))
    record_error(err, kErrTimeout);
}

}  // namespace

cudaError_t launch_fill(float* dst, int64_t rows, int64_t cols, int64_t ld, float value,
                        cudaStream_t s) {
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  const int64_t total = rows * cols;
  const int64_t want = (total + 255) / 256;
  const int grid = static_cast<int>(want < 152 * 16 ? want : 152 * 16);
  fill_kernel<<<grid, 256, 0, s>>>(dst, rows, cols, ld, value);
  return cudaGetLastError();
}

cudaError_t launch_wait_timeout_selftest(uint32_t* err, uint64_t timeout_ns, cudaStream_t s) {
  wait_timeout_selftest_kernel<<<1, 32, 0, s>>>(err, timeout_ns);
  return cudaGetLastError();
}

}  // namespace dsa

using namespace dsa;

extern "C" {

dsa_status_t dsa_indexer_logits(const void* q, const float* q_scale, const void* k,
                                const float* k_scale, dsa_dtype_t dtype, const float* weights,
                                const int32_t* row_starts, const int32_t* row_ends, int T, int S,
                                int H, int D, float* logits, int64_t ld, uint32_t flags,
                                dsa_stream_t stream) {
  const CallRange range("dsa_indexer_logits");
  dsa_status_t st = check_logits_args(q, q_scale, k, k_scale, dtype, weights, row_starts,
                                      row_ends, T, S, H, D);
  if (st != DSA_OK) return st;
  if (!logits || !aligned(logits, 4) || ld < S || ld < 1) return DSA_ERR_INVALID_ARG;
  if (flags & ~DSA_LOGITS_CLEAN) return DSA_ERR_INVALID_ARG;
  if (T == 0) return DSA_OK;
  if (flags & DSA_LOGITS_CLEAN) {
    st = from_cuda(launch_fill(logits, T, S, ld, -INFINITY, as_stream(stream)));
    if (st != DSA_OK) return st;
  }
  return run_logits(q, q_scale, k, k_scale, dtype, weights, row_starts, row_ends, T, S, H, D,
                    logits, ld, as_stream(stream));
}

dsa_status_t dsa_topk(const float* logits, int64_t ld, const int32_t* row_starts,
                      const int32_t* row_ends, int T, int S, int k, int32_t* out, void* workspace,
                      size_t ws_bytes, dsa_stream_t stream) {
  const CallRange range("dsa_topk");
  if (!logits || !row_starts || !row_ends || !out) return DSA_ERR_INVALID_ARG;
  if (T < 0 || S < 0 || k < 1 || ld < S || ld < 1) return DSA_ERR_INVALID_ARG;
  if (!aligned(logits, 4) || !aligned(out, 4) || !aligned(row_starts, 4) ||
      !aligned(row_ends, 4))
    return DSA_ERR_INVALID_ARG;
  if (!topk_supported(S)) return DSA_ERR_UNSUPPORTED;
  const size_t need = dsa_workspace_bytes(DSA_OP_TOPK, T, S, k);
  if (need > 0 && (!workspace || ws_bytes < need || !aligned(workspace, 256)))
    return DSA_ERR_INVALID_ARG;
  return run_topk(logits, ld, row_starts, row_ends, nullptr, 1, T, S, k, out, as_stream(stream),
                  need > 0 ? static_cast<uint32_t*>(workspace) : nullptr, false);
}

dsa_status_t dsa_indexer_topk(const void* q, const float* q_scale, const void* k,
                              const float* k_scale, dsa_dtype_t dtype, const float* weights,
                              const int32_t* row_starts, const int32_t* row_ends, int T, int S,
                              int H, int D, int topk, int32_t* out, void* workspace,
                              size_t ws_bytes, dsa_stream_t stream) {
  const CallRange range("dsa_indexer_topk");
  dsa_status_t st = check_logits_args(q, q_scale, k, k_scale, dtype, weights, row_starts,
                                      row_ends, T, S, H, D);
  if (st != DSA_OK) return st;
  if (!out || !aligned(out, 4) || topk < 1) return DSA_ERR_INVALID_ARG;
  if (!topk_supported(S)) return DSA_ERR_UNSUPPORTED;
  const size_t need = dsa_workspace_bytes(DSA_OP_INDEXER_TOPK, T, S, topk);
  if (need > 0 && (!workspace || ws_bytes < need || !aligned(workspace, 256)))
    return DSA_ERR_INVALID_ARG;
  if (T == 0) return DSA_OK;
  const int64_t ld = round_up(S > 0 ? S : 1, 4);
  float* lg = static_cast<float*>(workspace);
  uint32_t* split = split_scratch(workspace, T, S);
  st = from_cuda(clear_split(split, T, S, as_stream(stream)));
  if (st != DSA_OK) return st;
  st = run_logits(q, q_scale, k, k_scale, dtype, weights, row_starts, row_ends, T, S, H, D, lg, ld,
                  as_stream(stream));
  if (st != DSA_OK) return st;
  return run_topk(lg, ld, row_starts, row_ends, nullptr, 1, T, S, topk, out, as_stream(stream),
                  split, true);
}

dsa_status_t dsa_indexer_logits_mxfp4(const void* q, const uint8_t* q_sf, const void* k,
                                      const uint8_t* k_sf, const float* weights,
                                      const int32_t* row_starts, const int32_t* row_ends, int T,
                                      int S, int H, int D, float* logits, int64_t ld,
                                      uint32_t flags, dsa_stream_t stream) {
  const CallRange range("dsa_indexer_logits_mxfp4");
  dsa_status_t st =
      check_mx_args(q, q_sf, k, k_sf, weights, row_starts, row_ends, T, S, H, D);
  if (st != DSA_OK) return st;
  if (!logits || !aligned(logits, 4) || ld < S || ld < 1) return DSA_ERR_INVALID_ARG;
  if (flags & ~DSA_LOGITS_CLEAN) return DSA_ERR_INVALID_ARG;
  if (T == 0) return DSA_OK;
  if (flags & DSA_LOGITS_CLEAN) {
    st = from_cuda(launch_fill(logits, T, S, ld, -INFINITY, as_stream(stream)));
    if (st != DSA_OK) return st;
  }
  return run_logits_mx(q, q_sf, k, k_sf, weights, row_starts, row_ends, T, S, H, logits, ld,
                       as_stream(stream));
}

dsa_status_t dsa_indexer_topk_mxfp4(const void* q, const uint8_t* q_sf, const void* k,
                                    const uint8_t* k_sf, const float* weights,
                                    const int32_t* row_starts, const int32_t* row_ends, int T,
                                    int S, int H, int D, int topk, int32_t* out, void* workspace,
                                    size_t ws_bytes, dsa_stream_t stream) {
  const CallRange range("dsa_indexer_topk_mxfp4");
  dsa_status_t st =
      check_mx_args(q, q_sf, k, k_sf, weights, row_starts, row_ends, T, S, H, D);
  if (st != DSA_OK) return st;
  if (!out || !aligned(out, 4) || topk < 1) return DSA_ERR_INVALID_ARG;
  if (!topk_supported(S)) return DSA_ERR_UNSUPPORTED;
  const size_t need = dsa_workspace_bytes(DSA_OP_INDEXER_TOPK, T, S, topk);
  if (need > 0 && (!workspace || ws_bytes < need || !aligned(workspace, 256)))
    return DSA_ERR_INVALID_ARG;
  if (T == 0) return DSA_OK;
  const int64_t ld = round_up(S > 0 ? S : 1, 4);
  float* lg = static_cast<float*>(workspace);
  uint32_t* split = split_scratch(workspace, T, S);
  st = from_cuda(clear_split(split, T, S, as_stream(stream)));
  if (st != DSA_OK) return st;
  st = run_logits_mx(q, q_sf, k, k_sf, weights, row_starts, row_ends, T, S, H, lg, ld,
                     as_stream(stream));
  if (st != DSA_OK) return st;
  return run_topk(lg, ld, row_starts, row_ends, nullptr, 1, T, S, topk, out, as_stream(stream),
                  split, true);
}

// ---------------------------------------------------- host-buffer pipeline

namespace {

// Device-buffer layout of dsa_indexer_topk_host: the inputs, the indices, and
// one chunk's workspace, each region 256-byte aligned.
struct HostPlan {
  int64_t chunk;                // rows per full chunk
  std::vector<int64_t> bounds;  // chunk c holds rows [bounds[c], bounds[c+1])
  size_t k, ks, q, qs, w, rs, re, out, ws, total;
};

HostPlan host_plan(int T, int S, int H, int D, int topk, dsa_dtype_t dtype, bool q_scale,
                   bool k_scale) {
  HostPlan pl = {};
  const size_t esz = dtype == DSA_E4M3 ? 1 : 2;
  const int64_t nchunks = T <= 0 ? 1 : std::min<int64_t>(12, (T + 511) / 512);
  // Chunks of whole rounds of the persistent scoring kernel (its rows per
  // group times this device's SM count), so that no chunk's kernel ends on a
  // partial round of its longest groups; the remainder is the first chunk,
  // whose rows are the shortest under a causal mask.  Rows in multiples of
  // 64 where a round is larger than a chunk (or there is no device).
  const int64_t even = (static_cast<int64_t>(T) + nchunks - 1) / nchunks;
  const int64_t round_rows =
      static_cast<int64_t>(score_tokens_per_group(H)) * std::max(device_sm_count(), 0);
  const int64_t unit = round_rows > 0 && round_rows <= even ? round_rows : 64;
  pl.chunk = std::max<int64_t>(1, round_up(even, unit));
  // The remainder first, then full chunks; with three or more chunks the
  // first and the last are cut down to one unit each (the rest of each
  // becomes a chunk of its own): the pipeline waits for the first chunk's
  // upload before anything is scored and for the last chunk's download after
  // everything is, so both are kept short.
  const int64_t first = T > 0 ? T - (T - 1) / pl.chunk * pl.chunk : 1;
  pl.bounds.push_back(0);
  if (T > 0) {
    const int64_t nfull = (T - first) / pl.chunk;
    const bool cut = nfull >= 2;
    if (cut && first > unit) pl.bounds.push_back(unit);
    pl.bounds.push_back(first);
    for (int64_t c = 1; c <= nfull; ++c) {
      if (cut && c == nfull && pl.chunk > unit) pl.bounds.push_back(T - unit);
      pl.bounds.push_back(first + c * pl.chunk);
    }
  }
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += static_cast<size_t>(round_up(static_cast<int64_t>(bytes), 256));
    return at;
  };
  pl.k = take(static_cast<size_t>(S) * D * esz);
  pl.ks = take(k_scale ? static_cast<size_t>(S) * 4 : 0);
  pl.q = take(static_cast<size_t>(T) * H * D * esz);
  pl.qs = take(q_scale ? static_cast<size_t>(T) * H * 4 : 0);
  pl.w = take(static_cast<size_t>(T) * H * 4);
  pl.rs = take(static_cast<size_t>(T) * 4);
  pl.re = take(static_cast<size_t>(T) * 4);
  pl.out = take(static_cast<size_t>(T) * topk * 4);
  // The chunks share one workspace; a short last chunk may take the split
  // top-k path (more scratch per row) where a full one does not.
  size_t ws = dsa_workspace_bytes(DSA_OP_INDEXER_TOPK, 1, S, topk);
  for (size_t c = 0; c + 1 < pl.bounds.size(); ++c)
    ws = std::max(ws, dsa_workspace_bytes(DSA_OP_INDEXER_TOPK,
                                          static_cast<int>(pl.bounds[c + 1] - pl.bounds[c]), S,
                                          topk));
  pl.ws = take(ws);
  pl.total = off;
  return pl;
}

}  // namespace

size_t dsa_indexer_topk_host_bytes(int T, int S, int H, int D, int topk, dsa_dtype_t dtype) {
  if (T < 0 || S < 0 || H < 1 || D < 1 || topk < 1) return static_cast<size_t>(-1);
  if (dtype != DSA_BF16 && dtype != DSA_E4M3) return static_cast<size_t>(-1);
  return host_plan(T, S, H, D, topk, dtype, true, dtype == DSA_E4M3).total;
}

dsa_status_t dsa_indexer_topk_host(const void* q, const float* q_scale, const void* k,
                                   const float* k_scale, dsa_dtype_t dtype, const float* weights,
                                   const int32_t* row_starts, const int32_t* row_ends, int T,
                                   int S, int H, int D, int topk, int32_t* out,
                                   void* device_buffer, size_t device_bytes,
                                   dsa_stream_t stream) {
  const CallRange range("dsa_indexer_topk_host");
  // Arrays indexed by row may be null when there are no rows, k when there
  // are no keys.
  if (T < 0 || S < 0 || H < 1 || D < 1 || topk < 1) return DSA_ERR_INVALID_ARG;
  if ((T > 0 && (!q || !weights || !row_starts || !row_ends || !out)) || (S > 0 && !k))
    return DSA_ERR_INVALID_ARG;
  dsa_status_t st = check_elems(dtype, H, D, k_scale);
  if (st != DSA_OK) return st;
  if (static_cast<int64_t>(T) * H >= (int64_t(1) << 31)) return DSA_ERR_UNSUPPORTED;
  if (!topk_supported(S)) return DSA_ERR_UNSUPPORTED;
  // Sized as dsa_indexer_topk_host_bytes, which cannot know whether q_scale
  // will be given: its region is always reserved.
  const HostPlan pl = host_plan(T, S, H, D, topk, dtype, true, dtype == DSA_E4M3);
  if (!device_buffer || device_bytes < pl.total || !aligned(device_buffer, 256))
    return DSA_ERR_INVALID_ARG;
  if (T == 0) return DSA_OK;
  char* base = static_cast<char*>(device_buffer);
  const size_t esz = dtype == DSA_E4M3 ? 1 : 2;
  void* k_d = base + pl.k;
  float* ks_d = k_scale ? reinterpret_cast<float*>(base + pl.ks) : nullptr;
  char* q_d = base + pl.q;
  float* qs_d = q_scale ? reinterpret_cast<float*>(base + pl.qs) : nullptr;
  float* w_d = reinterpret_cast<float*>(base + pl.w);
  int32_t* rs_d = reinterpret_cast<int32_t*>(base + pl.rs);
  int32_t* re_d = reinterpret_cast<int32_t*>(base + pl.re);
  int32_t* out_d = reinterpret_cast<int32_t*>(base + pl.out);
  void* ws_d = base + pl.ws;
  const int64_t ld = round_up(S > 0 ? S : 1, 4);
  const int64_t nch = static_cast<int64_t>(pl.bounds.size()) - 1;

  // Three streams: uploads, compute (the caller's), downloads.  Chunk c's
  // upload overlaps chunk c-1's compute and chunk c-2's download.
  cudaStream_t comp = as_stream(stream), up = nullptr, down = nullptr;
  std::vector<cudaEvent_t> ev;
  auto event = [&]() {
    cudaEvent_t e = nullptr;
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return e;
    ev.push_back(e);
    return e;
  };
  cudaError_t e = cudaStreamCreateWithFlags(&up, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&down, cudaStreamNonBlocking);
  cudaEvent_t start = event(), k_in = event(), done = event(), up_done = event();
  if (e == cudaSuccess && (!start || !k_in || !done || !up_done)) e = cudaErrorMemoryAllocation;
  if (e == cudaSuccess) e = cudaEventRecord(start, comp);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(up, start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(down, start, 0);
  // K and the row ranges first, then each chunk's queries; the weights (and
  // query scales) go with their chunk when a chunk's share is large enough
  // to be worth a copy of its own (every copy costs the copy engine a few
  // microseconds however small it is), else all at once up front.
  const size_t t4 = static_cast<size_t>(T) * 4, th = static_cast<size_t>(T) * H * 4;
  const bool w_by_chunk = static_cast<size_t>(pl.chunk) * H * 4 >= (512u << 10);
  if (e == cudaSuccess && !w_by_chunk)
    e = cudaMemcpyAsync(w_d, weights, th, cudaMemcpyHostToDevice, up);
  if (e == cudaSuccess && !w_by_chunk && q_scale)
    e = cudaMemcpyAsync(qs_d, q_scale, th, cudaMemcpyHostToDevice, up);
  if (e == cudaSuccess && S > 0)
    e = cudaMemcpyAsync(k_d, k, static_cast<size_t>(S) * D * esz, cudaMemcpyHostToDevice, up);
  if (e == cudaSuccess && S > 0 && k_scale)
    e = cudaMemcpyAsync(ks_d, k_scale, static_cast<size_t>(S) * 4, cudaMemcpyHostToDevice, up);
  if (e == cudaSuccess) e = cudaMemcpyAsync(rs_d, row_starts, t4, cudaMemcpyHostToDevice, up);
  if (e == cudaSuccess) e = cudaMemcpyAsync(re_d, row_ends, t4, cudaMemcpyHostToDevice, up);
  if (e == cudaSuccess) e = cudaEventRecord(k_in, up);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(comp, k_in, 0);
  for (int64_t c = 0; c < nch && e == cudaSuccess && st == DSA_OK; ++c) {
    const int64_t r0 = pl.bounds[c];
    const int64_t rows = pl.bounds[c + 1] - r0;
    const int64_t qe = static_cast<int64_t>(H) * D;
    cudaEvent_t in = event(), computed = event();
    if (!in || !computed) {
      e = cudaErrorMemoryAllocation;
      break;
    }
    // upload chunk c's queries and weights
    e = cudaMemcpyAsync(q_d + r0 * qe * esz, static_cast<const char*>(q) + r0 * qe * esz,
                        rows * qe * esz, cudaMemcpyHostToDevice, up);
    if (e == cudaSuccess && w_by_chunk)
      e = cudaMemcpyAsync(w_d + r0 * H, weights + r0 * H, static_cast<size_t>(rows) * H * 4,
                          cudaMemcpyHostToDevice, up);
    if (e == cudaSuccess && w_by_chunk && q_scale)
      e = cudaMemcpyAsync(qs_d + r0 * H, q_scale + r0 * H, static_cast<size_t>(rows) * H * 4,
                          cudaMemcpyHostToDevice, up);
    if (e == cudaSuccess) e = cudaEventRecord(in, up);
    // compute chunk c on the caller's stream
    if (e == cudaSuccess) e = cudaStreamWaitEvent(comp, in, 0);
    if (e != cudaSuccess) break;
    float* lg = static_cast<float*>(ws_d);
    uint32_t* split = split_scratch(ws_d, rows, S);
    st = from_cuda(clear_split(split, rows, S, comp));
    if (st == DSA_OK)
      st = run_logits(q_d + r0 * qe * esz, qs_d ? qs_d + r0 * H : nullptr, k_d, ks_d, dtype,
                      w_d + r0 * H, rs_d + r0, re_d + r0, static_cast<int>(rows), S, H, D, lg,
                      ld, comp);
    if (st == DSA_OK)
      st = run_topk(lg, ld, rs_d + r0, re_d + r0, nullptr, 1, static_cast<int>(rows), S, topk,
                    out_d + r0 * topk, comp, split, true);
    if (st != DSA_OK) break;
    e = cudaEventRecord(computed, comp);
    // download chunk c
    if (e == cudaSuccess) e = cudaStreamWaitEvent(down, computed, 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(out + r0 * topk, out_d + r0 * topk, rows * topk * 4,
                          cudaMemcpyDeviceToHost, down);
  }
  // Join both streams, also after an error part-way: later work on the
  // caller's stream sees every copy this call queued.
  cudaError_t j = cudaSuccess;
  if (done && down) j = cudaEventRecord(done, down);
  if (j == cudaSuccess && done) j = cudaStreamWaitEvent(comp, done, 0);
  if (j == cudaSuccess && up_done && up) j = cudaEventRecord(up_done, up);
  if (j == cudaSuccess && up_done) j = cudaStreamWaitEvent(comp, up_done, 0);
  if (up) cudaStreamDestroy(up);      // released once their work is done
  if (down) cudaStreamDestroy(down);
  for (cudaEvent_t x : ev) cudaEventDestroy(x);
  if (st != DSA_OK) return st;
  return from_cuda(e != cudaSuccess ? e : j);
}

dsa_status_t dsa_indexer_logits_paged(const void* q, const float* q_scale, const float* weights,
                                      const void* k_cache, const float* k_scale, int num_blocks,
                                      dsa_dtype_t dtype, const int32_t* block_table,
                                      int max_blocks, const int32_t* context_lens, int B,
                                      int next_n, int block_size, int H, int D, float* logits,
                                      int64_t ld, dsa_stream_t stream) {
  const CallRange range("dsa_indexer_logits_paged");
  const PagedShape s = {B, next_n, block_size, max_blocks, num_blocks, H, D};
  dsa_status_t st = check_paged_args(q, q_scale, weights, k_cache, k_scale, dtype, block_table,
                                     context_lens, s);
  if (st != DSA_OK) return st;
  if (!logits || !aligned(logits, 4) || ld < static_cast<int64_t>(max_blocks) * block_size)
    return DSA_ERR_INVALID_ARG;
  return run_logits_paged(q, q_scale, weights, k_cache, k_scale, dtype, block_table, context_lens,
                          s, logits, ld, as_stream(stream));
}

dsa_status_t dsa_indexer_topk_paged(const void* q, const float* q_scale, const float* weights,
                                    const void* k_cache, const float* k_scale, int num_blocks,
                                    dsa_dtype_t dtype, const int32_t* block_table, int max_blocks,
                                    const int32_t* context_lens, int B, int next_n,
                                    int block_size, int H, int D, int topk, int32_t* out,
                                    void* workspace, size_t ws_bytes, dsa_stream_t stream) {
  const CallRange range("dsa_indexer_topk_paged");
  const PagedShape s = {B, next_n, block_size, max_blocks, num_blocks, H, D};
  dsa_status_t st = check_paged_args(q, q_scale, weights, k_cache, k_scale, dtype, block_table,
                                     context_lens, s);
  if (st != DSA_OK) return st;
  if (!out || !aligned(out, 4) || topk < 1) return DSA_ERR_INVALID_ARG;
  const int64_t R = static_cast<int64_t>(B) * next_n;
  const int64_t max_ctx = static_cast<int64_t>(max_blocks) * block_size;
  if (!topk_supported(static_cast<int>(max_ctx))) return DSA_ERR_UNSUPPORTED;
  const size_t need = dsa_workspace_bytes(DSA_OP_INDEXER_TOPK_PAGED, R, max_ctx, topk);
  if (need > 0 && (!workspace || ws_bytes < need || !aligned(workspace, 256)))
    return DSA_ERR_INVALID_ARG;
  if (B == 0) return DSA_OK;
  const int64_t ld = round_up(max_ctx, 4);
  float* lg = static_cast<float*>(workspace);
  uint32_t* split = split_scratch(workspace, R, max_ctx);
  st = from_cuda(clear_split(split, R, max_ctx, as_stream(stream)));
  if (st != DSA_OK) return st;
  st = run_logits_paged(q, q_scale, weights, k_cache, k_scale, dtype, block_table, context_lens, s,
                        lg, ld, as_stream(stream));
  if (st != DSA_OK) return st;
  return run_topk(lg, ld, nullptr, nullptr, context_lens, next_n, static_cast<int>(R),
                  static_cast<int>(max_ctx), topk, out, as_stream(stream), split, true);
}

dsa_status_t dsa_topk_sort_by_score(const float* logits, int64_t ld, int32_t* topk, int T, int k,
                                    dsa_stream_t stream) {
  const CallRange range("dsa_topk_sort_by_score");
  if (!logits || !topk || T < 0 || k < 1 || ld < 1) return DSA_ERR_INVALID_ARG;
  if (!aligned(logits, 4) || !aligned(topk, 4)) return DSA_ERR_INVALID_ARG;
  if (k > kTopkSortMax) return DSA_ERR_UNSUPPORTED;
  if (T == 0) return DSA_OK;
  return from_cuda(launch_topk_sort(logits, ld, topk, T, k, error_word(), as_stream(stream)));
}

dsa_status_t dsa_topk_merge(const float* cand_scores, const int32_t* cand_cols, int T, int C,
                            int k, int32_t* out, dsa_stream_t stream) {
  const CallRange range("dsa_topk_merge");
  if (!cand_scores || !cand_cols || !out || T < 0 || C < 1 || k < 1) return DSA_ERR_INVALID_ARG;
  if (!aligned(cand_scores, 4) || !aligned(cand_cols, 4) || !aligned(out, 4))
    return DSA_ERR_INVALID_ARG;
  if (C > kTopkMergeMax || k > kTopkMergeMax) return DSA_ERR_UNSUPPORTED;
  return from_cuda(launch_topk_merge(cand_scores, cand_cols, T, 1, C, k, out, as_stream(stream)));
}

dsa_status_t dsa_topk_merge_ranks(const float* cand_scores, const int32_t* cand_cols, int W,
                                  int T, int kr, int k, int32_t* out, dsa_stream_t stream) {
  const CallRange range("dsa_topk_merge_ranks");
  if (!cand_scores || !cand_cols || !out || W < 1 || T < 0 || kr < 1 || k < 1)
    return DSA_ERR_INVALID_ARG;
  if (!aligned(cand_scores, 4) || !aligned(cand_cols, 4) || !aligned(out, 4))
    return DSA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(W) * kr > kTopkMergeMax || k > kTopkMergeMax)
    return DSA_ERR_UNSUPPORTED;
  return from_cuda(launch_topk_merge(cand_scores, cand_cols, T, W, kr, k, out, as_stream(stream)));
}

dsa_status_t dsa_topk_dcp_candidates(const float* logits, int64_t ld, const int32_t* row_starts,
                                     const int32_t* row_ends, int T, int S, int k, int rank,
                                     int world, int interleave, float* cand_scores,
                                     int32_t* cand_cols, void* workspace, size_t ws_bytes,
                                     dsa_stream_t stream) {
  const CallRange range("dsa_topk_dcp_candidates");
  if (!logits || !row_starts || !row_ends || !cand_scores || !cand_cols) return DSA_ERR_INVALID_ARG;
  if (T < 0 || S < 0 || k < 1 || ld < S || ld < 1 || world < 1 || rank < 0 || rank >= world ||
      interleave < 1)
    return DSA_ERR_INVALID_ARG;
  if (!aligned(logits, 4) || !aligned(cand_scores, 4) || !aligned(cand_cols, 4) ||
      !aligned(row_starts, 4) || !aligned(row_ends, 4))
    return DSA_ERR_INVALID_ARG;
  if (!topk_supported(S)) return DSA_ERR_UNSUPPORTED;
  // The largest global position a local column can map to must fit int32.
  if (S > 0) {
    const int64_t runs = (static_cast<int64_t>(S) - 1) / interleave;
    const int64_t gmax = (runs * world + (world - 1)) * interleave + (interleave - 1);
    if (gmax > INT32_MAX) return DSA_ERR_UNSUPPORTED;
  }
  const size_t need = dsa_workspace_bytes(DSA_OP_TOPK, T, S, k);
  if (need > 0 && (!workspace || ws_bytes < need || !aligned(workspace, 256)))
    return DSA_ERR_INVALID_ARG;
  dsa_status_t st = run_topk(logits, ld, row_starts, row_ends, nullptr, 1, T, S, k, cand_cols,
                             as_stream(stream),
                             need > 0 ? static_cast<uint32_t*>(workspace) : nullptr, false);
  if (st != DSA_OK) return st;
  return from_cuda(launch_dcp_pairs(logits, ld, T, k, rank, world, interleave, cand_scores,
                                    cand_cols, as_stream(stream)));
}

dsa_status_t dsa_q_quant_fold_weights(const void* q, const float* weights, float weight_scale,
                                      int T, int H, int D, int padded_heads, void* q_fp8,
                                      float* weights_out, dsa_stream_t stream) {
  const CallRange range("dsa_q_quant_fold_weights");
  if (!q || !weights || !q_fp8 || !weights_out || T < 0 || H < 1 || padded_heads < H)
    return DSA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(q_fp8, 8) || !aligned(weights, 4) || !aligned(weights_out, 4))
    return DSA_ERR_INVALID_ARG;
  if (D != 128 || padded_heads > 64) return DSA_ERR_UNSUPPORTED;
  return from_cuda(launch_q_quant_fold(q, weights, weight_scale, T, H, padded_heads, q_fp8,
                                       weights_out, as_stream(stream)));
}

dsa_status_t dsa_k_norm_quant_insert(const void* k, const float* ln_weight, const float* ln_bias,
                                     float eps, const int64_t* slot_mapping, int T, int D,
                                     dsa_dtype_t cache_dtype, void* k_cache, float* k_scale,
                                     int num_blocks, int block_size, dsa_stream_t stream) {
  const CallRange range("dsa_k_norm_quant_insert");
  if (!k || !ln_weight || !ln_bias || !slot_mapping || !k_cache || T < 0 || num_blocks < 1 ||
      block_size < 1 || !(eps >= 0.f))
    return DSA_ERR_INVALID_ARG;
  if (cache_dtype != DSA_BF16 && cache_dtype != DSA_E4M3) return DSA_ERR_INVALID_ARG;
  const bool fp8 = cache_dtype == DSA_E4M3;
  if (fp8 != (k_scale != nullptr)) return DSA_ERR_INVALID_ARG;  // scales exactly for e4m3
  if (!aligned(k, 16) || !aligned(k_cache, 16) || !aligned(ln_weight, 16) || !aligned(ln_bias, 16) ||
      !aligned(slot_mapping, 8) || (k_scale && !aligned(k_scale, 4)))
    return DSA_ERR_INVALID_ARG;
  if (D != 128) return DSA_ERR_UNSUPPORTED;
  const int64_t capacity = static_cast<int64_t>(num_blocks) * block_size;
  return from_cuda(launch_k_norm_insert(k, ln_weight, ln_bias, eps, slot_mapping, T, fp8, capacity,
                                        k_cache, k_scale, error_word(), as_stream(stream)));
}

size_t dsa_workspace_bytes(dsa_op_t op, int64_t rows, int64_t cols, int k) {
  if (rows < 0 || cols < 0 || k < 0) return static_cast<size_t>(-1);
  switch (op) {
    case DSA_OP_INDEXER_LOGITS:
    case DSA_OP_INDEXER_LOGITS_PAGED:
      return 0;
    case DSA_OP_TOPK:
      return topk_split_rows(rows, cols) ? split_scratch_bytes(rows, cols) : 0;
    case DSA_OP_INDEXER_TOPK:
    case DSA_OP_INDEXER_TOPK_PAGED:
      if (rows == 0) return 0;
      return logits_scratch_bytes(rows, cols) +
             (topk_split_rows(rows, cols) ? split_scratch_bytes(rows, cols) : 0);
    default:
      return static_cast<size_t>(-1);
  }
}

const char* dsa_status_string(dsa_status_t status) {
  switch (status) {
    case DSA_OK:
      return "ok";
    case DSA_ERR_INVALID_ARG:
      return "invalid argument";
    case DSA_ERR_UNSUPPORTED:
      return "unsupported shape or dtype";
    case DSA_ERR_CUDA:
      return "CUDA error";
    case DSA_ERR_TIMEOUT:
      return "device-side wait timed out";
    default:
      return "unknown status";
  }
}

dsa_status_t dsa_get_last_device_error(void) {
  if (cudaDeviceSynchronize() != cudaSuccess) return DSA_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpyFromSymbol(&word, g_error_word, sizeof(word)) != cudaSuccess) return DSA_ERR_CUDA;
  const uint32_t zero = 0;
  if (word && cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero)) != cudaSuccess)
    return DSA_ERR_CUDA;
  if (word & kErrTimeout) return DSA_ERR_TIMEOUT;
  if (word & kErrBadIndex) return DSA_ERR_INVALID_ARG;
  return DSA_OK;
}

dsa_status_t dsa_selftest_wait_timeout(uint64_t timeout_ns, dsa_stream_t stream) {
  if (timeout_ns < 1000) timeout_ns = 1000;
  if (timeout_ns > 1000000000ull) timeout_ns = 1000000000ull;
  uint32_t* err = error_word();
  if (!err) return DSA_ERR_CUDA;
  return from_cuda(launch_wait_timeout_selftest(err, timeout_ns, as_stream(stream)));
}

}  // extern "C"

// ------------------------------------------------------------------------
// dsa_indexer_topk_noalloc: the logits scratch is a fixed device array of the
// library, for callers that cannot allocate device memory at call time.

namespace dsa {
namespace {

constexpr size_t kNoallocScratchFloats = DSA_NOALLOC_SCRATCH_BYTES / sizeof(float);

// Shared by every call on a device; held for the life of the process.
static __device__ __align__(256) float g_noalloc_scratch[kNoallocScratchFloats];

// Device address of g_noalloc_scratch on the current device.  In host code the
// array's name only stands in for the symbol; the address is looked up once
// per device, with that device current, and cached.
float* noalloc_scratch() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  static std::mutex mu;
  static float* addr[kMaxDevices] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, g_noalloc_scratch) != cudaSuccess || !a) return nullptr;
    addr[dev] = static_cast<float*>(a);
  }
  return addr[dev];
}

}  // namespace
}  // namespace dsa

extern "C" dsa_status_t dsa_indexer_topk_noalloc(const void* q, const float* q_scale,
                                                 const void* k, const float* k_scale,
                                                 dsa_dtype_t dtype, const float* weights,
                                                 const int32_t* row_starts,
                                                 const int32_t* row_ends, int T, int S, int H,
                                                 int D, int topk, int32_t* out,
                                                 dsa_stream_t stream) {
  const CallRange range("dsa_indexer_topk_noalloc");
  dsa_status_t st = check_logits_args(q, q_scale, k, k_scale, dtype, weights, row_starts,
                                      row_ends, T, S, H, D);
  if (st != DSA_OK) return st;
  if (!out || !aligned(out, 4) || topk < 1) return DSA_ERR_INVALID_ARG;
  if (!topk_supported(S)) return DSA_ERR_UNSUPPORTED;
  if (T == 0) return DSA_OK;
  const int64_t ld = round_up(S > 0 ? S : 1, 4);
  if (static_cast<uint64_t>(T) * static_cast<uint64_t>(ld) > kNoallocScratchFloats)
    return DSA_ERR_UNSUPPORTED;
  float* lg = noalloc_scratch();
  if (!lg) return DSA_ERR_CUDA;
  st = run_logits(q, q_scale, k, k_scale, dtype, weights, row_starts, row_ends, T, S, H, D, lg, ld,
                  as_stream(stream));
  if (st != DSA_OK) return st;
  return run_topk(lg, ld, row_starts, row_ends, nullptr, 1, T, S, topk, out, as_stream(stream),
                  nullptr, true);
}
