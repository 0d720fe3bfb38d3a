// dsa_internal.h -- parameter blocks and launchers shared between the kernel
// translation units and the C-ABI unit (dsa_api.cu).  Not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dsa {

// Scoring kernel parameters.  Passed by value as a __grid_constant__ kernel
// argument, so the two TMA descriptors live in parameter space.
struct ScoreParams {
  CUtensorMap tmap_q;  // q viewed as [R*H, D] elements, 128-byte swizzled boxes
  CUtensorMap tmap_k;  // prefill: k [S, D]; paged: k_cache [num_blocks, block_size, D]
  const float* weights;       // [R, H]
  const float* q_scale;       // [R, H] or null
  const float* k_scale;       // prefill [S]; paged [num_blocks*block_size]; or null
  const int32_t* row_starts;  // prefill [R]
  const int32_t* row_ends;    // prefill [R]
  const int32_t* block_table;   // paged [B, max_blocks]
  const int32_t* context_lens;  // paged [B]
  float* logits;              // [R, ld]
  int64_t ld;
  int R;            // query rows (prefill T, paged B*next_n)
  int S;            // prefill: number of keys; paged: ld bound on columns written
  int max_blocks;   // paged
  int next_n;       // paged
  int block_size;   // paged
  int num_blocks;   // paged
  int chunk_keys;   // paged: keys per CTA (multiple of 128)
  int chunks_per_req;  // paged
  uint32_t* err;    // device error word
};

// Largest batch of paged-decode requests one call takes (the scoring kernel
// keeps a per-request prefix sum of its work list in shared memory).
constexpr int kMaxPagedRequests = 2048;

struct TopkParams {
  const float* logits;  // [R, ld]
  int64_t ld;
  const int32_t* row_starts;    // [R] (prefill) or null
  const int32_t* row_ends;      // [R] (prefill) or null
  const int32_t* context_lens;  // [B] (paged) or null
  int next_n;                   // paged
  int R;
  int S;          // column bound: prefill S, paged max context
  int k;
  int bitmap_words;  // ceil(S / 32): shared-memory selection bitmaps per row
  int32_t* out;      // [R, k]
  uint32_t* split;   // null, or [R, split_words] scratch of the split path (topk_split_rows)
  int split_words;   // words of split scratch per row (topk_split_words(S))
  // 1 when the kernel queued just before on the stream is this library's own
  // scoring kernel (the composed calls): the first top-k kernel may then be
  // its programmatic dependent, since the row ranges it reads before waiting
  // were written before that scoring kernel started; the split path's
  // scratch was then cleared before the scoring kernel (topk_split_clear).
  // 0 for the standalone dsa_topk, whose predecessor may be the caller's
  // kernel writing the ranges.
  int after_score;
};

// Launchers (return the launch error, if any).  Shapes were validated by the
// caller; `supported` variants report whether a template instance exists.
bool score_prefill_bf16_supported(int H, int D);
cudaError_t launch_score_prefill_bf16(const ScoreParams& p, int H, int D, cudaStream_t s);
bool score_prefill_fp8_supported(int H, int D);
cudaError_t launch_score_prefill_fp8(const ScoreParams& p, int H, int D, cudaStream_t s);
bool score_paged_supported(bool fp8, int H, int D, int next_n);
// MMA columns (and q-tile rows) of the paged kernel: next_n*H rounded up to 64/128/256.
int score_paged_cols(int H, int next_n);
cudaError_t launch_score_paged(const ScoreParams& p, bool fp8, int H, int D, cudaStream_t s);
// MXFP4 prefill (packed E2M1 q [R*H, D/2], k [S, D/2]; E8M0 scales q_sf
// [R*H, D/32], k_sf [S, D/32]); H = 64, D = 128 only.
bool score_mx_supported(int H, int D);
// Rows of q ([R*H, D/2] packed) the MXFP4 kernel loads per group: the TMA box
// height of its q map.
int score_mx_q_rows();
cudaError_t launch_score_mx(const ScoreParams& p, const uint8_t* q_sf, const uint8_t* k_sf,
                            cudaStream_t s);
// Tokens (query rows) per prefill tile group for a head count.
int score_tokens_per_group(int H);

cudaError_t launch_topk(const TopkParams& p, cudaStream_t s);
int topk_bitmap_words(int max_row);
// Whether rows of up to max_row columns fit the top-k kernels.
bool topk_supported(int max_row);
// Few long rows take the split path: every phase runs on many CTAs per row
// (one per 4096-key unit), exchanging per-row histograms, candidate keys,
// the threshold and per-unit offsets through global scratch of
// topk_split_words(max_row) words per row.  Depends on the shape only, so the
// workspace size is known on the host.
bool topk_split_rows(int64_t rows, int64_t max_row);
int topk_split_words(int64_t max_row);
// Zeroes each split-path row's histogram and state words (before its first phase).
cudaError_t topk_split_clear(uint32_t* split, int split_words, int rows, cudaStream_t s);
cudaError_t launch_fill(float* dst, int64_t rows, int64_t cols, int64_t ld, float value,
                        cudaStream_t s);
// Rows of k top-k indices reordered by descending score in place (k <=
// kTopkSortMax); indices outside [0, ld) are treated as padding and recorded.
constexpr int kTopkSortMax = 8192;
// Merge of C (score, global column) candidates per row into the k best,
// ascending columns, -1 padding (C, k <= kTopkMergeMax).
constexpr int kTopkMergeMax = 16384;
cudaError_t launch_topk_merge(const float* scores, const int32_t* cols, int T, int W, int kr,
                              int k, int32_t* out, cudaStream_t s);
cudaError_t launch_dcp_pairs(const float* logits, int64_t ld, int T, int k, int rank, int W,
                             int inter, float* scores, int32_t* cols, cudaStream_t s);
cudaError_t launch_topk_sort(const float* logits, int64_t ld, int32_t* topk, int T, int k,
                             uint32_t* err, cudaStream_t s);
cudaError_t launch_wait_timeout_selftest(uint32_t* err, uint64_t timeout_ns, cudaStream_t s);
// SM count of the current device (queried once per device).
int device_sm_count();
// The steps before the indexer (dsa_prologue.cu); D = 128.
cudaError_t launch_q_quant_fold(const void* q, const float* w, float weight_scale, int T, int H,
                                int Hp, void* q8, float* w_out, cudaStream_t s);
cudaError_t launch_k_norm_insert(const void* k, const float* gamma, const float* beta, float eps,
                                 const int64_t* slots, int T, bool fp8, int64_t capacity,
                                 void* cache, float* cache_scale, uint32_t* err, cudaStream_t s);

}  // namespace dsa
