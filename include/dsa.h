/*
 * dsa.h -- C ABI of the GB300 (sm_103a) DSA lightning-indexer library.
 *
 * The library computes the two stages of the DeepSeek sparse-attention
 * lightning indexer on one GPU:
 *
 *   1. index logits   logit[t,s] = sum_h w[t,h] * max(0, q[t,h,:] . k[s,:])
 *      for the key columns s of query row t's range, -inf elsewhere.  This is
 *      the quantity KimiK3DSAIndexer.score hands to
 *      torch.ops.vllm.sparse_attn_indexer (vLLM API docs,
 *      "vllm.models.kimi_k3.nvidia.dsa"): index_q [T,H,D], one index_k row
 *      [D] shared by all heads, per-head weights [T,H] into which the query
 *      scale and the softmax/head scales have already been folded.
 *   2. masked top-k   for every row, the index_topk best columns inside
 *      [row_start, row_end), written as int32 and padded with -1 wherever
 *      fewer valid keys exist -- the semantics of torch_dsa_topk as corrected
 *      in GitHub "vllm-project/vime" pull request #502 (third review comment),
 *      written into a caller-owned buffer like the model-level
 *      topk_indices_buffer of KimiK3DSAAttention.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor pointers are DEVICE memory owned by the caller, dense and
 *    row-major.  The library keeps no pointer after the call returns, frees
 *    nothing and allocates no device memory; scratch space is the caller's
 *    `workspace` (size from dsa_workspace_bytes).
 *  - Every call is asynchronous on `stream` (NULL = legacy default stream).
 *  - Element types (dsa_dtype_t): DSA_BF16 -> q and k are bf16 (2 bytes);
 *    DSA_E4M3 -> q and k are OCP fp8 e4m3 codes (1 byte) with fp32
 *    power-of-two block scales, one per D-element row (UE8M0 scales,
 *    quant_block_size = index_head_dim, KimiK3DSAIndexer.__init__).
 *  - Shapes: H (index heads) is a power of two in [1, 64] (the page's
 *    DeepGEMM limit of 64 heads); D is 64 or 128 for bf16 and 128 for e4m3.
 *  - Row ranges are half-open [row_start, row_end) and are clamped to [0, S);
 *    an empty or inverted range gives an all -1 top-k row.
 *  - Top-k output rows hold the selected column indices in ascending order,
 *    then -1 up to k.  Ties go to the lower column; -0.0 equals +0.0; -inf
 *    and NaN scores are never selected.
 *  - Errors that can be detected on the host are returned before anything is
 *    launched and leave every output untouched.  Asynchronous failures (a
 *    CUDA error, or a device-side wait that gave up) surface as DSA_ERR_CUDA
 *    from a later call, or from dsa_get_last_device_error().
 *  - No C++ exception crosses this boundary.  All entry points are safe to
 *    call from several host threads at once.
 *  - Each call that queues GPU work is wrapped in an NVTX range named after
 *    its entry point (visible in Nsight timelines; free without a tool).
 *  - CUDA graphs: once one of dsa_indexer_logits, dsa_topk,
 *    dsa_indexer_topk, the paged and MXFP4 calls, dsa_topk_sort_by_score or
 *    dsa_topk_merge has run on a device (its first call looks up per-device
 *    state), its calls can be captured into a CUDA graph.
 *    A capture fixes the shapes (rows, key capacity, k) and the pointers;
 *    row ranges, context lengths, block tables and the inputs themselves are
 *    read when the graph runs, so one graph serves every step of a decode
 *    loop.  dsa_get_last_device_error synchronises and is not capturable.
 */
#ifndef DSA_H_
#define DSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* == cudaStream_t / CUstream */
typedef struct CUstream_st* dsa_stream_t;

typedef enum {
    DSA_OK = 0,
    DSA_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned pointer, small workspace */
    DSA_ERR_UNSUPPORTED = 2, /* valid request this build does not handle (H, D, dtype) */
    DSA_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed */
    DSA_ERR_TIMEOUT = 4      /* a device-side wait gave up (see dsa_get_last_device_error) */
} dsa_status_t;

typedef enum { DSA_BF16 = 0, DSA_E4M3 = 1 } dsa_dtype_t;

typedef enum {
    DSA_OP_INDEXER_LOGITS = 0,
    DSA_OP_TOPK = 1,
    DSA_OP_INDEXER_TOPK = 2,
    DSA_OP_INDEXER_LOGITS_PAGED = 3,
    DSA_OP_INDEXER_TOPK_PAGED = 4
} dsa_op_t;

/* dsa_indexer_logits flag: also write -inf into every column of [0, S)
 * outside the row's range (by default only the key tiles the row touches are
 * written, and columns of skipped tiles keep whatever the buffer held). */
#define DSA_LOGITS_CLEAN 1u

/*
 * Index logits, contiguous keys (prefill; packed THD sequences use per-row
 * ranges in packed coordinates, as the THD packing of the vime "Day-0 Model
 * Plugins" page and the offset rebase of PR #502's first review comment do).
 *
 *   q          [T, H, D] bf16 or e4m3, 16-byte aligned
 *   q_scale    NULL (scale folded into weights, as KimiK3DSAIndexer.score
 *              does for fp8 queries) or [T, H] fp32 block scales
 *   k          [S, D] same element type as q, 16-byte aligned
 *   k_scale    [S] fp32 power-of-two scales for DSA_E4M3; must be NULL for bf16
 *   weights    [T, H] fp32
 *   row_starts, row_ends  [T] int32
 *   logits     [T, ld] fp32 output, ld >= S.  For every row, the columns of
 *              every 128-key tile that overlaps the union of the ranges of
 *              the row's tile group are written (-inf outside the row's own
 *              range); with DSA_LOGITS_CLEAN every column in [0, S) is.
 *   flags      0 or DSA_LOGITS_CLEAN
 * Accumulation is fp32 on tensor cores; the head sum runs in one fixed order
 * (eight interleaved fp32 partial sums, combined pairwise), so every entry
 * point produces the same logits bit for bit and dsa_indexer_topk's
 * selection equals dsa_topk applied to these logits.
 */
dsa_status_t dsa_indexer_logits(const void* q, const float* q_scale, const void* k,
                                const float* k_scale, dsa_dtype_t dtype,
                                const float* weights, const int32_t* row_starts,
                                const int32_t* row_ends, int T, int S, int H, int D,
                                float* logits, int64_t ld, uint32_t flags,
                                dsa_stream_t stream);

/*
 * Masked per-row top-k of given fp32 logits (torch_dsa_topk, vime PR #502).
 *
 *   logits     [T, ld] fp32, ld >= S; only columns in the clamped row range
 *              are read, so the rest may hold anything
 *   row_starts, row_ends  [T] int32
 *   k          index_topk >= 1
 *   out        [T, k] int32 output
 *   workspace  dsa_workspace_bytes(DSA_OP_TOPK, T, S, k) bytes, 256-byte aligned.
 *              That is 0 (workspace may be NULL) except for few long rows
 *              (S > 16384 and T < 32, or S > 262144 and T <= 512), where
 *              many CTAs per row share per-row scratch there (about 75 KiB
 *              per row).
 */
dsa_status_t dsa_topk(const float* logits, int64_t ld, const int32_t* row_starts,
                      const int32_t* row_ends, int T, int S, int k, int32_t* out,
                      void* workspace, size_t ws_bytes, dsa_stream_t stream);

/*
 * Index logits + masked top-k in one call (the sparse_attn_indexer op of
 * KimiK3DSAIndexer.score, minus the cache insert).  Arguments as
 * dsa_indexer_logits plus k/out of dsa_topk.  `workspace` must hold
 * dsa_workspace_bytes(DSA_OP_INDEXER_TOPK, T, S, k) bytes, 256-byte aligned.
 * The result equals dsa_topk(dsa_indexer_logits(...)) bit for bit.
 */
dsa_status_t dsa_indexer_topk(const void* q, const float* q_scale, const void* k,
                              const float* k_scale, dsa_dtype_t dtype,
                              const float* weights, const int32_t* row_starts,
                              const int32_t* row_ends, int T, int S, int H, int D,
                              int topk, int32_t* out, void* workspace, size_t ws_bytes,
                              dsa_stream_t stream);

/*
 * Index logits with MXFP4 queries and keys (KimiK3DSAIndexer on the vLLM page
 * "vllm.models.kimi_k3.nvidia.dsa": MXFP4 keys with MXFP4 queries on an
 * explicit indexer_kv_dtype='mxfp4', where mxfp4_q_quant returns the query,
 * its block scales and the weights).  Element format (OCP Microscaling):
 * E2M1 codes (bias 1, magnitudes 0 .. 6) packed two per byte, the even
 * element in the low nibble; every 32 consecutive elements of a row share one
 * E8M0 scale byte, value 2^(code - 127).  The scales enter the tensor-core
 * contraction (tcgen05 kind::mxf4 with block scales), so
 *   logit[t,s] = sum_h w[t,h] * max(0, sum_d q[t,h,d] * k[s,d])
 * with q and k their decoded values.
 *
 *   q         [T, H, D/2] packed E2M1, 16-byte aligned
 *   q_sf      [T, H, D/32] E8M0 scale bytes, 4-byte aligned
 *   k         [S, D/2] packed E2M1, 16-byte aligned
 *   k_sf      [S, D/32] E8M0 scale bytes, 4-byte aligned
 *   weights   [T, H] fp32 (the query scales are in q_sf, not folded in)
 *   row_starts, row_ends, logits, ld, flags: as dsa_indexer_logits
 *   H = 64 and D = 128 only (else DSA_ERR_UNSUPPORTED).
 * Errors as dsa_indexer_logits.  The head sum runs in one fixed order, so
 * dsa_indexer_topk_mxfp4's selection equals dsa_topk on these logits.
 */
dsa_status_t dsa_indexer_logits_mxfp4(const void* q, const uint8_t* q_sf, const void* k,
                                      const uint8_t* k_sf, const float* weights,
                                      const int32_t* row_starts, const int32_t* row_ends, int T,
                                      int S, int H, int D, float* logits, int64_t ld,
                                      uint32_t flags, dsa_stream_t stream);

/*
 * MXFP4 index logits + masked top-k in one call: arguments as
 * dsa_indexer_logits_mxfp4 plus k/out of dsa_topk; `workspace` must hold
 * dsa_workspace_bytes(DSA_OP_INDEXER_TOPK, T, S, k) bytes, 256-byte aligned.
 * The result equals dsa_topk(dsa_indexer_logits_mxfp4(...)) bit for bit.
 */
dsa_status_t dsa_indexer_topk_mxfp4(const void* q, const uint8_t* q_sf, const void* k,
                                    const uint8_t* k_sf, const float* weights,
                                    const int32_t* row_starts, const int32_t* row_ends, int T,
                                    int S, int H, int D, int topk, int32_t* out, void* workspace,
                                    size_t ws_bytes, dsa_stream_t stream);

/*
 * Index logits of paged decode (the paged indexer K cache of
 * KimiK3DSAIndexer: KimiK3IndexerCache / DeepseekV32IndexerCache).
 *
 *   B            requests, 0 <= B <= 2048 (DSA_ERR_UNSUPPORTED above)
 *   q            [B*next_n, H, D]; query row r = b*next_n + j is token j of request b
 *   q_scale      NULL or [B*next_n, H] fp32
 *   weights      [B*next_n, H] fp32
 *   k_cache      [num_blocks, block_size, D], 16-byte aligned
 *   k_scale      NULL (bf16) or [num_blocks, block_size] fp32 (e4m3)
 *   num_blocks   number of physical blocks in k_cache (>= 1)
 *   block_table  [B, max_blocks] int32: physical block of each logical block;
 *                an entry outside [0, num_blocks) is never dereferenced: block
 *                0 is read in its place and the device error word records it
 *                (dsa_get_last_device_error -> DSA_ERR_INVALID_ARG)
 *   context_lens [B] int32, 0 <= L_b <= max_blocks*block_size; L_b counts the
 *                request's next_n new tokens (a larger L_b is clamped and
 *                recorded like a bad block id)
 *   block_size   a power of two in [8, 128]
 *   logits       [B*next_n, ld] fp32 over LOGICAL key positions,
 *                ld >= max_blocks*block_size.  Row r = b*next_n + j sees keys
 *                [0, L_b - next_n + j + 1); the columns of every 128-key tile
 *                below L_b are written (-inf past the row's end).
 * Only block-table entries of blocks below ceil(L_b / block_size) are read.
 */
dsa_status_t dsa_indexer_logits_paged(const void* q, const float* q_scale,
                                      const float* weights, const void* k_cache,
                                      const float* k_scale, int num_blocks,
                                      dsa_dtype_t dtype,
                                      const int32_t* block_table, int max_blocks,
                                      const int32_t* context_lens, int B, int next_n,
                                      int block_size, int H, int D, float* logits,
                                      int64_t ld, dsa_stream_t stream);

/*
 * Paged decode logits + masked top-k.  Indices are logical positions within
 * the request.  `workspace` must hold
 * dsa_workspace_bytes(DSA_OP_INDEXER_TOPK_PAGED, B*next_n, max_blocks*block_size, k)
 * bytes, 256-byte aligned.  out is [B*next_n, k] int32.
 */
dsa_status_t dsa_indexer_topk_paged(const void* q, const float* q_scale,
                                    const float* weights, const void* k_cache,
                                    const float* k_scale, int num_blocks,
                                    dsa_dtype_t dtype,
                                    const int32_t* block_table, int max_blocks,
                                    const int32_t* context_lens, int B, int next_n,
                                    int block_size, int H, int D, int topk,
                                    int32_t* out, void* workspace, size_t ws_bytes,
                                    dsa_stream_t stream);

/*
 * dsa_indexer_topk for callers that cannot allocate device memory.  The pages
 * have no counterpart to this entry point; it is an addition of this library.
 *
 * Some callers have no way to obtain a scratch buffer when they need one:
 * plugins inside a host framework that owns every device allocation, or
 * latency-critical serving loops that must not pay for cudaMalloc's implicit
 * synchronisation.  This variant keeps its fp32 logits
 * in a fixed device array inside the library instead of a caller workspace;
 * it calls no allocator of any kind.
 *   - The array holds DSA_NOALLOC_SCRATCH_BYTES (64 MiB) on every GPU that
 *     loads the library, for the life of the process.
 *   - It covers T * round_up(S, 4) fp32 logits, i.e. at most
 *     DSA_NOALLOC_SCRATCH_BYTES / 4 of them (T = S = 4096 fits); a larger
 *     request returns DSA_ERR_UNSUPPORTED before anything is launched.
 *   - The first call on a device looks up the array's device address (once
 *     per device, under a lock).
 *   - Every call on a device uses the same array and leaves its logits there.
 *     Calls whose work overlaps on the GPU (several streams, or several host
 *     threads) race on it and corrupt each other's results: order them on one
 *     stream or with events.
 *   - Arguments and result are those of dsa_indexer_topk without the
 *     workspace; the indices are bit-identical to it.
 */
#define DSA_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
dsa_status_t dsa_indexer_topk_noalloc(const void* q, const float* q_scale, const void* k,
                                      const float* k_scale, dsa_dtype_t dtype,
                                      const float* weights, const int32_t* row_starts,
                                      const int32_t* row_ends, int T, int S, int H, int D,
                                      int topk, int32_t* out, dsa_stream_t stream);

/*
 * dsa_indexer_topk with the inputs and the result in HOST memory -- the only
 * entry point whose tensor pointers are not device pointers.  The pages have
 * no counterpart; it is an addition of this library for callers whose q, k
 * and weights start on the host.
 *   - q, q_scale, k, k_scale, weights, row_starts, row_ends, out: host
 *     pointers, same shapes, types and meaning as dsa_indexer_topk.  Pinned
 *     (page-locked) memory lets the copies overlap; pageable memory works but
 *     each copy then waits for the host.  The arrays indexed by row may be
 *     NULL when T = 0, k when S = 0.
 *   - device_buffer: caller-owned device memory of at least
 *     dsa_indexer_topk_host_bytes(T, S, H, D, topk, dtype) bytes, 256-byte
 *     aligned.  It receives the inputs, the indices and one row chunk's
 *     logits; on return from the stream's work it holds the device copy of
 *     the inputs and of `out`.
 *   - The rows are split into up to 12 chunks (whole rounds of the scoring
 *     kernel, 256/H rows times the current device's SM count, where a chunk
 *     holds one; else multiples of 64 rows; about 512 or more each), the
 *     remainder first; with three or more, the first and the last are cut
 *     down to one round (or 64 rows) each, the rest of each a chunk of its
 *     own.  So dsa_indexer_topk_host_bytes is for the current device.  K, the key scales and the row ranges go up first;
 *     then chunk c's queries and weights go up while chunk c-1 is scored and
 *     selected (on `stream`) and chunk c-2's indices come down, on two
 *     streams the call creates and destroys.  Work queued on
 *     `stream` after the call sees all of `out`; host code must synchronise
 *     `stream` before it reads `out`.
 *   - The copies are queued asynchronously and run after the call returns:
 *     every host input must stay allocated and unchanged, and `out` must not
 *     be read or freed, until `stream` has completed the call's work.
 *   - Not capturable into a CUDA graph (it creates streams and events).
 *   - Errors as dsa_indexer_topk; the indices are bit-identical to it.
 */
size_t dsa_indexer_topk_host_bytes(int T, int S, int H, int D, int topk, dsa_dtype_t dtype);
dsa_status_t dsa_indexer_topk_host(const void* q, const float* q_scale, const void* k,
                                   const float* k_scale, dsa_dtype_t dtype,
                                   const float* weights, const int32_t* row_starts,
                                   const int32_t* row_ends, int T, int S, int H, int D,
                                   int topk, int32_t* out, void* device_buffer,
                                   size_t device_bytes, dsa_stream_t stream);

/*
 * Reorders top-k rows in place into descending order of score: the order of
 * torch.topk, which torch_dsa_topk (vime PR #502, third review comment)
 * returns, where every other entry point here writes ascending column order.
 * Equal scores keep the lower column first (-0.0 equals +0.0), -inf and NaN
 * scores (which no top-k entry point selects) come after the others, and the
 * -1 padding stays at the tail.  The pages fix no order for a consumer; this
 * is the optional score-sorted output.
 *
 *   logits  [T, ld] fp32, the scores the indices refer to.  After
 *           dsa_indexer_topk or dsa_indexer_topk_paged they are still at the
 *           start of that call's workspace, with ld = round_up(S, 4) or
 *           round_up(max_blocks * block_size, 4), until it is reused.
 *   topk    [T, k] int32, read and rewritten.  An entry outside [0, ld) other
 *           than -1 is treated as padding (written back as -1, its column is
 *           never read) and reported by dsa_get_last_device_error as
 *           DSA_ERR_INVALID_ARG.  Entries inside [0, ld) are trusted: every
 *           top-k entry point here writes columns below its S only, but the
 *           columns [S, ld) of a composed call's workspace are row padding
 *           that no call writes, so an index there (from elsewhere) sorts on
 *           whatever that memory holds.  Pass ld = S when the indices may
 *           come from another source and S is a multiple of 4.
 *   k       1 .. 8192 (larger k: DSA_ERR_UNSUPPORTED)
 */
dsa_status_t dsa_topk_sort_by_score(const float* logits, int64_t ld, int32_t* topk, int T, int k,
                                    dsa_stream_t stream);

/*
 * Merge of per-rank top-k candidates into the global top-k (decode context
 * parallelism: KimiK3DSAIndexer.__init__ on the vLLM page, where each rank
 * scores its interleaved share of the key cache, takes a local top-k, and the
 * op merges the ranks' local top-k into the global top-k).  Per row, of the C
 * candidates (score, global column) -- typically W ranks x k, gathered by
 * one exchange -- the k best by score are kept (ties to the lower column,
 * -0.0 equal to +0.0, -inf and NaN never), and written in ascending column
 * order with -1 padding: exactly dsa_topk's output on the whole row, because
 * every column of the global top-k is in its rank's local top-k.
 *
 *   cand_scores [T, C] fp32
 *   cand_cols   [T, C] int32 global columns; a negative column is an empty slot.
 *               Columns must be distinct within a row (ranks own disjoint
 *               positions).
 *   out         [T, k] int32
 *   C, k <= 16384 (else DSA_ERR_UNSUPPORTED)
 */
dsa_status_t dsa_topk_merge(const float* cand_scores, const int32_t* cand_cols, int T, int C,
                            int k, int32_t* out, dsa_stream_t stream);

/*
 * dsa_topk_merge over candidates laid out rank-major, [W, T, kr] (rank w's
 * [T, kr] block at offset w * T * kr), as an all-gather of every rank's
 * dsa_topk_dcp_candidates output into one buffer leaves them: row t's
 * candidates are the W * kr entries (w, t, 0 .. kr-1).  Same result as
 * dsa_topk_merge on those candidates in any order.
 *
 *   cand_scores [W, T, kr] fp32, cand_cols [W, T, kr] int32 global columns
 *               (negative = empty slot; distinct within a row)
 *   out         [T, k] int32
 *   W * kr, k <= 16384 (else DSA_ERR_UNSUPPORTED)
 */
dsa_status_t dsa_topk_merge_ranks(const float* cand_scores, const int32_t* cand_cols, int W,
                                  int T, int kr, int k, int32_t* out, dsa_stream_t stream);

/*
 * One rank's candidates for the merge under decode context parallelism
 * (KimiK3DSAIndexer.__init__ on the vLLM page: the key cache is dealt to the
 * W ranks in runs of `interleave` consecutive positions, cp_kv_cache_
 * interleave_size, so rank r owns the positions p with (p / interleave) % W
 * == r, in order).  Per row, dsa_topk of the rank's local logits, written as
 * pairs: cand_cols[t, i] = the global position of the i-th selected local
 * column j, ((j / interleave) * W + rank) * interleave + j % interleave, and
 * cand_scores[t, i] = logits[t, j]; empty slots get -1 and -inf.  The pairs
 * follow the local columns' ascending order, so the global positions ascend
 * too.
 *
 *   logits      [T, ld] fp32 scores over the rank's own keys (local columns)
 *   row_starts, row_ends  [T] int32 local column ranges, as dsa_topk
 *   rank, world 0 <= rank < world
 *   interleave  >= 1
 *   cand_scores [T, k] fp32 out; cand_cols [T, k] int32 out
 *   workspace   dsa_workspace_bytes(DSA_OP_TOPK, T, S, k) bytes, as dsa_topk
 * A global position past INT32_MAX gives DSA_ERR_UNSUPPORTED.
 */
dsa_status_t dsa_topk_dcp_candidates(const float* logits, int64_t ld, const int32_t* row_starts,
                                     const int32_t* row_ends, int T, int S, int k, int rank,
                                     int world, int interleave, float* cand_scores,
                                     int32_t* cand_cols, void* workspace, size_t ws_bytes,
                                     dsa_stream_t stream);

/*
 * The query side of the e4m3 path, before dsa_indexer_logits / _topk /
 * _topk_paged: indexer_q_quant_fold_weights of KimiK3DSAIndexer.score (vLLM
 * API docs, "vllm.models.kimi_k3.nvidia.dsa").  Every (t, h) row of D query
 * elements becomes e4m3 codes with one UE8M0 scale s (the smallest power of
 * two with max|q[t,h,:]| <= 448 s; 1 for an all-zero row), codes = q / s
 * rounded to nearest even; the scale is folded into the weight,
 * weights_out[t,h] = fl32(fl32(weights[t,h] * weight_scale) * s), so the
 * scoring calls take q_scale = NULL.  Heads H .. padded_heads-1 get zero codes
 * and zero weights (the page pads to 32 or 64 index heads).
 *
 *   q            [T, H, D] bf16, 16-byte aligned
 *   weights      [T, H] fp32
 *   weight_scale the page's index_softmax_scale * indexer_weight_scale
 *   q_fp8        [T, padded_heads, D] e4m3 output, 8-byte aligned
 *   weights_out  [T, padded_heads] fp32 output
 *   D = 128, H <= padded_heads <= 64 (else DSA_ERR_UNSUPPORTED)
 */
dsa_status_t dsa_q_quant_fold_weights(const void* q, const float* weights, float weight_scale,
                                      int T, int H, int D, int padded_heads, void* q_fp8,
                                      float* weights_out, dsa_stream_t stream);

/*
 * The key side: indexer_k_norm_quant_insert of KimiK3DSAIndexer._fused_k_insert
 * with KimiK3DSAIndexerKNorm (same page).  Every new key row goes through the
 * bias-full LayerNorm in fp32 -- (k - mean) / sqrt(var + eps) * ln_weight +
 * ln_bias, population variance -- is cast back to bf16, and is written to
 * row slot_mapping[t] of the paged cache (block slot / block_size, row
 * slot % block_size): as bf16 (DSA_BF16), or as e4m3 codes with one UE8M0
 * scale per row like the query side (DSA_E4M3, scale to k_scale[slot]).
 *
 *   k            [T, D] bf16 new keys, 16-byte aligned
 *   ln_weight, ln_bias  [D] fp32, 16-byte aligned
 *   slot_mapping [T] int64: a slot below 0 marks a padding token (skipped);
 *                a slot >= num_blocks * block_size is skipped and reported
 *                by dsa_get_last_device_error as DSA_ERR_INVALID_ARG
 *   k_cache      [num_blocks, block_size, D] of cache_dtype, the layout
 *                dsa_indexer_logits_paged reads
 *   k_scale      [num_blocks * block_size] fp32 for DSA_E4M3, NULL for bf16
 *   D = 128 (else DSA_ERR_UNSUPPORTED)
 */
dsa_status_t dsa_k_norm_quant_insert(const void* k, const float* ln_weight, const float* ln_bias,
                                     float eps, const int64_t* slot_mapping, int T, int D,
                                     dsa_dtype_t cache_dtype, void* k_cache, float* k_scale,
                                     int num_blocks, int block_size, dsa_stream_t stream);

/*
 * Scratch bytes an operation needs.  rows/cols are T/S for the prefill ops and
 * B*next_n / max_blocks*block_size for the paged ones; k is index_topk.  The
 * composed calls need the fp32 logits (rows * round_up(cols, 4) floats, padded
 * to 256 bytes) plus, for few long rows, the top-k scratch (about 75 KiB per
 * row).
 * Returns 0 for operations that need none, and (size_t)-1 for bad arguments.
 */
size_t dsa_workspace_bytes(dsa_op_t op, int64_t rows, int64_t cols, int k);

/* Static description of a status code (never NULL). */
const char* dsa_status_string(dsa_status_t status);

/*
 * Synchronises the current device, then reports and clears the sticky
 * device-side error word of the current device: DSA_ERR_TIMEOUT when a
 * kernel's bounded wait gave up since the last call, DSA_ERR_INVALID_ARG when
 * a paged call met a block id or context length out of range (or
 * dsa_topk_sort_by_score an index outside its row, or
 * dsa_k_norm_quant_insert a slot past the cache), DSA_ERR_CUDA
 * when the synchronisation itself failed, else DSA_OK.
 */
dsa_status_t dsa_get_last_device_error(void);

/*
 * Failure-detection self test: launches one block whose thread waits on a
 * shared-memory barrier that nothing ever arrives on, giving up after
 * timeout_ns nanoseconds (clamped to [1e3, 1e9]).  The kernel then records a
 * timeout in the device error word and returns normally, so the context
 * stays usable; dsa_get_last_device_error() reports DSA_ERR_TIMEOUT.
 */
dsa_status_t dsa_selftest_wait_timeout(uint64_t timeout_ns, dsa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DSA_H_ */
