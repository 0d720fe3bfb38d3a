/*
 * dsa_oracle.c -- plain, slow CPU oracle for the DSA lightning-indexer path.
 *
 * TEST INFRASTRUCTURE ONLY.  The product library never links, loads or calls
 * this file.  Only the test-suite, the package smoke check and the CPU
 * baseline leg of the benchmark use it.  It shares no code, header, table or
 * constant with the CUDA path.
 *
 * Everything is computed in double precision, straight from the definitions:
 * no blocking, no fusion and no reordering of the arithmetic.  The only
 * liberty taken is an OpenMP loop over independent query rows.
 *
 * Sources (web pages):
 *   [vLLM-dsa]  vLLM API docs, "vllm.models.kimi_k3.nvidia.dsa":
 *               - KimiK3DSAIndexer.__init__: index-cache scales are UE8M0
 *                 (power-of-two, read back as exact fp32) with
 *                 quant_block_size = index_head_dim; index heads padded with
 *                 zero heads;
 *               - KimiK3DSAIndexer.score: the query scale and the
 *                 softmax/head scales are folded into the per-head weights
 *                 before torch.ops.vllm.sparse_attn_indexer is called with
 *                 index_q [T,H,D], the shared index_k [T,D] and weights [T,H];
 *               - KimiK3DSAIndexer.__init__: the paged indexer K cache
 *                 (KimiK3IndexerCache, slot-addressed).
 *   [vime-502]  GitHub "vllm-project/vime" pull request #502, third review
 *               comment: the corrected torch_dsa_topk fallback (mask columns
 *               outside [row_start,row_end) to -inf, top-k, -1 where the
 *               score is -inf, -1 padding when k exceeds the row).
 *   [OCP-FP8]   the OCP 8-bit floating point specification, E4M3 encoding
 *               (bias 7, no infinities, S.1111.111 is NaN, max 448).
 *   [OCP-MX]    the OCP Microscaling Formats (MX) specification: MXFP4 =
 *               E2M1 elements (bias 1, max 6) in blocks of 32 sharing one
 *               E8M0 scale 2^(e-127).
 *
 * The index score itself is the DeepSeek sparse-attention lightning indexer:
 *     logit[t,s] = sum_h w[t,h] * max(0, sum_d q[t,h,d] * k[s,d])
 * taken over the columns s of row t's range; every other column is -inf.
 *
 * Readings taken where the pages are silent (each one also listed in the
 * design notes of the repository):
 *   - row ranges are half-open [row_start, row_end), clamped to [0, S);
 *     an empty or inverted range yields an all -1 row;
 *   - top-k ties go to the lower column index; -0.0 equals +0.0 (IEEE);
 *   - NaN is treated like -inf: never selected, not counted as valid;
 *   - the selected columns are written in ascending column order, followed by
 *     -1 padding up to k;
 *   - paged decode: a request of context length L owns logical key positions
 *     [0, L); its query j (0 <= j < next_n) sees keys [0, L - next_n + j + 1);
 *     returned indices are logical positions.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_BF16 = 0, ORACLE_E4M3 = 1 };

/* ------------------------------------------------------------------ decode */

/* bf16 is the upper half of an IEEE binary32: widen the bit pattern. */
double dsa_oracle_bf16_to_f64(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* E4M3 per [OCP-FP8]: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits.
 * Exponent field 0 is subnormal (m/8 * 2^-6); the all-ones pattern
 * S.1111.111 is NaN; there is no infinity, so S.1111.110 = 448 is the max. */
double dsa_oracle_e4m3_to_f64(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double mag;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, 1 - 7);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -mag : mag;
}

static double decode_elem(const void* base, int dtype, int64_t i)
{
    if (dtype == ORACLE_BF16)
        return dsa_oracle_bf16_to_f64(((const uint16_t*)base)[i]);
    return dsa_oracle_e4m3_to_f64(((const uint8_t*)base)[i]);
}

static int clamp64(int64_t v, int64_t lo, int64_t hi)
{
    return (int)(v < lo ? lo : (v > hi ? hi : v));
}

static void set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

/* One logit from dequantised operands.
 * qrow: [H, D] dequantised query of token t (its block scales applied);
 * krow: [D] dequantised key; w: [H] per-head weights of token t. */
static double index_score(const double* qrow, const double* krow,
                          const float* w, int H, int D)
{
    double logit = 0.0;
    for (int h = 0; h < H; ++h) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
            dot += qrow[(int64_t)h * D + d] * krow[d];
        double relu = dot > 0.0 ? dot : 0.0;
        logit += (double)w[h] * relu;
    }
    return logit;
}

/* Dequantise the query of token t into qrow[H*D].
 * q_scale (optional, [T,H]): one power-of-two scale per (t,h) block of D
 * elements (quant_block_size = index_head_dim in [vLLM-dsa]). */
static void load_query(const void* q, const float* q_scale, int dtype,
                       int64_t t, int H, int D, double* qrow)
{
    for (int h = 0; h < H; ++h) {
        double sc = q_scale ? (double)q_scale[t * H + h] : 1.0;
        for (int d = 0; d < D; ++d)
            qrow[(int64_t)h * D + d] =
                decode_elem(q, dtype, (t * H + h) * (int64_t)D + d) * sc;
    }
}

/* ------------------------------------------------------- prefill logits */

/*
 * Dense index logits over a contiguous key set.
 *   q        [T, H, D]  bf16 bits (uint16) or e4m3 codes (uint8), row-major
 *   q_scale  NULL or [T, H] fp32 block scales of q
 *   k        [S, D]     same element type as q
 *   k_scale  NULL or [S] fp32 block scales of k (one per key row)
 *   w        [T, H]     fp32 per-head weights (scales already folded in)
 *   row_starts/row_ends [T] int32, half-open range of row t
 *   rows     NULL (all T rows) or nrows row ids to evaluate
 *   out      [nrows, S] fp64; -inf outside the clamped range
 * Returns 0, or -1 on a bad argument.
 */
int dsa_oracle_logits(const void* q, const float* q_scale, const void* k,
                      const float* k_scale, int dtype, const float* w,
                      const int32_t* row_starts, const int32_t* row_ends,
                      int64_t T, int64_t S, int H, int D,
                      const int64_t* rows, int64_t nrows, double* out,
                      int nthreads)
{
    if (!q || !k || !w || !row_starts || !row_ends || !out || T < 0 ||
        S < 0 || H < 1 || D < 1 || (dtype != ORACLE_BF16 && dtype != ORACLE_E4M3))
        return -1;
    if (!rows)
        nrows = T;
    double* kd = (double*)malloc(sizeof(double) * (size_t)(S * D + 1));
    if (!kd)
        return -1;
    for (int64_t s = 0; s < S; ++s) {
        double sc = k_scale ? (double)k_scale[s] : 1.0;
        for (int d = 0; d < D; ++d)
            kd[s * D + d] = decode_elem(k, dtype, s * D + d) * sc;
    }
    int bad = 0;
    set_threads(nthreads);
#pragma omp parallel
    {
        double* qrow = (double*)malloc(sizeof(double) * (size_t)H * D);
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < nrows; ++i) {
            int64_t t = rows ? rows[i] : i;
            double* o = out + i * S;
            if (t < 0 || t >= T || !qrow) {
                bad = 1;
                continue;
            }
            int lo = clamp64(row_starts[t], 0, S);
            int hi = clamp64(row_ends[t], 0, S);
            load_query(q, q_scale, dtype, t, H, D, qrow);
            for (int64_t s = 0; s < S; ++s) {
                if (s >= lo && s < hi)
                    o[s] = index_score(qrow, kd + s * D, w + t * H, H, D);
                else
                    o[s] = -INFINITY;
            }
        }
        free(qrow);
    }
    free(kd);
    return bad ? -1 : 0;
}

/* ---------------------------------------------------- MXFP4 (OCP MX) */

/* E2M1 per [OCP-MX]: a 4-bit code S.EE.M, exponent bias 1.  E = 0 is
 * subnormal (M/2); otherwise (1 + M/2) * 2^(E-1).  Magnitudes 0, 0.5, 1, 1.5,
 * 2, 3, 4, 6; no infinities or NaN.  Only the low 4 bits of `code` count. */
double dsa_oracle_e2m1_to_f64(uint8_t code)
{
    int sign = (code >> 3) & 1;
    int e = (code >> 1) & 3;
    int m = code & 1;
    double mag = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return sign ? -mag : mag;
}

/* E8M0 (UE8M0) scale per [OCP-MX]: 2^(code - 127); code 255 is NaN. */
double dsa_oracle_e8m0_to_f64(uint8_t code)
{
    if (code == 255)
        return NAN;
    return ldexp(1.0, (int)code - 127);
}

/* Element i of a packed E2M1 array: byte i/2, the low nibble for even i. */
static double mxfp4_elem(const uint8_t* packed, const uint8_t* scales, int64_t i)
{
    uint8_t byte = packed[i / 2];
    uint8_t code = (i & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15);
    return dsa_oracle_e2m1_to_f64(code) * dsa_oracle_e8m0_to_f64(scales[i / 32]);
}

/*
 * Dense index logits with MXFP4 queries and keys ([vLLM-dsa]: MXFP4 keys with
 * MXFP4 queries, mxfp4_q_quant returning a separate q_scale): every block of
 * 32 consecutive elements of a row shares one E8M0 scale.
 *   q     [T, H, D/2] packed E2M1, q_sf [T, H, D/32] E8M0 codes
 *   k     [S, D/2]    packed E2M1, k_sf [S, D/32]    E8M0 codes
 *   w     [T, H] fp32 (the query scale is NOT folded in: it is in q_sf)
 * The rest as dsa_oracle_logits.  D must be a multiple of 32.
 */
int dsa_oracle_logits_mxfp4(const uint8_t* q, const uint8_t* q_sf, const uint8_t* k,
                            const uint8_t* k_sf, const float* w, const int32_t* row_starts,
                            const int32_t* row_ends, int64_t T, int64_t S, int H, int D,
                            const int64_t* rows, int64_t nrows, double* out, int nthreads)
{
    if (!q || !q_sf || !k || !k_sf || !w || !row_starts || !row_ends || !out || T < 0 ||
        S < 0 || H < 1 || D < 32 || D % 32 != 0)
        return -1;
    if (!rows)
        nrows = T;
    double* kd = (double*)malloc(sizeof(double) * (size_t)(S * D + 1));
    if (!kd)
        return -1;
    for (int64_t s = 0; s < S; ++s)
        for (int d = 0; d < D; ++d)
            kd[s * D + d] = mxfp4_elem(k + s * (D / 2), k_sf + s * (D / 32), d);
    int bad = 0;
    set_threads(nthreads);
#pragma omp parallel
    {
        double* qrow = (double*)malloc(sizeof(double) * (size_t)H * D);
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < nrows; ++i) {
            int64_t t = rows ? rows[i] : i;
            double* o = out + i * S;
            if (t < 0 || t >= T || !qrow) {
                bad = 1;
                continue;
            }
            int lo = clamp64(row_starts[t], 0, S);
            int hi = clamp64(row_ends[t], 0, S);
            for (int h = 0; h < H; ++h) {
                int64_t r = t * H + h;
                for (int d = 0; d < D; ++d)
                    qrow[(int64_t)h * D + d] = mxfp4_elem(q + r * (D / 2), q_sf + r * (D / 32), d);
            }
            for (int64_t s = 0; s < S; ++s) {
                if (s >= lo && s < hi)
                    o[s] = index_score(qrow, kd + s * D, w + t * H, H, D);
                else
                    o[s] = -INFINITY;
            }
        }
        free(qrow);
    }
    free(kd);
    return bad ? -1 : 0;
}

/* --------------------------------------------------------- paged decode */

/*
 * Row ranges of paged decode.  Request b (context length L_b, which counts its
 * next_n new tokens) owns query rows r = b*next_n + j, j in [0, next_n); row r
 * sees logical keys [0, L_b - next_n + j + 1), clamped at 0.
 */
int dsa_oracle_paged_row_ranges(const int32_t* context_lens, int B, int next_n,
                                int32_t* row_starts, int32_t* row_ends)
{
    if (!context_lens || !row_starts || !row_ends || B < 0 || next_n < 1)
        return -1;
    for (int b = 0; b < B; ++b)
        for (int j = 0; j < next_n; ++j) {
            int64_t end = (int64_t)context_lens[b] - next_n + j + 1;
            row_starts[b * next_n + j] = 0;
            row_ends[b * next_n + j] = (int32_t)(end < 0 ? 0 : end);
        }
    return 0;
}

/*
 * Index logits of paged decode.  Logical key s of request b lives in physical
 * block block_table[b, s / block_size] at slot s % block_size of
 * k_cache [num_blocks, block_size, D]; k_scale (optional) is
 * [num_blocks, block_size].
 *   q  [B*next_n, H, D],  w [B*next_n, H]
 *   out [nrows, ld] fp64 over logical positions; -inf outside the row range.
 */
int dsa_oracle_logits_paged(const void* q, const float* q_scale,
                            const void* k_cache, const float* k_scale, int dtype,
                            const float* w, const int32_t* block_table,
                            int64_t max_blocks, const int32_t* context_lens,
                            int B, int next_n, int block_size, int H, int D,
                            const int64_t* rows, int64_t nrows, int64_t ld,
                            double* out, int nthreads)
{
    if (!q || !k_cache || !w || !block_table || !context_lens || !out || B < 0 ||
        next_n < 1 || block_size < 1 || H < 1 || D < 1 || ld < 0 ||
        (dtype != ORACLE_BF16 && dtype != ORACLE_E4M3))
        return -1;
    int64_t R = (int64_t)B * next_n;
    if (!rows)
        nrows = R;
    int bad = 0;
    set_threads(nthreads);
#pragma omp parallel
    {
        double* qrow = (double*)malloc(sizeof(double) * (size_t)H * D);
        double* krow = (double*)malloc(sizeof(double) * (size_t)D);
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < nrows; ++i) {
            int64_t r = rows ? rows[i] : i;
            double* o = out + i * ld;
            if (r < 0 || r >= R || !qrow || !krow) {
                bad = 1;
                continue;
            }
            int b = (int)(r / next_n), j = (int)(r % next_n);
            int64_t end = (int64_t)context_lens[b] - next_n + j + 1;
            if (end < 0)
                end = 0;
            if (end > ld || (end + block_size - 1) / block_size > max_blocks) {
                bad = 1;
                continue;
            }
            load_query(q, q_scale, dtype, r, H, D, qrow);
            for (int64_t s = 0; s < ld; ++s) {
                if (s >= end) {
                    o[s] = -INFINITY;
                    continue;
                }
                int64_t blk = block_table[b * max_blocks + s / block_size];
                int64_t slot = blk * block_size + s % block_size;
                double sc = k_scale ? (double)k_scale[slot] : 1.0;
                for (int d = 0; d < D; ++d)
                    krow[d] = decode_elem(k_cache, dtype, slot * D + d) * sc;
                o[s] = index_score(qrow, krow, w + r * H, H, D);
            }
        }
        free(qrow);
        free(krow);
    }
    return bad ? -1 : 0;
}

/* ------------------------------------------------------------------ top-k */

typedef struct {
    float v;
    int32_t c;
} cand_t;

/* Larger score first; equal scores (IEEE equality, so -0.0 == +0.0) by the
 * lower column. */
static int by_score_then_column(const void* a, const void* b)
{
    const cand_t* x = (const cand_t*)a;
    const cand_t* y = (const cand_t*)b;
    if (x->v > y->v)
        return -1;
    if (x->v < y->v)
        return 1;
    return (x->c > y->c) - (x->c < y->c);
}

static int by_column(const void* a, const void* b)
{
    int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
    return (x > y) - (x < y);
}

/*
 * Masked per-row top-k of given fp32 logits, after torch_dsa_topk in
 * [vime-502]: columns outside [row_start,row_end) are excluded, a -inf (or
 * NaN) score is never selected, and the row is padded with -1 up to k.
 *   logits [T, ld] fp32; only columns [0, S) are considered
 *   out    [T, k]  int32: selected columns ascending, then -1
 */
int dsa_oracle_topk(const float* logits, int64_t ld, const int32_t* row_starts,
                    const int32_t* row_ends, int64_t T, int64_t S, int k,
                    int32_t* out, int nthreads)
{
    if (!logits || !row_starts || !row_ends || !out || T < 0 || S < 0 || k < 1 ||
        ld < S)
        return -1;
    int bad = 0;
    set_threads(nthreads);
#pragma omp parallel
    {
        cand_t* cand = (cand_t*)malloc(sizeof(cand_t) * (size_t)(S + 1));
        int32_t* pick = (int32_t*)malloc(sizeof(int32_t) * (size_t)k);
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < T; ++t) {
            if (!cand || !pick) {
                bad = 1;
                continue;
            }
            const float* row = logits + t * ld;
            int lo = clamp64(row_starts[t], 0, S);
            int hi = clamp64(row_ends[t], 0, S);
            int n = 0;
            for (int c = lo; c < hi; ++c) {
                float v = row[c];
                if (isnan(v) || v == -INFINITY)
                    continue;
                cand[n].v = v;
                cand[n].c = c;
                ++n;
            }
            qsort(cand, (size_t)n, sizeof(cand_t), by_score_then_column);
            int m = n < k ? n : k;
            for (int i = 0; i < m; ++i)
                pick[i] = cand[i].c;
            qsort(pick, (size_t)m, sizeof(int32_t), by_column);
            for (int i = 0; i < k; ++i)
                out[t * k + i] = i < m ? pick[i] : -1;
        }
        free(cand);
        free(pick);
    }
    return bad ? -1 : 0;
}

int dsa_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------- prologue
 *
 * The two steps just before the indexer on [vLLM-dsa]:
 *   - KimiK3DSAIndexer.score: indexer_q_quant_fold_weights(index_q,
 *     index_weights, weight_scale, padded_index_num_heads) -- the query rows
 *     quantised to e4m3 with one UE8M0 scale each, the scale and weight_scale
 *     folded into the head weights, heads padded with zeros;
 *   - KimiK3DSAIndexer._fused_k_insert + KimiK3DSAIndexerKNorm:
 *     indexer_k_norm_quant_insert -- F.layer_norm(x.float(), (D,), weight,
 *     bias, eps).type_as(x) (fp32 LayerNorm, cast back to bf16), then the
 *     row quantised like the query and written to its slot of the paged
 *     cache.
 * The pages show only the calls.  Readings: the UE8M0 scale of a row is the
 * smallest power of two s with max|x| <= 448 s (s = 1 for an all-zero row);
 * codes are x / s rounded to the nearest E4M3 value, ties to the even code,
 * saturating at 448; the folded weight is fl32(fl32(w * weight_scale) * s);
 * a negative slot is a padding token; the LayerNorm uses the population
 * variance.  The LayerNorm itself is computed here in double precision and
 * rounded once to bf16 (the pages fix fp32; results agree to within one bf16
 * step, which the tests allow). */

/* Nearest E4M3 code to v per [OCP-FP8]: the positive codes 0x00..0x7E are
 * decoded and searched for the closest value; an exact tie goes to the even
 * code (mantissa LSB 0); magnitudes above 448 saturate to 0x7E.  The sign
 * bit follows v's sign bit (so -0.0 -> 0x80).  v must not be NaN. */
uint8_t dsa_oracle_f64_to_e4m3(double v)
{
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs(v);
    int best = 0;
    double best_d = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        double d = fabs(dsa_oracle_e4m3_to_f64((uint8_t)c) - a);
        if (d < best_d || (d == best_d && (c & 1) == 0)) {
            best = c;
            best_d = d;
        }
    }
    return (uint8_t)(sign | best);
}

/* Exponent e of the UE8M0 scale 2^e: smallest integer with amax <= 448 * 2^e. */
static int ue8m0_exp(double amax)
{
    if (!(amax > 0.0))
        return 0;
    int e = -160;
    while (amax > 448.0 * ldexp(1.0, e))
        ++e;
    return e;
}

/* v rounded once to bf16 (the upper half of a binary32): of the two bf16
 * values around |v|, the nearer one, ties to the even one; v's sign kept. */
static uint16_t f64_to_bf16_rne(double v)
{
    double a = fabs(v);
    float fa = (float)a;
    uint32_t u;
    memcpy(&u, &fa, sizeof u);
    uint32_t lo = u & 0xFFFF0000u;          /* a bf16 value at or near a */
    float flo;
    memcpy(&flo, &lo, sizeof flo);
    if ((double)flo > a)                    /* fa was rounded up onto a bf16 value */
        lo -= 0x10000u;
    uint32_t hi = lo + 0x10000u;
    float f_lo, f_hi;
    memcpy(&f_lo, &lo, sizeof f_lo);
    memcpy(&f_hi, &hi, sizeof f_hi);
    double dl = a - (double)f_lo, dh = (double)f_hi - a;
    uint32_t r = dl < dh ? lo : (dh < dl ? hi : (((lo >> 16) & 1u) ? hi : lo));
    return (uint16_t)((r >> 16) | (signbit(v) ? 0x8000u : 0u));
}

/* q [T,H,D] bf16 -> q8 [T,Hp,D] e4m3 codes and w_out [T,Hp] fp32. */
int dsa_oracle_q_quant_fold(const uint16_t* q, const float* w, float weight_scale, int T, int H,
                            int D, int Hp, uint8_t* q8, float* w_out)
{
    if (!q || !w || !q8 || !w_out || T < 0 || H < 1 || Hp < H || D < 1)
        return -1;
    for (int64_t t = 0; t < T; ++t) {
        for (int h = 0; h < Hp; ++h) {
            uint8_t* dst = q8 + (t * Hp + h) * D;
            if (h >= H) {
                memset(dst, 0, (size_t)D);
                w_out[t * Hp + h] = 0.0f;
                continue;
            }
            const uint16_t* src = q + (t * H + h) * D;
            double amax = 0.0;
            for (int d = 0; d < D; ++d) {
                double x = fabs(dsa_oracle_bf16_to_f64(src[d]));
                if (x > amax)
                    amax = x;
            }
            int e = ue8m0_exp(amax);
            for (int d = 0; d < D; ++d)
                dst[d] = dsa_oracle_f64_to_e4m3(ldexp(dsa_oracle_bf16_to_f64(src[d]), -e));
            float wf = w[t * H + h] * weight_scale;          /* fl32(w * weight_scale) */
            w_out[t * Hp + h] = (float)((double)wf * ldexp(1.0, e));
        }
    }
    return 0;
}

/* The bias-full LayerNorm of KimiK3DSAIndexerKNorm on one bf16 row of D
 * elements, in double and not rounded: (x - mean) / sqrt(var + eps) *
 * gamma + beta, population variance. */
static void layer_norm_row(const uint16_t* src, const float* gamma, const float* beta, float eps,
                           int D, double* out)
{
    double mean = 0.0, var = 0.0;
    for (int d = 0; d < D; ++d)
        mean += dsa_oracle_bf16_to_f64(src[d]);
    mean /= D;
    for (int d = 0; d < D; ++d) {
        double c = dsa_oracle_bf16_to_f64(src[d]) - mean;
        var += c * c;
    }
    var /= D;
    double rstd = 1.0 / sqrt(var + (double)eps);
    for (int d = 0; d < D; ++d)
        out[d] = (dsa_oracle_bf16_to_f64(src[d]) - mean) * rstd * gamma[d] + beta[d];
}

/* k [T,D] bf16 -> out [T,D]: the LayerNorm values before the cast back to
 * bf16 (what the rounding of dsa_oracle_k_norm_insert starts from). */
int dsa_oracle_k_layer_norm(const uint16_t* k, const float* gamma, const float* beta, float eps,
                            int T, int D, double* out)
{
    if (!k || !gamma || !beta || !out || T < 0 || D < 1)
        return -1;
    for (int64_t t = 0; t < T; ++t)
        layer_norm_row(k + t * D, gamma, beta, eps, D, out + t * D);
    return 0;
}

/* k [T,D] bf16 -> LayerNorm -> bf16 -> the cache row at slots[t].
 * dtype 0: cache holds bf16 (uint16) rows; 1: e4m3 codes + scale[slot]. */
int dsa_oracle_k_norm_insert(const uint16_t* k, const float* gamma, const float* beta, float eps,
                             const int64_t* slots, int T, int D, int dtype, int64_t capacity,
                             void* cache, float* scale)
{
    if (!k || !gamma || !beta || !slots || !cache || T < 0 || D < 1 || (dtype == 1 && !scale))
        return -1;
    double* y = (double*)malloc(sizeof(double) * (size_t)D);
    if (!y)
        return -1;
    for (int64_t t = 0; t < T; ++t) {
        int64_t slot = slots[t];
        if (slot < 0 || slot >= capacity)
            continue;
        layer_norm_row(k + t * D, gamma, beta, eps, D, y);
        for (int d = 0; d < D; ++d)
            y[d] = dsa_oracle_bf16_to_f64(f64_to_bf16_rne(y[d]));   /* .type_as(x) */
        if (dtype == 0) {
            uint16_t* dst = (uint16_t*)cache + slot * D;
            for (int d = 0; d < D; ++d)
                dst[d] = f64_to_bf16_rne(y[d]);
        } else {
            uint8_t* dst = (uint8_t*)cache + slot * D;
            double amax = 0.0;
            for (int d = 0; d < D; ++d)
                if (fabs(y[d]) > amax)
                    amax = fabs(y[d]);
            int e = ue8m0_exp(amax);
            for (int d = 0; d < D; ++d)
                dst[d] = dsa_oracle_f64_to_e4m3(ldexp(y[d], -e));
            scale[slot] = (float)ldexp(1.0, e);
        }
    }
    free(y);
    return 0;
}
