// dsa_prologue.cu -- the two steps just before the indexer (sm_103a):
//
//   q quantisation + weight fold  (KimiK3DSAIndexer.score, vLLM API docs
//     "vllm.models.kimi_k3.nvidia.dsa": indexer_q_quant_fold_weights(index_q,
//     index_weights, weight_scale, padded_index_num_heads)).  Every (t, h) row
//     of D = 128 query elements becomes e4m3 codes with one power-of-two
//     (UE8M0) scale; the scale times weight_scale is folded into the head
//     weight, so the scoring kernel needs no query scale; heads are padded to
//     the padded head count with zero codes and zero weights.
//   K norm + quantise + paged insert  (KimiK3DSAIndexer._fused_k_insert and
//     KimiK3DSAIndexerKNorm on the same page: indexer_k_norm_quant_insert).
//     Every new key row goes through the bias-full fp32 LayerNorm, is cast
//     back to bf16, and is written to its slot of the paged cache -- as bf16,
//     or as e4m3 codes with one UE8M0 scale per row.
//
// Readings where the page shows only the call: the UE8M0 scale of a row is
// the smallest power of two s with amax <= 448 s (1 for an all-zero row),
// codes are x / s rounded to nearest even and saturated to +-448; the folded
// weight is fl32(fl32(w * weight_scale) * s); a slot below 0 is a padding
// token and is skipped; a slot past the cache is skipped and reported.
//
// Both are memory-bound: 16 lanes per row, 16-byte loads, one row's codes in
// 8 bytes per lane.
#include <cuda_bf16.h>

#include "dsa_common.cuh"
#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr int kRowLanes = 16;           // lanes per 128-element row
constexpr int kProThreads = 256;
constexpr int kRowsPerCta = kProThreads / kRowLanes;

// Exponent e of the UE8M0 scale 2^e of a row whose largest magnitude is amax:
// the smallest e with amax <= 448 * 2^e (448 = 0.875 * 2^9), 0 for amax == 0.
__device__ __forceinline__ int ue8m0_exponent(float amax) {
  if (!(amax > 0.f)) return 0;
  int x;
  const float m = frexpf(amax, &x);  // amax = m * 2^x, m in [0.5, 1)
  return m <= 0.875f ? x - 9 : x - 8;
}

// Two fp32 values -> two e4m3 codes (round to nearest even, saturating); lo
// lands in the low byte.
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float half_warp_max(float v) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float half_warp_sum(float v) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4 u, float (&x)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// Eight values scaled by 2^-e (exact) -> eight e4m3 codes.
__device__ __forceinline__ uint2 quantize8(const float (&x)[8], int e) {
  const float inv = ldexpf(1.f, -e);
  uint32_t c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) c[i] = e4m3x2(x[2 * i] * inv, x[2 * i + 1] * inv);
  return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

// Each half-warp takes kQRows consecutive (t, h) rows per step, all loads
// issued before any is used (64 bytes in flight per lane).
constexpr int kQRows = 4;

__global__ void __launch_bounds__(kProThreads) q_quant_fold_kernel(
    const uint16_t* __restrict__ q, const float* __restrict__ w, float weight_scale, int T,
    int H, int Hp, uint8_t* __restrict__ q8, float* __restrict__ w_out) {
  const int sub = threadIdx.x & (kRowLanes - 1);
  const int64_t rows = static_cast<int64_t>(T) * Hp;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kRowsPerCta * kQRows;
  for (int64_t base = (static_cast<int64_t>(blockIdx.x) * kRowsPerCta + threadIdx.x / kRowLanes) *
                      kQRows;
       base < rows; base += stride) {
    uint4 raw[kQRows];
    float wv[kQRows];
#pragma unroll
    for (int r = 0; r < kQRows; ++r) {
      const int64_t row = base + r;
      const int64_t t = row / Hp;
      const int h = static_cast<int>(row - t * Hp);
      raw[r] = make_uint4(0u, 0u, 0u, 0u);
      wv[r] = 0.f;
      if (row < rows && h < H) {
        raw[r] = __ldg(reinterpret_cast<const uint4*>(q + (t * H + h) * 128) + sub);
        if (sub == 0) wv[r] = __ldg(w + t * H + h);
      }
    }
#pragma unroll
    for (int r = 0; r < kQRows; ++r) {
      const int64_t row = base + r;
      if (row >= rows) break;  // uniform across the half-warp
      // A padded head (h >= H) was loaded as zeros: zero codes, scale 1,
      // and a zero weight.
      float x[8];
      bf16x8_to_f32(raw[r], x);
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
      amax = half_warp_max(amax);
      const int e = ue8m0_exponent(amax);
      *reinterpret_cast<uint2*>(q8 + row * 128 + sub * 8) = quantize8(x, e);
      if (sub == 0) w_out[row] = (wv[r] * weight_scale) * ldexpf(1.f, e);
    }
  }
}

__global__ void __launch_bounds__(kProThreads) k_norm_insert_kernel(
    const uint16_t* __restrict__ k, const float* __restrict__ gamma,
    const float* __restrict__ beta, float eps, const int64_t* __restrict__ slots, int T,
    bool fp8, int64_t capacity, uint8_t* __restrict__ cache, float* __restrict__ cache_scale,
    uint32_t* err) {
  const int sub = threadIdx.x & (kRowLanes - 1);
  float g[8], b[8];
  {
    const float4 g0 = __ldg(reinterpret_cast<const float4*>(gamma) + 2 * sub);
    const float4 g1 = __ldg(reinterpret_cast<const float4*>(gamma) + 2 * sub + 1);
    const float4 b0 = __ldg(reinterpret_cast<const float4*>(beta) + 2 * sub);
    const float4 b1 = __ldg(reinterpret_cast<const float4*>(beta) + 2 * sub + 1);
    g[0] = g0.x; g[1] = g0.y; g[2] = g0.z; g[3] = g0.w; g[4] = g1.x; g[5] = g1.y; g[6] = g1.z; g[7] = g1.w;
    b[0] = b0.x; b[1] = b0.y; b[2] = b0.z; b[3] = b0.w; b[4] = b1.x; b[5] = b1.y; b[6] = b1.z; b[7] = b1.w;
  }
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * kRowsPerCta + threadIdx.x / kRowLanes;
       t < T; t += static_cast<int64_t>(gridDim.x) * kRowsPerCta) {
    const int64_t slot = __ldg(slots + t);
    if (slot < 0) continue;  // padding token (uniform across the row's lanes)
    if (slot >= capacity) {
      if (sub == 0) record_error(err, kErrBadIndex);
      continue;
    }
    float x[8];
    bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(k + t * 128) + sub), x);
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) s += x[i];
    const float mean = half_warp_sum(s) * (1.f / 128.f);
    float v = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) v += (x[i] - mean) * (x[i] - mean);
    const float rstd = rsqrtf(half_warp_sum(v) * (1.f / 128.f) + eps);
    // LayerNorm in fp32, then the cast back to bf16 (round to nearest even).
    float y[8];
    uint32_t yb[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float a = (x[2 * i] - mean) * rstd * g[2 * i] + b[2 * i];
      const float c = (x[2 * i + 1] - mean) * rstd * g[2 * i + 1] + b[2 * i + 1];
      const __nv_bfloat162 p = __floats2bfloat162_rn(a, c);  // .x = a (low half)
      yb[i] = *reinterpret_cast<const uint32_t*>(&p);
      y[2 * i] = __low2float(p);
      y[2 * i + 1] = __high2float(p);
    }
    if (!fp8) {
      *reinterpret_cast<uint4*>(cache + slot * 256 + sub * 16) = make_uint4(yb[0], yb[1], yb[2], yb[3]);
      continue;
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(y[i]));
    amax = half_warp_max(amax);
    const int e = ue8m0_exponent(amax);
    *reinterpret_cast<uint2*>(cache + slot * 128 + sub * 8) = quantize8(y, e);
    if (sub == 0) cache_scale[slot] = ldexpf(1.f, e);
  }
}

int prologue_grid(int64_t rows) {
  const int64_t need = (rows + kRowsPerCta - 1) / kRowsPerCta;
  const int64_t cap = static_cast<int64_t>(device_sm_count() > 0 ? device_sm_count() : 1) * 16;
  return static_cast<int>(need < cap ? need : cap);
}

}  // namespace

cudaError_t launch_q_quant_fold(const void* q, const float* w, float weight_scale, int T, int H,
                                int Hp, void* q8, float* w_out, cudaStream_t s) {
  const int64_t rows = static_cast<int64_t>(T) * Hp;
  if (rows <= 0) return cudaSuccess;
  q_quant_fold_kernel<<<prologue_grid((rows + kQRows - 1) / kQRows), kProThreads, 0, s>>>(
      static_cast<const uint16_t*>(q), w, weight_scale, T, H, Hp, static_cast<uint8_t*>(q8), w_out);
  return cudaGetLastError();
}

cudaError_t launch_k_norm_insert(const void* k, const float* gamma, const float* beta, float eps,
                                 const int64_t* slots, int T, bool fp8, int64_t capacity,
                                 void* cache, float* cache_scale, uint32_t* err, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  k_norm_insert_kernel<<<prologue_grid(T), kProThreads, 0, s>>>(
      static_cast<const uint16_t*>(k), gamma, beta, eps, slots, T, fp8, capacity,
      static_cast<uint8_t*>(cache), cache_scale, err);
  return cudaGetLastError();
}

}  // namespace dsa
