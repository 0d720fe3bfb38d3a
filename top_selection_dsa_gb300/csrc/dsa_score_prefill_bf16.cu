// dsa_score_prefill_bf16.cu -- bf16 prefill instances of the scoring kernel
// (contiguous keys; D = 64 or 128; H a power of two up to 64; 256 MMA columns).
#include "dsa_score.cuh"

namespace dsa {

int score_tokens_per_group(int H) { return H >= 1 && H <= 256 ? 256 / H : 0; }

bool score_prefill_bf16_supported(int H, int D) {
  return (D == 64 || D == 128) && H >= 1 && H <= 64 && (H & (H - 1)) == 0;
}

cudaError_t launch_score_prefill_bf16(const ScoreParams& p, int H, int D, cudaStream_t s) {
  const int tok = score_tokens_per_group(H);
  const int grid = tok ? (p.R + tok - 1) / tok : 0;
#define DSA_CASE(HH)                                                              \
  case HH:                                                                        \
    return D == 128 ? launch_score_instance<HH, 256, 128, false, false>(p, grid, s) \
                    : launch_score_instance<HH, 256, 64, false, false>(p, grid, s);
  switch (H) {
    DSA_CASE(1)
    DSA_CASE(2)
    DSA_CASE(4)
    DSA_CASE(8)
    DSA_CASE(16)
    DSA_CASE(32)
    DSA_CASE(64)
    default:
      return cudaErrorInvalidValue;
  }
#undef DSA_CASE
}

}  // namespace dsa
