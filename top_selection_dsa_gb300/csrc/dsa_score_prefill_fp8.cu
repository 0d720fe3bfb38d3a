// dsa_score_prefill_fp8.cu -- e4m3 prefill instances of the scoring kernel
// (kind::f8f6f4 MMA; D = 128, i.e. one UE8M0 scale per key row; the key
// scale is applied after the head sum, which is exact for powers of two).
#include "dsa_score.cuh"

namespace dsa {

bool score_prefill_fp8_supported(int H, int D) {
  return D == 128 && H >= 1 && H <= 64 && (H & (H - 1)) == 0;
}

cudaError_t launch_score_prefill_fp8(const ScoreParams& p, int H, int D, cudaStream_t s) {
  (void)D;
  const int tok = score_tokens_per_group(H);
  const int grid = tok ? (p.R + tok - 1) / tok : 0;
#define DSA_CASE(HH) \
  case HH:           \
    return launch_score_instance<HH, 256, 128, true, false>(p, grid, s);
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
