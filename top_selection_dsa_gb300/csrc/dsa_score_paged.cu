// dsa_score_paged.cu -- paged-decode instances of the scoring kernel.
//
// A CTA scores one chunk of one request's keys against that request's next_n
// query tokens (N = next_n * H columns, rounded up to 64/128/256); key tiles
// are gathered block by block through the block table with 3-D TMA boxes of
// [block_size rows x 128 bytes].
#include "dsa_score.cuh"

namespace dsa {

int score_paged_cols(int H, int next_n) {
  const int need = H * next_n;
  if (need <= 64) return 64;
  if (need <= 128) return 128;
  if (need <= 256) return 256;
  return 0;
}

namespace {

template <bool kFp8, int H>
cudaError_t by_cols(const ScoreParams& p, int N, int grid, cudaStream_t s) {
  switch (N) {
    case 64:
      return launch_score_instance<H, 64, 128, kFp8, true>(p, grid, s);
    case 128:
      return launch_score_instance<H, 128, 128, kFp8, true>(p, grid, s);
    case 256:
      return launch_score_instance<H, 256, 128, kFp8, true>(p, grid, s);
    default:
      return cudaErrorInvalidValue;
  }
}

template <bool kFp8>
cudaError_t by_heads(const ScoreParams& p, int H, int N, int grid, cudaStream_t s) {
  switch (H) {
    case 8:
      return by_cols<kFp8, 8>(p, N, grid, s);
    case 16:
      return by_cols<kFp8, 16>(p, N, grid, s);
    case 32:
      return by_cols<kFp8, 32>(p, N, grid, s);
    case 64:
      return by_cols<kFp8, 64>(p, N, grid, s);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace

bool score_paged_supported(bool fp8, int H, int D, int next_n) {
  (void)fp8;
  return D == 128 && (H == 8 || H == 16 || H == 32 || H == 64) && next_n >= 1 &&
         score_paged_cols(H, next_n) != 0;
}

cudaError_t launch_score_paged(const ScoreParams& p, bool fp8, int H, int D, cudaStream_t s) {
  (void)D;
  const int N = score_paged_cols(H, p.next_n);
  const int B = p.R / p.next_n;
  const int grid = B * p.chunks_per_req;
  return fp8 ? by_heads<true>(p, H, N, grid, s) : by_heads<false>(p, H, N, grid, s);
}

}  // namespace dsa
