// dsa_score_prefill_mxfp4.cu -- the MXFP4 prefill scoring kernel's launch
// (H = 64, D = 128: 4 blocks of 32 elements per row, one 32-bit word of four
// E8M0 scale bytes per row).
#include "dsa_score_mx.cuh"

namespace dsa {

bool score_mx_supported(int H, int D) { return H == MxCfg::H && D == MxCfg::D; }

int score_mx_q_rows() { return MxCfg::N; }

cudaError_t launch_score_mx(const ScoreParams& p, const uint8_t* q_sf, const uint8_t* k_sf,
                            cudaStream_t s) {
  using C = MxCfg;
  cudaError_t e = cudaFuncSetAttribute(score_mx_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  const int groups = (p.R + C::TOK - 1) / C::TOK;
  if (groups <= 0) return cudaSuccess;
  const int sms = device_sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  score_mx_kernel<<<groups < sms ? groups : sms, C::THREADS, C::SMEM, s>>>(
      p, reinterpret_cast<const uint32_t*>(q_sf), reinterpret_cast<const uint32_t*>(k_sf));
  return cudaGetLastError();
}

}  // namespace dsa
