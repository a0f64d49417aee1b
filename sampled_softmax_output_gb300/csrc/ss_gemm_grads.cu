// ss_gemm_grads.cu -- the two gradient GEMMs of the backward pass:
//   dH  = G . W_c          (M = T, N = D, K = C)
//   dWc = G^T . H          (M = C, N = D, K = T), scattered into dW[cand].
// G is read in place in both: K-major for dH, MN-major (transposed through the
// MMA's operand descriptor) for dW, so no transposed copy is ever made.
#include "ss_gemm.cuh"
#include "ss_internal.h"

namespace ss {

constexpr int kStagesGrad = 4;

cudaError_t launch_grad_h(const CUtensorMap& tG_kmaj, const CUtensorMap& tWc_mn, int T, int C,
                          int D, uint16_t* dH, int* status, int num_sms, cudaStream_t stream) {
  GemmShape shp{(T + BM - 1) / BM, (D + kBnGrad - 1) / kBnGrad, (C + BK - 1) / BK};
  EpiDh::Params ep{T, D, dH};
  return launch_gemm<kBnGrad, kStagesGrad, false, true, EpiDh>(tG_kmaj, tWc_mn, shp, ep, status,
                                                               num_sms, stream);
}

cudaError_t launch_grad_w(const CUtensorMap& tG_mn, const CUtensorMap& tH_mn, int T, int C, int D,
                          int V, int accumulate, const int32_t* cand, float* dW, int* status,
                          int num_sms, cudaStream_t stream) {
  GemmShape shp{(C + BM - 1) / BM, (D + kBnGrad - 1) / kBnGrad, (T + BK - 1) / BK};
  EpiDw::Params ep{C, D, V, accumulate, cand, dW, status};
  return launch_gemm<kBnGrad, kStagesGrad, true, true, EpiDw>(tG_mn, tH_mn, shp, ep, status,
                                                              num_sms, stream);
}

}  // namespace ss
