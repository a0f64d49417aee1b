// ss_gemm_logits.cu -- the two GEMMs over the T x C logit matrix S = H . W_c^T
// (K = D): the forward pass (log-sum-exp partials, target logit) and the
// backward recompute (softmax gradient G in bf16). Neither writes S itself.
#include "ss_gemm.cuh"
#include "ss_gemm2.cuh"
#include "ss_internal.h"

namespace ss {

constexpr int kStagesLogits = 4;

namespace {

template <bool CAP>
cudaError_t forward_logits(const CUtensorMap& tH, const CUtensorMap& tWc, int T, int C, int D,
                           const int32_t* slot, float2* part, float* tgt, const HeadCap& head,
                           int* status, int num_sms, cudaStream_t stream) {
  GemmShape shp{(T + BM - 1) / BM, (C + kBnLogits - 1) / kBnLogits, D / BK};
  typename EpiFwdT<CAP>::Params ep{T, C, slot, part, tgt, status, head};
  // the capped head's epilogue (three MUFU operations per logit) runs eight
  // warps in two column groups, two partials per row per tile
  return launch_gemm<kBnLogits, kStagesLogits, false, false, EpiFwdT<CAP>, CAP ? 8 : 4>(
      tH, tWc, shp, ep, status, num_sms, stream);
}

template <bool CAP>
cudaError_t softmax_grad(const CUtensorMap& tH, const CUtensorMap& tWc,
                         const CUtensorMap& tWc_half, const CUtensorMap& tG_store, int T, int C,
                         int D, const int32_t* slot, const float* lse, float scale,
                         const HeadCap& head, int* status, int num_sms, cudaStream_t stream) {
  typename EpiGT<CAP>::Params ep;
  ep.tmG = tG_store;
  ep.T = T;
  ep.C = C;
  ep.slot = slot;
  ep.lse = lse;
  ep.scale = scale;
  ep.log2_scale = scale == 0.f ? -INFINITY : log2f(fabsf(scale));
  ep.status = status;
  ep.head = head;
  // eight epilogue warps in two column groups, one staging buffer each; CTA
  // pairs (each SM stages half of the W_c tile, a 6-deep ring beside the G
  // staging) once the operands exceed L2 (measured on GB300: the pair is 5%
  // slower at (T + C) * D * 2 = 41 MB, 2-3% faster at 138 and 177 MB)
  const int n_tiles = (C + kBnLogits - 1) / kBnLogits;
  if (operands_exceed_l2(T, C, D)) {
    GemmShape shp{(T + 2 * BM - 1) / (2 * BM), n_tiles, D / BK};
    return launch_gemm2<kBnLogits, 6, false, false, EpiGT<CAP>, 8>(tH, tWc_half, shp, ep,
                                                                   status, num_sms, stream);
  }
  GemmShape shp{(T + BM - 1) / BM, n_tiles, D / BK};
  return launch_gemm<kBnLogits, kStagesLogits, false, false, EpiGT<CAP>, 8>(tH, tWc, shp, ep,
                                                                            status, num_sms,
                                                                            stream);
}

HeadCap head_cap(float cap, float tau) {
  const float log2e = 1.4426950408889634f;
  return cap > 0.f ? HeadCap{cap, log2e / tau, 1.f / (cap * tau)} : HeadCap{0.f, 0.f, 0.f};
}

}  // namespace

// One CTA per 128 x 256 logit tile. (CTA pairs on 256 x 256 tiles with a
// 6-deep ring measured slower or even on GB300 at every size tried: this GEMM's
// epilogue is light and K = D is short.)
cudaError_t launch_forward_logits(const CUtensorMap& tH, const CUtensorMap& tWc, int T, int C,
                                  int D, const int32_t* slot, float2* part, float* tgt,
                                  float cap, float tau, int* status, int num_sms,
                                  cudaStream_t stream) {
  const HeadCap h = head_cap(cap, tau);
  return cap > 0.f ? forward_logits<true>(tH, tWc, T, C, D, slot, part, tgt, h, status, num_sms,
                                          stream)
                   : forward_logits<false>(tH, tWc, T, C, D, slot, part, tgt, h, status, num_sms,
                                           stream);
}

cudaError_t launch_softmax_grad(const CUtensorMap& tH, const CUtensorMap& tWc,
                                const CUtensorMap& tWc_half,
                                const CUtensorMap& tG_store, int T, int C, int D,
                                const int32_t* slot, const float* lse, float scale, float cap,
                                float tau, int* status, int num_sms, cudaStream_t stream) {
  const HeadCap h = head_cap(cap, tau);
  return cap > 0.f ? softmax_grad<true>(tH, tWc, tWc_half, tG_store, T, C, D, slot, lse, scale,
                                        h, status, num_sms, stream)
                   : softmax_grad<false>(tH, tWc, tWc_half, tG_store, T, C, D, slot, lse, scale,
                                         h, status, num_sms, stream);
}

}  // namespace ss
