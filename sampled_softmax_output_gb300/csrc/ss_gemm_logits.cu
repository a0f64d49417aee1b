// ss_gemm_logits.cu -- the two GEMMs over the T x C logit matrix S = H . W_c^T
// (K = D): the forward pass (log-sum-exp partials, target logit) and the
// backward recompute (softmax gradient G in bf16). Neither writes S itself.
#include "ss_gemm_logits.cuh"

namespace ss {


// One CTA per 128 x 256 logit tile. (CTA pairs on 256 x 256 tiles with a
// 6-deep ring measured slower or even on GB300 at every size tried: this GEMM's
// epilogue is light and K = D is short.)
cudaError_t launch_forward_logits(const CUtensorMap& tH, const CUtensorMap& tWc, int T, int C,
                                  int D, const int32_t* slot, float2* part, float* tgt,
                                  float cap, float tau, const Targets& tg, const float* amax,
                                  int* status, int num_sms, cudaStream_t stream) {
  if (amax) {  // the FP8 head (one target per token)
    const HeadCap h = head_cap(cap, tau);
    return cap > 0.f ? forward_logits<true, 1, true>(tH, tWc, T, C, D, slot, part, tgt, h, tg,
                                                     amax, status, num_sms, stream)
                     : forward_logits<false, 1, true>(tH, tWc, T, C, D, slot, part, tgt, h, tg,
                                                      amax, status, num_sms, stream);
  }
  if (tg.K > 1)
    return launch_forward_logits_mtp(tH, tWc, T, C, D, slot, part, tgt, cap, tau, tg, status,
                                     num_sms, stream);
  const HeadCap h = head_cap(cap, tau);
  return cap > 0.f ? forward_logits<true, 1>(tH, tWc, T, C, D, slot, part, tgt, h, tg, nullptr,
                                             status, num_sms, stream)
                   : forward_logits<false, 1>(tH, tWc, T, C, D, slot, part, tgt, h, tg, nullptr,
                                              status, num_sms, stream);
}

cudaError_t launch_softmax_grad(const CUtensorMap& tH, const CUtensorMap& tWc,
                                const CUtensorMap& tWc_half,
                                const CUtensorMap& tG_store, int T, int C, int D,
                                const int32_t* slot, const float* lse, float scale, float cap,
                                float tau, const Targets& tg, const float* amax, int* status,
                                int num_sms, cudaStream_t stream) {
  if (amax) {
    const HeadCap h = head_cap(cap, tau);
    return cap > 0.f ? softmax_grad<true, 1, true>(tH, tWc, tWc_half, tG_store, T, C, D, slot,
                                                   lse, scale, h, tg, amax, status, num_sms,
                                                   stream, false)
                     : softmax_grad<false, 1, true>(tH, tWc, tWc_half, tG_store, T, C, D, slot,
                                                    lse, scale, h, tg, amax, status, num_sms,
                                                    stream, false);
  }
  if (tg.K > 1)
    return launch_softmax_grad_mtp(tH, tWc, tWc_half, tG_store, T, C, D, slot, lse, scale, cap,
                                   tau, tg, status, num_sms, stream);
  const HeadCap h = head_cap(cap, tau);
  return cap > 0.f ? softmax_grad<true, 1>(tH, tWc, tWc_half, tG_store, T, C, D, slot, lse,
                                           scale, h, tg, nullptr, status, num_sms, stream,
                                           false)
                   : softmax_grad<false, 1>(tH, tWc, tWc_half, tG_store, T, C, D, slot, lse,
                                            scale, h, tg, nullptr, status, num_sms, stream,
                                            false);
}

// The stored-probability forward and its fallback, one target per token
// (forward_stored and softmax_grad_gated in ss_gemm_logits.cuh; several
// targets in ss_gemm_logits_mtp.cu).
cudaError_t launch_forward_stored(const CUtensorMap& tH, const CUtensorMap& tWc,
                                  const CUtensorMap& tWc_half, const CUtensorMap& tP, int T, int C,
                                  int D, const int32_t* slot, float2* part, float* tgt,
                                  float* ref, int* clear_word, const HeadCap& head,
                                  const Targets& tg, int* status, int num_sms,
                                  cudaStream_t stream) {
  if (tg.K > 1)
    return launch_forward_stored_mtp(tH, tWc, tWc_half, tP, T, C, D, slot, part, tgt, ref,
                                     clear_word, head, tg, status, num_sms, stream);
  return head.cap > 0.f
             ? forward_stored<true, 1>(tH, tWc, tWc_half, tP, T, C, D, slot, part, tgt, ref,
                                       clear_word, head, 1, status, num_sms, stream)
             : forward_stored<false, 1>(tH, tWc, tWc_half, tP, T, C, D, slot, part, tgt, ref,
                                        clear_word, head, 1, status, num_sms, stream);
}

cudaError_t launch_softmax_grad_gated(const CUtensorMap& tH, const CUtensorMap& tWc,
                                      const CUtensorMap& tWc_half, const CUtensorMap& tG_store,
                                      int T, int C, int D, const int32_t* slot, const float* lse,
                                      int* gate, const uint16_t* H, uint16_t* Hs, float* rowfac,
                                      const Targets& tg, float scale, int* status, int num_sms,
                                      cudaStream_t stream) {
  if (tg.K > 1)
    return launch_softmax_grad_gated_mtp(tH, tWc, tWc_half, tG_store, T, C, D, slot, lse, gate, H,
                                         Hs, rowfac, tg, scale, status, num_sms, stream);
  return softmax_grad_gated<1>(tH, tWc, tWc_half, tG_store, T, C, D, slot, lse, gate, H, Hs,
                               rowfac, tg, scale, status, num_sms, stream);
}

// FP8 gradients: G8 and G8^T in e5m2 from the e4m3 logits (one target)
template <bool CAP>
cudaError_t softmax_grad_fp8(const CUtensorMap& tH8, const CUtensorMap& tW8,
                             const CUtensorMap& tG8_store, const CUtensorMap& tG8t_store, int T,
                             int C, int D, const int32_t* slot, const float* lse, float cap,
                             float tau, int g8e, const float* amax, int* status, int num_sms,
                             cudaStream_t stream) {
  typename EpiG8T<CAP>::Params ep;
  ep.tmG = tG8_store;
  ep.tmGt = tG8t_store;
  ep.T = T;
  ep.C = C;
  ep.slot = slot;
  ep.lse = lse;
  ep.status = status;
  ep.amax = amax;
  ep.head = head_cap(cap, tau);
  ep.g8e = g8e;
  GemmShape shp{(T + BM - 1) / BM, (C + kBnLogits - 1) / kBnLogits, D / (2 * BK)};
  return launch_gemm<kBnLogits, kStagesGradF8, false, false, EpiG8T<CAP>, 8, true>(
      tH8, tW8, shp, ep, status, num_sms, stream);
}

cudaError_t launch_softmax_grad_fp8(const CUtensorMap& tH8, const CUtensorMap& tW8,
                                    const CUtensorMap& tG8_store, const CUtensorMap& tG8t_store,
                                    int T, int C, int D, const int32_t* slot, const float* lse,
                                    float cap, float tau, int g8e, const float* amax, int* status,
                                    int num_sms, cudaStream_t stream) {
  return cap > 0.f ? softmax_grad_fp8<true>(tH8, tW8, tG8_store, tG8t_store, T, C, D, slot, lse,
                                            cap, tau, g8e, amax, status, num_sms, stream)
                   : softmax_grad_fp8<false>(tH8, tW8, tG8_store, tG8t_store, T, C, D, slot, lse,
                                             cap, tau, g8e, amax, status, num_sms, stream);
}

}  // namespace ss
