// ss_gemm_logits_mtp.cu -- the logit GEMMs for several targets per token
// (multi-token prediction over one set of logits): up to kMaxTargets target
// logits per row in the forward, the weighted one-hot terms in the softmax
// gradient. A translation unit of its own so that the instantiations compile
// in parallel with the single-target ones.
#include "ss_gemm_logits.cuh"

namespace ss {

cudaError_t launch_forward_logits_mtp(const CUtensorMap& tH, const CUtensorMap& tWc, int T, int C,
                                      int D, const int32_t* slot, float2* part, float* tgt,
                                      float cap, float tau, const Targets& tg, int* status,
                                      int num_sms, cudaStream_t stream) {
  const HeadCap h = head_cap(cap, tau);
  return cap > 0.f ? forward_logits<true, kMaxTargets>(tH, tWc, T, C, D, slot, part, tgt, h, tg,
                                                       nullptr, status, num_sms, stream)
                   : forward_logits<false, kMaxTargets>(tH, tWc, T, C, D, slot, part, tgt, h, tg,
                                                        nullptr, status, num_sms, stream);
}

cudaError_t launch_softmax_grad_mtp(const CUtensorMap& tH, const CUtensorMap& tWc,
                                    const CUtensorMap& tWc_half, const CUtensorMap& tG_store,
                                    int T, int C, int D, const int32_t* slot, const float* lse,
                                    float scale, float cap, float tau, const Targets& tg,
                                    int* status, int num_sms, cudaStream_t stream) {
  const HeadCap h = head_cap(cap, tau);
  return cap > 0.f ? softmax_grad<true, kMaxTargets>(tH, tWc, tWc_half, tG_store, T, C, D, slot,
                                                     lse, scale, h, tg, nullptr, status, num_sms,
                                                     stream, false)
                   : softmax_grad<false, kMaxTargets>(tH, tWc, tWc_half, tG_store, T, C, D, slot,
                                                      lse, scale, h, tg, nullptr, status,
                                                      num_sms, stream, false);
}

cudaError_t launch_forward_stored_mtp(const CUtensorMap& tH, const CUtensorMap& tWc,
                                      const CUtensorMap& tWc_half, const CUtensorMap& tP, int T,
                                      int C, int D, const int32_t* slot, float2* part, float* tgt,
                                      float* ref, int* clear_word, const HeadCap& head,
                                      const Targets& tg, int* status, int num_sms,
                                      cudaStream_t stream) {
  // two targets (the next two tokens) have their own instantiation: the
  // per-chunk target search and registers of eight cost the forward ~10%
  if (tg.K <= 2)
    return head.cap > 0.f
               ? forward_stored<true, 2>(tH, tWc, tWc_half, tP, T, C, D, slot, part, tgt, ref,
                                         clear_word, head, tg.K, status, num_sms, stream)
               : forward_stored<false, 2>(tH, tWc, tWc_half, tP, T, C, D, slot, part, tgt, ref,
                                          clear_word, head, tg.K, status, num_sms, stream);
  return head.cap > 0.f
             ? forward_stored<true, kMaxTargets>(tH, tWc, tWc_half, tP, T, C, D, slot, part, tgt,
                                                 ref, clear_word, head, tg.K, status, num_sms,
                                                 stream)
             : forward_stored<false, kMaxTargets>(tH, tWc, tWc_half, tP, T, C, D, slot, part, tgt,
                                                  ref, clear_word, head, tg.K, status, num_sms,
                                                  stream);
}

cudaError_t launch_softmax_grad_gated_mtp(const CUtensorMap& tH, const CUtensorMap& tWc,
                                          const CUtensorMap& tWc_half,
                                          const CUtensorMap& tG_store, int T, int C, int D,
                                          const int32_t* slot, const float* lse, int* gate,
                                          const uint16_t* H, uint16_t* Hs, float* rowfac,
                                          const Targets& tg, float scale, int* status,
                                          int num_sms, cudaStream_t stream) {
  return softmax_grad_gated<kMaxTargets>(tH, tWc, tWc_half, tG_store, T, C, D, slot, lse, gate,
                                         H, Hs, rowfac, tg, scale, status, num_sms, stream);
}

}  // namespace ss
