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
                                int num_sms, cudaStream_t stream, bool late_wait) {
  if (amax) {
    const HeadCap h = head_cap(cap, tau);
    return cap > 0.f ? softmax_grad<true, 1, true>(tH, tWc, tWc_half, tG_store, T, C, D, slot,
                                                   lse, scale, h, tg, amax, status, num_sms,
                                                   stream, late_wait)
                     : softmax_grad<false, 1, true>(tH, tWc, tWc_half, tG_store, T, C, D, slot,
                                                    lse, scale, h, tg, amax, status, num_sms,
                                                    stream, late_wait);
  }
  if (tg.K > 1)
    return launch_softmax_grad_mtp(tH, tWc, tWc_half, tG_store, T, C, D, slot, lse, scale, cap,
                                   tau, tg, status, num_sms, stream, late_wait);
  const HeadCap h = head_cap(cap, tau);
  return cap > 0.f ? softmax_grad<true, 1>(tH, tWc, tWc_half, tG_store, T, C, D, slot, lse,
                                           scale, h, tg, nullptr, status, num_sms, stream,
                                           late_wait)
                   : softmax_grad<false, 1>(tH, tWc, tWc_half, tG_store, T, C, D, slot, lse,
                                            scale, h, tg, nullptr, status, num_sms, stream,
                                            late_wait);
}

// The stored-probability forward: on CTA pairs whenever every pair gets a
// tile (each SM stages its 128 rows of H and half of every W_c tile, two
// thirds of the operand intake per flop of one CTA per 128 x 256 tile;
// measured on GB300: 0.507 against 0.521 ms per step at T16384_C10240, 1.399
// against 1.447 ms at T32768_C14336, 10.20 against 10.45 ms at T65536_C50304),
// single CTAs for small batches. Units walk groups of row tiles column by column (kFwdGroupRows rows per
// group), so W_c is read from DRAM once per group rather than once per row
// tile while the Pt stream passes through L2 (10.20 ms against 10.58 ms
// row by row, on pairs at T65536_C50304).
constexpr int kFwdGroupRows = 8192;
// ring stages and staging buffers per column group: CTA pairs, single CTAs.
// The epilogue hands its accumulator back before its stores, so it has slack
// and one staging buffer per group is enough; the 32 KB this frees buys a
// sixth ring stage (measured on GB300 at T65536_C50304: time x SM clock per
// step 1.8% lower than five stages with two buffers).
constexpr int kFwdPairStages = 6, kFwdPairBufs = 1;
constexpr int kFwdStages = 4, kFwdBufs = 1;

// The first logit tile of every row block finds r and clears *clear_word;
// the launch over the other tiles starts its mainloop at once (H and W_c are
// older than the first launch) and its epilogue waits for r.
cudaError_t launch_forward_stored(const CUtensorMap& tH, const CUtensorMap& tWc,
                                  const CUtensorMap& tWc_half, const CUtensorMap& tP, int T, int C,
                                  int D, const int32_t* slot, float2* part, float* tgt,
                                  float* ref, int* clear_word, int* status, int num_sms,
                                  cudaStream_t stream) {
  const int n_tiles = (C + kBnLogits - 1) / kBnLogits;
  const int pair_units = (T + 2 * BM - 1) / (2 * BM) * (n_tiles - 1);
  if (pair_units >= num_sms / 2) {
    using Pre = EpiFwdP<true, kFwdPairBufs>;
    using Rest = EpiFwdP<false, kFwdPairBufs>;
    typename Pre::Params pre{tP, T, C, slot, part, tgt, ref, clear_word, status};
    typename Rest::Params rest{tP, T, C, slot, part, tgt, ref, nullptr, status};
    const int m_tiles = (T + 2 * BM - 1) / (2 * BM);
    GemmShape first{m_tiles, 1, D / BK};
    cudaError_t e = launch_gemm2<kBnLogits, kFwdPairStages, false, false, Pre, 8>(
        tH, tWc_half, first, pre, status, num_sms, stream);
    if (e != cudaSuccess || n_tiles == 1) return e;
    GemmShape others{m_tiles, n_tiles, D / BK, 1, 1, nullptr, kFwdGroupRows / (2 * BM)};
    return launch_gemm2<kBnLogits, kFwdPairStages, false, false, Rest, 8>(
        tH, tWc_half, others, rest, status, num_sms, stream);
  }
  using Pre = EpiFwdP<true, kFwdBufs>;
  using Rest = EpiFwdP<false, kFwdBufs>;
  typename Pre::Params pre{tP, T, C, slot, part, tgt, ref, clear_word, status};
  typename Rest::Params rest{tP, T, C, slot, part, tgt, ref, nullptr, status};
  const int m_tiles = (T + BM - 1) / BM;
  GemmShape first{m_tiles, 1, D / BK};
  cudaError_t e = launch_gemm<kBnLogits, kFwdStages, false, false, Pre, 8>(
      tH, tWc, first, pre, status, num_sms, stream);
  if (e != cudaSuccess || n_tiles == 1) return e;
  GemmShape others{m_tiles, n_tiles, D / BK, 1, 1, nullptr, kFwdGroupRows / BM};
  return launch_gemm<kBnLogits, kFwdStages, false, false, Rest, 8>(tH, tWc, others, rest, status,
                                                                    num_sms, stream);
}

// The capped head's stored forward: one launch over every logit tile (the
// reference is cap, known before any tile), on CTA pairs whenever every pair
// gets a tile.
cudaError_t launch_forward_stored_cap(const CUtensorMap& tH, const CUtensorMap& tWc,
                                      const CUtensorMap& tWc_half, const CUtensorMap& tP, int T,
                                      int C, int D, const int32_t* slot, float2* part, float* tgt,
                                      const HeadCap& head, int* status, int num_sms,
                                      cudaStream_t stream) {
  const int n_tiles = (C + kBnLogits - 1) / kBnLogits;
  const int pair_m = (T + 2 * BM - 1) / (2 * BM);
  if (pair_m * n_tiles >= num_sms / 2) {
    using Epi = EpiFwdP<false, kFwdPairBufs, true>;
    typename Epi::Params ep{tP, T, C, slot, part, tgt, nullptr, nullptr, status, head};
    GemmShape shp{pair_m, n_tiles, D / BK, 0, 0, nullptr, kFwdGroupRows / (2 * BM)};
    return launch_gemm2<kBnLogits, kFwdPairStages, false, false, Epi, 8>(tH, tWc_half, shp, ep,
                                                                         status, num_sms, stream);
  }
  using Epi = EpiFwdP<false, kFwdBufs, true>;
  typename Epi::Params ep{tP, T, C, slot, part, tgt, nullptr, nullptr, status, head};
  GemmShape shp{(T + BM - 1) / BM, n_tiles, D / BK, 0, 0, nullptr, kFwdGroupRows / BM};
  return launch_gemm<kBnLogits, kFwdStages, false, false, Epi, 8>(tH, tWc, shp, ep, status,
                                                                 num_sms, stream);
}

cudaError_t launch_softmax_grad_gated(const CUtensorMap& tH, const CUtensorMap& tWc,
                                      const CUtensorMap& tWc_half, const CUtensorMap& tG_store,
                                      int T, int C, int D, const int32_t* slot, const float* lse,
                                      int* gate, const uint16_t* H, uint16_t* Hs, float* rowfac,
                                      float scale, int* status, int num_sms,
                                      cudaStream_t stream) {
  const Targets one = {1, {1.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f}};
  return softmax_grad<false, 1>(tH, tWc, tWc_half, tG_store, T, C, D, slot, lse, 1.f,
                                head_cap(0.f, 1.f), one, nullptr, status, num_sms, stream, false,
                                gate, H, Hs, rowfac, scale);
}

// FP8 gradients: G8 and G8^T in e5m2 from the e4m3 logits (one target)
template <bool CAP>
cudaError_t softmax_grad_fp8(const CUtensorMap& tH8, const CUtensorMap& tW8,
                             const CUtensorMap& tG8_store, const CUtensorMap& tG8t_store, int T,
                             int C, int D, const int32_t* slot, const float* lse, float cap,
                             float tau, int g8e, const float* amax, int* status, int num_sms,
                             cudaStream_t stream, bool late_wait) {
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
  GemmShape shp{(T + BM - 1) / BM, (C + kBnLogits - 1) / kBnLogits, D / (2 * BK),
                late_wait ? 1 : 0};
  return launch_gemm<kBnLogits, kStagesGradF8, false, false, EpiG8T<CAP>, 8, true>(
      tH8, tW8, shp, ep, status, num_sms, stream);
}

cudaError_t launch_softmax_grad_fp8(const CUtensorMap& tH8, const CUtensorMap& tW8,
                                    const CUtensorMap& tG8_store, const CUtensorMap& tG8t_store,
                                    int T, int C, int D, const int32_t* slot, const float* lse,
                                    float cap, float tau, int g8e, const float* amax, int* status,
                                    int num_sms, cudaStream_t stream, bool late_wait) {
  return cap > 0.f ? softmax_grad_fp8<true>(tH8, tW8, tG8_store, tG8t_store, T, C, D, slot, lse,
                                            cap, tau, g8e, amax, status, num_sms, stream,
                                            late_wait)
                   : softmax_grad_fp8<false>(tH8, tW8, tG8_store, tG8t_store, T, C, D, slot, lse,
                                             cap, tau, g8e, amax, status, num_sms, stream,
                                             late_wait);
}

}  // namespace ss
