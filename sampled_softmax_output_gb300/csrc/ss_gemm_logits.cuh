// ss_gemm_logits.cuh -- launch templates of the two logit GEMMs (forward
// partials, softmax gradient) for a head (plain or capped) and a number of
// targets per token; instantiated by ss_gemm_logits.cu (one target) and
// ss_gemm_logits_mtp.cu (several).
#pragma once

#include <math.h>

#include "ss_gemm.cuh"
#include "ss_gemm2.cuh"
#include "ss_internal.h"

namespace ss {

constexpr int kStagesLogits = 4;
// the softmax-gradient GEMM on e4m3 operands: a 3-deep ring beside its 64 KB
// of store staging (measured on GB300: the e4m3 mainloop runs as fast with 3
// stages as with 4)
constexpr int kStagesGradF8 = 3;

// F8: e4m3 operands (tH, tWc are maps of the e4m3 copies), logits rescaled
// from amax in the epilogue. (CTA pairs measured 18% slower for the e4m3
// logit GEMMs on GB300.)
template <bool CAP, int KMAX, bool F8 = false>
cudaError_t forward_logits(const CUtensorMap& tH, const CUtensorMap& tWc, int T, int C, int D,
                           const int32_t* slot, float2* part, float* tgt, const HeadCap& head,
                           const Targets& tg, const float* amax, int* status, int num_sms,
                           cudaStream_t stream) {
  GemmShape shp{(T + BM - 1) / BM, (C + kBnLogits - 1) / kBnLogits, D / (F8 ? 2 * BK : BK)};
  typename EpiFwdT<CAP, KMAX, F8>::Params ep{T, C, slot, part, tgt, status, head, tg, amax};
  // the capped head's epilogue (three MUFU operations per logit), the FP8
  // head's (its mainloop is twice as fast) and that of several targets run
  // eight warps in two column groups, two partials per row per tile
  return launch_gemm<kBnLogits, kStagesLogits, false, false, EpiFwdT<CAP, KMAX, F8>,
                     (CAP || F8 || KMAX > 1) ? 8 : 4, F8>(tH, tWc, shp, ep, status, num_sms,
                                                          stream);
}

template <bool CAP, int KMAX, bool F8 = false>
cudaError_t softmax_grad(const CUtensorMap& tH, const CUtensorMap& tWc,
                         const CUtensorMap& tWc_half, const CUtensorMap& tG_store, int T, int C,
                         int D, const int32_t* slot, const float* lse, float scale,
                         const HeadCap& head, const Targets& tg, const float* amax, int* status,
                         int num_sms, cudaStream_t stream, bool late_wait, int* gate = nullptr,
                         const uint16_t* fix_H = nullptr, uint16_t* fix_Hs = nullptr,
                         float* fix_rowfac = nullptr, float fix_scale = 0.f) {
  typename EpiGT<CAP, KMAX, F8>::Params ep;
  ep.fix_H = fix_H;
  ep.fix_Hs = fix_Hs;
  ep.fix_rowfac = fix_rowfac;
  ep.fix_scale = fix_scale;
  ep.D = D;
  ep.tmG = tG_store;
  ep.T = T;
  ep.C = C;
  ep.slot = slot;
  ep.lse = lse;
  ep.scale = scale;
  float wsum = 0.f;
  for (int k = 0; k < tg.K; ++k) wsum += tg.w[k];
  const float sw = fabsf(scale) * wsum;  // the bulk term is scale * W * P
  ep.log2_scale = sw == 0.f ? -INFINITY : log2f(sw);
  ep.status = status;
  ep.head = head;
  ep.tg = tg;
  ep.amax = amax;
  // eight epilogue warps in two column groups, one staging buffer each; CTA
  // pairs (each SM stages half of the W_c tile, a 6-deep ring beside the G
  // staging) whenever every pair gets a tile. The epilogue hands its
  // accumulator back before its stores; before it did, pairs were 5% slower
  // at (T + C) * D * 2 = 41 MB (2-3% faster at 138 and 177 MB); with it,
  // measured on GB300 at T16384_C10240: the separate calls 0.640 -> 0.624 ms
  // per step, the capped head's step 0.670 -> 0.658 ms.
  const int n_tiles = (C + kBnLogits - 1) / kBnLogits;
  if constexpr (!F8) {  // the e4m3 operands are half the bytes: single CTAs throughout
    if (softmax_grad_on_pairs(T, C, num_sms)) {
      GemmShape shp{(T + 2 * BM - 1) / (2 * BM), n_tiles, D / BK};
      shp.gate = gate;
      return launch_gemm2<kBnLogits, 6, false, false, EpiGT<CAP, KMAX>, 8>(tH, tWc_half, shp, ep,
                                                                           status, num_sms,
                                                                           stream);
    }
  }
  GemmShape shp{(T + BM - 1) / BM, n_tiles, D / (F8 ? 2 * BK : BK), late_wait ? 1 : 0};
  shp.gate = gate;
  return launch_gemm<kBnLogits, F8 ? kStagesGradF8 : kStagesLogits, false, false,
                     EpiGT<CAP, KMAX, F8>, 8, F8>(tH, tWc, shp, ep, status, num_sms, stream);
}

}  // namespace ss
