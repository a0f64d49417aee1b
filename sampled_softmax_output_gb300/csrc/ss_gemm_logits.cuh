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

// The stored-probability forward: on CTA pairs whenever every pair gets a
// tile (each SM stages its 128 rows of H and half of every W_c tile, two
// thirds of the operand intake per flop of one CTA per 128 x 256 tile;
// measured on GB300: 0.507 against 0.521 ms per step at T16384_C10240, 1.399
// against 1.447 ms at T32768_C14336, 10.20 against 10.45 ms at T65536_C50304),
// single CTAs for small batches. Units walk groups of row tiles column by
// column (kFwdGroupRows rows per group), so W_c is read from DRAM once per
// group rather than once per row tile while the Pt stream passes through L2
// (10.20 ms against 10.58 ms row by row, on pairs at T65536_C50304).
constexpr int kFwdGroupRows = 8192;
// ring stages and staging buffers per column group: CTA pairs, single CTAs.
// The epilogue hands its accumulator back before its stores, so it has slack
// and one staging buffer per group is enough; the 32 KB this frees buys a
// sixth ring stage (measured on GB300 at T65536_C50304: time x SM clock per
// step 1.8% lower than five stages with two buffers).
constexpr int kFwdPairStages = 6, kFwdPairBufs = 1;
constexpr int kFwdStages = 4, kFwdBufs = 1;

// Plain head: the first logit tile of every row block finds r and clears
// *clear_word; the launch over the other tiles starts its mainloop at once
// (H and W_c are older than the first launch) and its epilogue waits for r.
// CAP: the reference is cap, known before any tile: one launch over every
// tile. K targets per token (K <= KMAX).
template <bool CAP, int KMAX>
cudaError_t forward_stored(const CUtensorMap& tH, const CUtensorMap& tWc,
                           const CUtensorMap& tWc_half, const CUtensorMap& tP, int T, int C,
                           int D, const int32_t* slot, float2* part, float* tgt, float* ref,
                           int* clear_word, const HeadCap& head, int K, int* status, int num_sms,
                           cudaStream_t stream) {
  const int n_tiles = (C + kBnLogits - 1) / kBnLogits;
  const int pair_m = (T + 2 * BM - 1) / (2 * BM);
  if constexpr (CAP) {
    if (pair_m * n_tiles >= num_sms / 2) {
      using Epi = EpiFwdP<false, kFwdPairBufs, true, KMAX>;
      typename Epi::Params ep{tP, T, C, slot, part, tgt, nullptr, nullptr, status, head, K};
      GemmShape shp{pair_m, n_tiles, D / BK, 0, 0, nullptr, kFwdGroupRows / (2 * BM)};
      return launch_gemm2<kBnLogits, kFwdPairStages, false, false, Epi, 8>(
          tH, tWc_half, shp, ep, status, num_sms, stream);
    }
    using Epi = EpiFwdP<false, kFwdBufs, true, KMAX>;
    typename Epi::Params ep{tP, T, C, slot, part, tgt, nullptr, nullptr, status, head, K};
    GemmShape shp{(T + BM - 1) / BM, n_tiles, D / BK, 0, 0, nullptr, kFwdGroupRows / BM};
    return launch_gemm<kBnLogits, kFwdStages, false, false, Epi, 8>(tH, tWc, shp, ep, status,
                                                                   num_sms, stream);
  } else {
    if (pair_m * (n_tiles - 1) >= num_sms / 2) {
      using Pre = EpiFwdP<true, kFwdPairBufs, false, KMAX>;
      using Rest = EpiFwdP<false, kFwdPairBufs, false, KMAX>;
      typename Pre::Params pre{tP, T, C, slot, part, tgt, ref, clear_word, status, head, K};
      typename Rest::Params rest{tP, T, C, slot, part, tgt, ref, nullptr, status, head, K};
      GemmShape first{pair_m, 1, D / BK};
      cudaError_t e = launch_gemm2<kBnLogits, kFwdPairStages, false, false, Pre, 8>(
          tH, tWc_half, first, pre, status, num_sms, stream);
      if (e != cudaSuccess || n_tiles == 1) return e;
      GemmShape others{pair_m, n_tiles, D / BK, 1, 1, nullptr, kFwdGroupRows / (2 * BM)};
      return launch_gemm2<kBnLogits, kFwdPairStages, false, false, Rest, 8>(
          tH, tWc_half, others, rest, status, num_sms, stream);
    }
    using Pre = EpiFwdP<true, kFwdBufs, false, KMAX>;
    using Rest = EpiFwdP<false, kFwdBufs, false, KMAX>;
    typename Pre::Params pre{tP, T, C, slot, part, tgt, ref, clear_word, status, head, K};
    typename Rest::Params rest{tP, T, C, slot, part, tgt, ref, nullptr, status, head, K};
    const int m_tiles = (T + BM - 1) / BM;
    GemmShape first{m_tiles, 1, D / BK};
    cudaError_t e = launch_gemm<kBnLogits, kFwdStages, false, false, Pre, 8>(
        tH, tWc, first, pre, status, num_sms, stream);
    if (e != cudaSuccess || n_tiles == 1) return e;
    GemmShape others{m_tiles, n_tiles, D / BK, 1, 1, nullptr, kFwdGroupRows / BM};
    return launch_gemm<kBnLogits, kFwdStages, false, false, Rest, 8>(tH, tWc, others, rest,
                                                                      status, num_sms, stream);
  }
}

// The stored-probability step's fallback: G = P - sum_k (w[k] / W) Y_k (W =
// sum_k w[k]) from the logits, run only if *gate != 0, which then also resets
// Hs = H and rowfac = scale W, the factors the stored path's gradient GEMMs
// apply (rowfac per row of dH, scale W to dW_c).
template <int KMAX>
cudaError_t softmax_grad_gated(const CUtensorMap& tH, const CUtensorMap& tWc,
                               const CUtensorMap& tWc_half, const CUtensorMap& tG_store, int T,
                               int C, int D, const int32_t* slot, const float* lse, int* gate,
                               const uint16_t* H, uint16_t* Hs, float* rowfac, const Targets& tg,
                               float scale, int* status, int num_sms, cudaStream_t stream) {
  float wsum = 0.f;
  for (int k = 0; k < tg.K; ++k) wsum += tg.w[k];
  return softmax_grad<false, KMAX>(tH, tWc, tWc_half, tG_store, T, C, D, slot, lse, 1.f / wsum,
                                   head_cap(0.f, 1.f), tg, nullptr, status, num_sms, stream,
                                   false, gate, H, Hs, rowfac, scale * wsum);
}

}  // namespace ss
