// ss_internal.h -- declarations shared by the translation units of libss.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

namespace ss {

// Sets a kernel's dynamic shared-memory limit and the largest shared-memory
// carveout, once per kernel, device and process. Every kernel of the library
// asks for the same L1/shared split, so consecutive launches need no SM
// reconfiguration between them.
cudaError_t prepare_kernel(const void* kern, int dyn_smem_bytes);
template <typename... KArgs>
cudaError_t prepare_kernel(void (*kern)(KArgs...), int dyn_smem_bytes) {
  return prepare_kernel(reinterpret_cast<const void*>(kern), dyn_smem_bytes);
}

// Kernels launched by this host thread so far (for the launch trace).
extern thread_local int g_kernel_launches;

// Launch with programmatic stream serialization: the kernel may be scheduled
// while its predecessor in the stream drains, and waits for it in pdl_enter().
// Every kernel of the library is launched here.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  const cudaError_t e = prepare_kernel(kern, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t le = cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
  if (le == cudaSuccess) ++g_kernel_launches;
  return le;
}

// Tile widths of the GEMMs (output columns per tile).
constexpr int kBnLogits = 256;  // logit tiles: forward and softmax-gradient
constexpr int kBnGrad = 256;    // dH and dW tiles along D
// Softmax partials per row per logit tile: 1 for the plain single-target
// head (four epilogue warps); 2 (eight warps in two column groups) for the
// heads whose epilogue does more per logit than the MMAs can hide: the capped
// head (three MUFU operations per logit), the FP8 head (a mainloop twice as
// fast) and several targets per token. The workspace holds 2.
constexpr int kFwdGroupsMax = 2;
inline int fwd_groups(float cap, bool fp8 = false, int targets = 1) {
  return cap > 0.f || fp8 || targets > 1 ? 2 : 1;
}

struct GemmShape;

// The capped head z = cap / (1 + exp(-s / tau)): cap, log2(e) / tau and
// 1 / (cap tau) (dz/ds = z (cap - z) / (cap tau)); all zero for the plain head.
struct HeadCap {
  float cap, k1, icap_tau;
};
inline HeadCap head_cap(float cap, float tau) {
  const float log2e = 1.4426950408889634f;
  return cap > 0.f ? HeadCap{cap, log2e / tau, 1.f / (cap * tau)} : HeadCap{0.f, 0.f, 0.f};
}
// The stored-probability step takes the capped head up to this cap (exp(z -
// cap) must stay a normal number); above it the step recomputes the logits.
constexpr float kStoredCapMax = 64.f;

// Targets per token: K (at most kMaxTargets) target slots per row,
// slot[k * T + t], with weights w[k] (K = 1, w = 1: the single-target loss).
constexpr int kMaxTargets = 8;
struct Targets {
  int K;
  float w[kMaxTargets];
};

// Above this size, H [T, D] and W_c [C, D] together (bf16) no longer stay in
// L2 while a GEMM sweeps over them. The softmax-gradient GEMM then runs on
// CTA pairs (each SM loads half of every W_c tile) and the two gradient GEMMs
// in two phase-separated launches.
constexpr double kL2OperandBytes = 96.0 * (1 << 20);
inline bool operands_exceed_l2(int T, int C, int D) {
  return (static_cast<double>(T) + C) * D * 2.0 > kL2OperandBytes;
}
// The bf16 softmax-gradient GEMM runs on CTA pairs whenever every pair gets a
// 256 x 256 logit tile (single CTAs for small batches).
inline bool softmax_grad_on_pairs(int T, int C, int num_sms) {
  return static_cast<int64_t>((T + 255) / 256) * ((C + 255) / 256) >= num_sms / 2;
}

// ---- candidate build (ss_candidates.cu)
size_t build_candidates_smem_bytes(int64_t V);
// The candidate kernel's entry (for locating its node in a captured graph);
// its parameters are (targets, T, V, C, seed, cand, slot, hdr).
const void* build_candidates_kernel();
cudaError_t launch_build_candidates(const int32_t* targets, int T, int V, int C, uint64_t seed,
                                    int32_t* cand, int32_t* slot, int* hdr, cudaStream_t stream);

// ---- logit GEMMs (ss_gemm_logits.cu): A = H [T, D] (K-major), B = W_c [C, D] (K-major)
// tWc: box 64 x 256 (one 1-CTA tile); tWc_half: box 64 x 128 (a CTA's half of
// a pair's tile).
// cap > 0: the capped head z = cap / (1 + exp(-s / tau)) replaces the logits.
// tg: the targets per token (K = 1, w = 1 for the single-target loss).
cudaError_t launch_forward_logits(const CUtensorMap& tH, const CUtensorMap& tWc, int T, int C,
                                  int D, const int32_t* slot, float2* part, float* tgt,
                                  float cap, float tau, const Targets& tg, const float* amax,
                                  int* status, int num_sms, cudaStream_t stream);
// amax != nullptr: the FP8 head, tH / tWc map the e4m3 copies (box 128 x 128
// and 128 x 256 bytes), amax[2] their tensors' max |x|; plain logits, one
// target per token.
// G is written through tG_store: G [T, C] bf16, box 64 x 128, 128-byte swizzle.
cudaError_t launch_softmax_grad(const CUtensorMap& tH, const CUtensorMap& tWc,
                                const CUtensorMap& tWc_half,
                                const CUtensorMap& tG_store, int T, int C, int D,
                                const int32_t* slot, const float* lse, float scale, float cap,
                                float tau, const Targets& tg, const float* amax, int* status,
                                int num_sms, cudaStream_t stream);
// FP8 gradients (one target; cap > 0: the capped head): tH8 / tW8 as for
// amax above; G8 = e5m2(2^g8e (P - Y) dz/ds) [T, C] through tG8_store (box
// 64 x 128 bytes, 64-byte swizzle) and G8^T [C, T] through tG8t_store (box
// 128 x 64 bytes, 128-byte swizzle).
cudaError_t launch_softmax_grad_fp8(const CUtensorMap& tH8, const CUtensorMap& tW8,
                                    const CUtensorMap& tG8_store, const CUtensorMap& tG8t_store,
                                    int T, int C, int D, const int32_t* slot, const float* lse,
                                    float cap, float tau, int g8e, const float* amax, int* status,
                                    int num_sms, cudaStream_t stream);
// The forward that keeps the probabilities for the backward (bf16 head,
// plain or capped with cap <= kStoredCapMax, tg.K targets per token): Pt in
// bf16 through tP (as tG_store above) -- exp(S - r) with r[t] the row's
// largest logit over the first logit tile (stored in ref), or exp(z - cap)
// dz/ds with the cap --, the softmax partials (two per row per tile) and the
// target logits ([K, T]). Plain head: two launches, the first logit tile of
// every row block (which finds r and clears *clear_word), then the others;
// capped: one launch. tg.K > 1 runs the instantiations of
// ss_gemm_logits_mtp.cu.
cudaError_t launch_forward_stored(const CUtensorMap& tH, const CUtensorMap& tWc,
                                  const CUtensorMap& tWc_half, const CUtensorMap& tP, int T, int C,
                                  int D, const int32_t* slot, float2* part, float* tgt,
                                  float* ref, int* clear_word, const HeadCap& head,
                                  const Targets& tg, int* status, int num_sms,
                                  cudaStream_t stream);
cudaError_t launch_forward_stored_mtp(const CUtensorMap& tH, const CUtensorMap& tWc,
                                      const CUtensorMap& tWc_half, const CUtensorMap& tP, int T,
                                      int C, int D, const int32_t* slot, float2* part, float* tgt,
                                      float* ref, int* clear_word, const HeadCap& head,
                                      const Targets& tg, int* status, int num_sms,
                                      cudaStream_t stream);
// The stored-probability step's fallback (plain bf16 head): launch_softmax_grad
// with G = P - sum_k (w[k] / W) Y_k, W = sum_k w[k], that runs only if
// *gate != 0, and then also sets Hs = H and rowfac[t] = scale W for every row.
cudaError_t launch_softmax_grad_gated(const CUtensorMap& tH, const CUtensorMap& tWc,
                                      const CUtensorMap& tWc_half, const CUtensorMap& tG_store,
                                      int T, int C, int D, const int32_t* slot, const float* lse,
                                      int* gate, const uint16_t* H, uint16_t* Hs, float* rowfac,
                                      const Targets& tg, float scale, int* status, int num_sms,
                                      cudaStream_t stream);
cudaError_t launch_softmax_grad_gated_mtp(const CUtensorMap& tH, const CUtensorMap& tWc,
                                          const CUtensorMap& tWc_half,
                                          const CUtensorMap& tG_store, int T, int C, int D,
                                          const int32_t* slot, const float* lse, int* gate,
                                          const uint16_t* H, uint16_t* Hs, float* rowfac,
                                          const Targets& tg, float scale, int* status,
                                          int num_sms, cudaStream_t stream);
// the same GEMMs for K > 1 targets per token (ss_gemm_logits_mtp.cu)
cudaError_t launch_forward_logits_mtp(const CUtensorMap& tH, const CUtensorMap& tWc, int T, int C,
                                      int D, const int32_t* slot, float2* part, float* tgt,
                                      float cap, float tau, const Targets& tg, int* status,
                                      int num_sms, cudaStream_t stream);
cudaError_t launch_softmax_grad_mtp(const CUtensorMap& tH, const CUtensorMap& tWc,
                                    const CUtensorMap& tWc_half, const CUtensorMap& tG_store,
                                    int T, int C, int D, const int32_t* slot, const float* lse,
                                    float scale, float cap, float tau, const Targets& tg,
                                    int* status, int num_sms, cudaStream_t stream);

// ---- gradient GEMMs (ss_gemm_grads.cu)
// dH = G . W_c : A = G [T, C] (K-major), B = W_c [C, D] (MN-major)
// rowfac: null, or a factor per row of dH that the accumulator is multiplied by
cudaError_t launch_grad_h(const CUtensorMap& tG_kmaj, const CUtensorMap& tWc_mn, int T, int C,
                          int D, uint16_t* dH, int* status, int num_sms, cudaStream_t stream,
                          const float* rowfac = nullptr);
// dW[cand] (=|+=) G^T . H : A = G (MN-major), B = H [T, D] (MN-major)
// out_scale: null, or a factor the accumulator is multiplied by
cudaError_t launch_grad_w(const CUtensorMap& tG_mn, const CUtensorMap& tH_mn, int T, int C, int D,
                          int V, int accumulate, const int32_t* cand, float* dW, int* status,
                          int num_sms, cudaStream_t stream, const float* out_scale = nullptr);
// Both gradient GEMMs in one launch with a host-computed balanced schedule
// (falls back to the two launches above for very large problems).
cudaError_t launch_grads(const CUtensorMap& tG_kmaj, const CUtensorMap& tWc_mn,
                         const CUtensorMap& tG_mn, const CUtensorMap& tH_mn, int T, int C, int D,
                         int V, int accumulate, const int32_t* cand, uint16_t* dH, float* dW,
                         int* status, int num_sms, cudaStream_t stream,
                         const float* rowfac = nullptr, const float* out_scale = nullptr);

// FP8 gradients: dH = G8 . W8 and dW[cand] (=|+=) G8^T . H8 on e5m2 x e4m3,
// all operands K-major in boxes of 128 x 128 bytes: tG8 [T, C], tW8t [D, C],
// tG8t [C, T], tH8t [D, T]; the accumulators times scale * 2^-(15 + e) with e
// the other operand's e4m3 exponent (amax[0] = max |H|, amax[1] = max |W_c|)
// and g8e G8's power of two.
cudaError_t launch_grads_fp8(const CUtensorMap& tG8, const CUtensorMap& tW8t,
                             const CUtensorMap& tG8t, const CUtensorMap& tH8t, int T, int C, int D,
                             int V, int accumulate, const int32_t* cand, float scale, int g8e,
                             const float* amax, uint16_t* dH, float* dW, int* status, int num_sms,
                             cudaStream_t stream);

}  // namespace ss
