// ss_gemm_grads.cu -- the two gradient GEMMs of the backward pass:
//   dH  = G . W_c          (M = T, N = D, K = C)
//   dWc = G^T . H          (M = C, N = D, K = T), scattered into dW[cand].
// bf16: G is read in place in both, K-major for dH and MN-major (transposed
// through the MMA's operand descriptor) for dW, so no transposed copy is made.
// FP8 gradients: e5m2 G and e4m3 H, W_c, all K-major (G8 and G8^T as the
// softmax-gradient GEMM wrote them, H^T and W_c^T from the quantizer).
#include <algorithm>
#include <map>
#include <memory>
#include <mutex>
#include <queue>
#include <tuple>
#include <vector>

#include "ss_gemm.cuh"
#include "ss_gemm2.cuh"
#include "ss_internal.h"

namespace ss {


// the dW launch of the two-launch path does not wait for the dH launch
constexpr bool kDwNoWait = true;

cudaError_t launch_grad_h(const CUtensorMap& tG_kmaj, const CUtensorMap& tWc_mn, int T, int C,
                          int D, uint16_t* dH, int* status, int num_sms, cudaStream_t stream,
                          const float* rowfac) {
  GemmShape shp{(T + 2 * BM - 1) / (2 * BM), (D + kBnGrad - 1) / kBnGrad, (C + BK - 1) / BK};
  EpiDh::Params ep{T, D, dH, 0.f, nullptr, 0, rowfac};
  return launch_gemm2<kBnGrad, 6, false, true, EpiDh, 8>(tG_kmaj, tWc_mn, shp, ep, status, num_sms,
                                                         stream);
}

cudaError_t launch_grad_w(const CUtensorMap& tG_mn, const CUtensorMap& tH_mn, int T, int C, int D,
                          int V, int accumulate, const int32_t* cand, float* dW, int* status,
                          int num_sms, cudaStream_t stream, const float* out_scale) {
  // launched right after the dH GEMM, which it neither reads nor writes: it
  // need not wait for it (every kernel before dH has finished once dH's CTAs
  // have started), so its CTAs fill the SMs of dH's ragged last round
  GemmShape shp{(C + 2 * BM - 1) / (2 * BM), (D + kBnGrad - 1) / kBnGrad, (T + BK - 1) / BK,
                kDwNoWait ? 2 : 0};
  EpiDw::Params ep{C, D, V, accumulate, cand, dW, status, out_scale ? *out_scale : 1.f, nullptr,
                   0, out_scale ? 1 : 0};
  return launch_gemm2<kBnGrad, 6, true, true, EpiDw, 8>(tG_mn, tH_mn, shp, ep, status, num_sms,
                                                        stream);
}

// ------------------------------------------------- both GEMMs in one launch
//
// One persistent kernel runs the dW tiles and the dH tiles together. Which CTA
// pair runs which tiles, in which order, is decided on the host and passed in
// the kernel parameters: the per-pair mix of long (dW, K = T) and short (dH,
// K = C) tiles with the shortest makespan (exact for two tile lengths; at
// T = 16384, C = 10240 it balances to 97% where a greedy longest-first list
// schedule reaches 90%), tiles handed out in the order the pairs become free.
// Tiles handed out at the same moment start together, so the pairs keep
// marching through K side by side (the shared B operand stays in L2, and the
// three tiles of a row block read their common A rows at the same time).

namespace {

constexpr int kSchedMaxCtas = 256;
constexpr int kSchedMaxUnits = 14080;

struct GradSched {
  uint16_t offs[kSchedMaxCtas + 1];  // CTA c runs units[offs[c] .. offs[c+1])
  uint16_t units[kSchedMaxUnits];    // [0, n_dw): dW tiles, then dH tiles
};

template <bool F8G>
struct GradBoth {
  int n_dw, n_nt, kb_dw, kb_dh;  // n_dw counts 256-row dW tiles (x column tiles)
  int n_units;  // used when F8G: with rr, pair p runs units p, p + pairs, ... < n_units
  int rr;
  typename EpiDhT<F8G>::Params dh;
  typename EpiDwT<F8G>::Params dw;
  int* status;
};

constexpr int kStagesPairGrad = 6;
constexpr int kGradEpiWarps = 8;
using LG2 = Gemm2Smem<kBnGrad, kStagesPairGrad, 0>;

// Both gradient GEMMs on CTA pairs (see ss_gemm2.cuh for the pair protocol):
// pair p runs the 256-row tiles sch.units[sch.offs[p] .. sch.offs[p + 1]).
// Operand maps: dH tiles read A from tmAh and B from tmBh, dW tiles A from
// tmAw and B from tmBw. bf16: G (K-major), W_c (MN-major), G (MN-major), H
// (MN-major). F8G: G8, W8^T, G8^T, H8^T, all K-major, 128 of K per k-block.
template <bool F8G>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(64 + 32 * kGradEpiWarps, 1)
    k_grads(const __grid_constant__ CUtensorMap tmAh, const __grid_constant__ CUtensorMap tmBh,
            const __grid_constant__ CUtensorMap tmAw, const __grid_constant__ CUtensorMap tmBw,
            const __grid_constant__ GradBoth<F8G> p, const __grid_constant__ GradSched sch) {
  pdl_enter();
  constexpr int BN = kBnGrad;
  constexpr int STAGES = kStagesPairGrad;
  constexpr int NCG = kGradEpiWarps / 4;
  constexpr int KB = F8G ? 2 * BK : BK;  // elements of K per k-block
  using L = LG2;
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_go;
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  GemmCtrl* ctrl = reinterpret_cast<GemmCtrl*>(smem + L::CTRL_OFFSET);
  const uint32_t tiles = smem_u32(smem);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();
  const int pair = blockIdx.x >> 1;
  int* status = p.status;
  // this pair's units: i = u_begin, u_begin + u_step, ... < u_end; unit(i)
  const bool rr = F8G && p.rr != 0;
  const int u_begin = rr ? pair : sch.offs[pair];
  const int u_end = rr ? p.n_units : sch.offs[pair + 1];
  const int u_step = rr ? static_cast<int>(gridDim.x >> 1) : 1;
  auto unit = [&](int i) { return rr ? i : static_cast<int>(sch.units[i]); };

  if (threadIdx.x == 0) s_go = (read_status(status) == 0);
  cluster_sync_all();
  if (threadIdx.x == 0) s_go = s_go && ld_shared_cluster_u32(mapa_shared(smem_u32(&s_go), rank ^ 1u));
  cluster_sync_all();
  if (!s_go) return;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&ctrl->full[s], 1);
      mbar_init(&ctrl->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&ctrl->tfull[b], 1);
      mbar_init(&ctrl->tempty[b], 2 * kGradEpiWarps);
    }
    mbar_init(&ctrl->drain, 1);
    ctrl->abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_map(&tmAh);
    tma_prefetch_map(&tmBh);
    tma_prefetch_map(&tmAw);
    tma_prefetch_map(&tmBw);
  }
  if (warp == 1) {
    tmem_alloc_pair(&ctrl->tmem_base, 2 * BN);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = ctrl->tmem_base;
  volatile int* abort_flag = &ctrl->abort_flag;

  if (warp == 0) {
    // ------------------------------------------------ producer (both CTAs)
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0, issued = 0, issued_ph = 0;
      bool ok = true;
      for (int i = u_begin; ok && i < u_end; i += u_step) {
        const int u = unit(i);
        const bool is_dw = u < p.n_dw;
        const int v = is_dw ? u : u - p.n_dw;
        const int mt = v / p.n_nt, nt = v % p.n_nt;
        const int m0 = mt * 2 * BM + static_cast<int>(rank) * BM;
        const int n0 = nt * BN + static_cast<int>(rank) * (BN / 2);
        const int kbs = is_dw ? p.kb_dw : p.kb_dh;
        for (int kb = 0; kb < kbs; ++kb) {
          if (!mbar_wait(&ctrl->empty[s], ph ^ 1u, abort_flag, status)) {
            ok = false;
            break;
          }
          const uint32_t fb_local = smem_u32(&ctrl->full[s]);
          if (rank == 0) mbar_arrive_expect_tx(&ctrl->full[s], 2 * L::STAGE_BYTES);
          const uint32_t fb = rank == 0 ? fb_local : mapa_shared(fb_local, 0);
          const uint32_t a_dst = tiles + s * L::STAGE_BYTES;
          const uint32_t b_dst = a_dst + L::A_BYTES;
          // B (H or W_c) is re-read by every row tile: keep it in L2
          const uint64_t keep = l2_evict_last();
          if constexpr (F8G) {  // one 128 x 128-byte box of A and of B, K-major
            const CUtensorMap* ma = is_dw ? &tmAw : &tmAh;
            const CUtensorMap* mb = is_dw ? &tmBw : &tmBh;
            tma_load_2d_pair_hint(a_dst, ma, fb, kb * KB, m0, l2_evict_first());
            tma_load_2d_pair_hint(b_dst, mb, fb, kb * KB, n0, keep);
          } else if (is_dw) {  // A = G columns (MN-major), B = H (MN-major); K = tokens
            const uint64_t first = l2_evict_first();  // G streams through
            tma_load_2d_pair_hint(a_dst, &tmAw, fb, m0, kb * BK, first);
            tma_load_2d_pair_hint(a_dst + 8192, &tmAw, fb, m0 + 64, kb * BK, first);
            tma_load_2d_pair_hint(b_dst, &tmBw, fb, n0, kb * BK, keep);
            tma_load_2d_pair_hint(b_dst + 8192, &tmBw, fb, n0 + 64, kb * BK, keep);
          } else {      // A = G rows (K-major), B = W_c (MN-major); K = candidates
            tma_load_2d_pair_hint(a_dst, &tmAh, fb, kb * BK, m0, l2_evict_first());
            tma_load_2d_pair_hint(b_dst, &tmBh, fb, n0, kb * BK, keep);
            tma_load_2d_pair_hint(b_dst + 8192, &tmBh, fb, n0 + 64, kb * BK, keep);
          }
          issued |= 1u << s;
          issued_ph = (issued_ph & ~(1u << s)) | (ph << s);
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      if (rank == 0) {
        for (int j = 0; j < STAGES; ++j)
          if ((issued >> j) & 1u) mbar_drain(&ctrl->full[j], (issued_ph >> j) & 1u, status);
      } else if (!ok) {
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 200000ull) {
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer (leader)
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc_dw = idesc_bf16_f32(2 * BM, BN, true, true);
      constexpr uint32_t idesc_dh = idesc_bf16_f32(2 * BM, BN, false, true);
      constexpr uint32_t idesc_f8 = idesc_f8_f32(2 * BM, BN, kFmtE5M2, kFmtE4M3);
      int s = 0, b = 0;
      uint32_t ph = 0, aph = 0;
      bool ok = true;
      for (int i = u_begin; ok && i < u_end; i += u_step) {
        const bool is_dw = unit(i) < p.n_dw;
        const int kbs = is_dw ? p.kb_dw : p.kb_dh;
        if (!mbar_wait(&ctrl->tempty[b], aph ^ 1u, abort_flag, status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * BN);
        for (int kb = 0; kb < kbs; ++kb) {
          if (!mbar_wait(&ctrl->full[s], ph, abort_flag, status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = tiles + s * L::STAGE_BYTES;
          const uint32_t b_addr = a_addr + L::A_BYTES;
#pragma unroll
          for (int k = 0; k < BK / UMMA_K; ++k) {
            if constexpr (F8G) {  // K = 32 e5m2 / e4m3 per instruction: 32 bytes along K
              const uint64_t ad = sdesc_sw128(a_addr + k * 32, 16, 1024);
              const uint64_t bd = sdesc_sw128(b_addr + k * 32, 16, 1024);
              mma_f8_pair(d_tmem, ad, bd, idesc_f8, (kb | k) != 0 ? 1u : 0u);
            } else {
              const uint64_t ad = is_dw ? sdesc_sw128(a_addr + k * 2048, 8192, 1024)
                                        : sdesc_sw128(a_addr + k * 32, 16, 1024);
              const uint64_t bd = sdesc_sw128(b_addr + k * 2048, 8192, 1024);
              mma_bf16_pair(d_tmem, ad, bd, is_dw ? idesc_dw : idesc_dh,
                            (kb | k) != 0 ? 1u : 0u);
            }
          }
          mma_commit_pair(&ctrl->empty[s], 0x3);
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit_pair(&ctrl->tfull[b], 0x3);
        if (++b == 2) {
          b = 0;
          aph ^= 1u;
        }
      }
      mma_commit_pair(&ctrl->drain, 0x1);
      mbar_drain(&ctrl->drain, 0, status);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;
    const int cg = (warp - 2) / 4;
    const int row = q * 32 + lane;
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    // one EpiState per kind of tile: each holds that epilogue's per-launch scale
    EpiState es{0u, 0, 0u, 0.f}, es_h{0u, 0, 0u, 0.f};
    EpiDwT<F8G>::begin(p.dw, es);
    EpiDhT<F8G>::begin(p.dh, es_h);
    int b = 0;
    uint32_t aph = 0;
    for (int i = u_begin; i < u_end; i += u_step) {
      const bool ok = mbar_wait(&ctrl->tfull[b], aph, abort_flag, status);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const int u = unit(i);
      const bool is_dw = u < p.n_dw;
      const int v = is_dw ? u : u - p.n_dw;
      const int mt = (v / p.n_nt) * 2 + static_cast<int>(rank), nt = v % p.n_nt;
      const uint32_t taddr = lane_addr + static_cast<uint32_t>(b * BN);
      if (is_dw) EpiDwT<F8G>::template apply<BN, NCG>(p.dw, mt, nt, row, taddr, es, cg);
      else EpiDhT<F8G>::template apply<BN, NCG>(p.dh, mt, nt, row, taddr, es_h, cg);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        const uint32_t te = smem_u32(&ctrl->tempty[b]);
        if (rank == 0) mbar_arrive(&ctrl->tempty[b]);
        else mbar_arrive_cluster(mapa_shared(te, 0));
      }
      if (++b == 2) {
        b = 0;
        aph ^= 1u;
      }
    }
  }
  __syncthreads();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, 2 * BN);
  }
}

// Greedy longest-first list schedule of the tiles over `ctas` CTAs; cached by
// problem shape. Returns nullptr if it does not fit the kernel parameters.
// Makespan (in k-blocks) of the greedy longest-first list schedule; also the
// per-pair unit counts it gives.
long long lpt_counts(int n_dw, int kb_dw, int n_dh, int kb_dh, int pairs, std::vector<int>& na,
                     std::vector<int>& nb) {
  using Slot = std::pair<long long, int>;  // (time the pair becomes free, pair)
  std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> free_at;
  for (int c = 0; c < pairs; ++c) free_at.push({0, c});
  auto place = [&](int len, std::vector<int>& cnt) {
    const Slot sl = free_at.top();
    free_at.pop();
    ++cnt[sl.second];
    free_at.push({sl.first + len, sl.second});
  };
  const bool dw_first = kb_dw >= kb_dh;
  for (int pass = 0; pass < 2; ++pass) {
    if ((pass == 0) == dw_first)
      for (int u = 0; u < n_dw; ++u) place(kb_dw, na);
    else
      for (int u = 0; u < n_dh; ++u) place(kb_dh, nb);
  }
  long long ms = 0;
  while (!free_at.empty()) {
    ms = std::max(ms, free_at.top().first);
    free_at.pop();
  }
  return ms;
}

// Per-pair counts (na[p] dW units, nb[p] dH units) of a shortest schedule:
// with only two unit lengths A = kb_dw and B = kb_dh, makespan M is feasible
// iff some choice of a_p dW units per pair covers n_dw while the dH room left,
// sum of floor((M - a_p A) / B), covers n_dh; a dynamic program over (pairs
// used, dW units covered) keeps the largest dH room. M runs over the values
// a A + b B between the averaged lower bound and the greedy makespan.
void plan_counts(int n_dw, int kb_dw, int n_dh, int kb_dh, int pairs, std::vector<int>& na,
                 std::vector<int>& nb) {
  const long long A = kb_dw, B = kb_dh;
  const long long ub = lpt_counts(n_dw, kb_dw, n_dh, kb_dh, pairs, na, nb);
  const long long total = n_dw * A + n_dh * B;
  long long lb = (total + pairs - 1) / pairs;
  if (n_dw > 0) lb = std::max(lb, A);
  if (n_dh > 0) lb = std::max(lb, B);
  std::vector<long long> cand;
  for (long long a = 0; a * A <= ub && a <= n_dw; ++a)
    for (long long b = 0; a * A + b * B <= ub && b <= n_dh; ++b)
      if (a * A + b * B >= lb) cand.push_back(a * A + b * B);
  std::sort(cand.begin(), cand.end());
  cand.erase(std::unique(cand.begin(), cand.end()), cand.end());
  const int D = n_dw + 1;
  std::vector<int> f(static_cast<size_t>(pairs + 1) * D), from(f.size()), pick(f.size());
  for (long long M : cand) {
    if (M >= ub) return;  // the greedy counts are as short
    const int amax = static_cast<int>(std::min<long long>(n_dw, M / A));
    auto room = [&](int a) { return static_cast<int>(std::min<long long>(n_dh, (M - a * A) / B)); };
    std::fill(f.begin(), f.end(), -1);
    f[0] = 0;
    for (int k = 0; k < pairs; ++k)
      for (int d = 0; d < D; ++d) {
        const int cur = f[static_cast<size_t>(k) * D + d];
        if (cur < 0) continue;
        for (int a = 0; a <= amax; ++a) {
          const int nd = std::min(n_dw, d + a);
          const int val = std::min(n_dh, cur + room(a));
          const size_t at = static_cast<size_t>(k + 1) * D + nd;
          if (val > f[at]) {
            f[at] = val;
            from[at] = d;
            pick[at] = a;
          }
        }
      }
    if (f[static_cast<size_t>(pairs) * D + n_dw] < n_dh) continue;
    // walk back: pair k - 1 takes pick[k][d] dW units
    int d = n_dw, left_dw = n_dw, left_dh = n_dh;
    for (int k = pairs; k > 0; --k) {
      const size_t at = static_cast<size_t>(k) * D + d;
      const int a = std::min(pick[at], left_dw);
      na[k - 1] = a;
      left_dw -= a;
      d = from[at];
    }
    for (int k = 0; k < pairs; ++k) {
      nb[k] = std::min(room(na[k]), left_dh);
      left_dh -= nb[k];
    }
    return;
  }
}

// The schedule of both gradient GEMMs over `pairs` CTA pairs: per-pair counts
// from plan_counts; each pair runs its dW tiles, then its dH tiles, and the
// tiles are handed out in the order the pairs become free, so the tiles
// running at the same time have neighbouring indices (they share operand rows
// in L2).
std::shared_ptr<const GradSched> grad_schedule(int n_dw, int kb_dw, int n_dh, int kb_dh, int ctas) {
  static std::mutex mu;
  static std::map<std::tuple<int, int, int, int, int>, std::shared_ptr<const GradSched>> cache;
  const auto key = std::make_tuple(n_dw, kb_dw, n_dh, kb_dh, ctas);
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  const long long n = static_cast<long long>(n_dw) + n_dh;
  if (n > kSchedMaxUnits || ctas > kSchedMaxCtas || ctas < 1) return nullptr;
  std::vector<int> na(ctas, 0), nb(ctas, 0);
  plan_counts(n_dw, kb_dw, n_dh, kb_dh, ctas, na, nb);
  std::vector<std::vector<uint16_t>> lists(ctas);
  using Slot = std::pair<long long, int>;
  std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> free_at;
  for (int c = 0; c < ctas; ++c) free_at.push({0, c});
  int next_dw = 0, next_dh = 0;
  while (!free_at.empty()) {
    const Slot sl = free_at.top();
    free_at.pop();
    const int c = sl.second;
    const int done = static_cast<int>(lists[c].size());
    if (done < na[c]) {
      lists[c].push_back(static_cast<uint16_t>(next_dw++));
      free_at.push({sl.first + kb_dw, c});
    } else if (done < na[c] + nb[c]) {
      lists[c].push_back(static_cast<uint16_t>(n_dw + next_dh++));
      free_at.push({sl.first + kb_dh, c});
    }
  }
  if (next_dw != n_dw || next_dh != n_dh) return nullptr;  // cannot happen: counts add up
  auto sch = std::make_shared<GradSched>();
  int at = 0;
  for (int c = 0; c < ctas; ++c) {
    sch->offs[c] = static_cast<uint16_t>(at);
    for (uint16_t u : lists[c]) sch->units[at++] = u;
  }
  sch->offs[ctas] = static_cast<uint16_t>(at);
  if (cache.size() > 64) cache.clear();
  cache[key] = sch;
  return sch;
}

}  // namespace

cudaError_t launch_grads(const CUtensorMap& tG_kmaj, const CUtensorMap& tWc_mn,
                         const CUtensorMap& tG_mn, const CUtensorMap& tH_mn, int T, int C, int D,
                         int V, int accumulate, const int32_t* cand, uint16_t* dH, float* dW,
                         int* status, int num_sms, cudaStream_t stream, const float* rowfac,
                         const float* out_scale) {
  GradBoth<false> p;
  p.n_nt = (D + kBnGrad - 1) / kBnGrad;
  p.n_dw = (C + 2 * BM - 1) / (2 * BM) * p.n_nt;
  const int n_dh = (T + 2 * BM - 1) / (2 * BM) * p.n_nt;
  p.kb_dw = (T + BK - 1) / BK;
  p.kb_dh = (C + BK - 1) / BK;
  p.n_units = 0;
  p.rr = 0;
  p.dh = EpiDh::Params{T, D, dH, 0.f, nullptr, 0, rowfac};
  p.dw = EpiDw::Params{C, D, V, accumulate, cand, dW, status, out_scale ? *out_scale : 1.f,
                       nullptr, 0, out_scale ? 1 : 0};
  p.status = status;
  const int pairs = std::min(num_sms / 2, kSchedMaxCtas);
  // Running dW and dH tiles side by side pays when their B operands (H and
  // W_c) fit in L2 together; beyond that they evict each other and two
  // phase-separated launches are faster (measured on GB300: merged is 5-17%
  // faster at (T + C) * D * 2 = 41-72 MB, 10% slower at 138-177 MB).
  auto sch = !operands_exceed_l2(T, C, D)
                 ? grad_schedule(p.n_dw, p.kb_dw, n_dh, p.kb_dh, pairs)
                 : std::shared_ptr<const GradSched>();
  if (!sch) {  // two phase-separated round-robin launches
    cudaError_t e = launch_grad_h(tG_kmaj, tWc_mn, T, C, D, dH, status, num_sms, stream, rowfac);
    if (e != cudaSuccess) return e;
    return launch_grad_w(tG_mn, tH_mn, T, C, D, V, accumulate, cand, dW, status, num_sms, stream,
                         out_scale);
  }
  return launch_pdl(k_grads<false>, dim3(2 * pairs), dim3(64 + 32 * kGradEpiWarps), LG2::TOTAL,
                    stream, tG_kmaj, tWc_mn, tG_mn, tH_mn, p, *sch);
}

cudaError_t launch_grads_fp8(const CUtensorMap& tG8, const CUtensorMap& tW8t,
                             const CUtensorMap& tG8t, const CUtensorMap& tH8t, int T, int C, int D,
                             int V, int accumulate, const int32_t* cand, float scale, int g8e,
                             const float* amax, uint16_t* dH, float* dW, int* status, int num_sms,
                             cudaStream_t stream) {
  constexpr int KB = 2 * BK;
  GradBoth<true> p;
  p.n_nt = (D + kBnGrad - 1) / kBnGrad;
  p.n_dw = (C + 2 * BM - 1) / (2 * BM) * p.n_nt;
  const int n_dh = (T + 2 * BM - 1) / (2 * BM) * p.n_nt;
  p.kb_dw = (T + KB - 1) / KB;
  p.kb_dh = (C + KB - 1) / KB;
  p.n_units = p.n_dw + n_dh;
  p.dh = EpiDhT<true>::Params{T, D, dH, scale, amax + 1, g8e, nullptr};
  p.dw = EpiDwT<true>::Params{C, D, V, accumulate, cand, dW, status, scale, amax, g8e, 0};
  p.status = status;
  const int pairs = std::min(num_sms / 2, kSchedMaxCtas);
  // the balanced schedule where it fits the kernel parameters, else every
  // pair walks the units round-robin (dW tiles first)
  auto sch = grad_schedule(p.n_dw, p.kb_dw, n_dh, p.kb_dh, pairs);
  static const GradSched kNone = {};
  p.rr = sch ? 0 : 1;
  return launch_pdl(k_grads<true>, dim3(2 * pairs), dim3(64 + 32 * kGradEpiWarps), LG2::TOTAL,
                    stream, tG8, tW8t, tG8t, tH8t, p, sch ? *sch : kNone);
}

}  // namespace ss
