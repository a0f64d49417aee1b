// ss_gemm2.cuh -- the GEMM core of ss_gemm.cuh on CTA pairs: one 2-SM
// tcgen05.mma.cta_group::2 per 256 x BN x 16 step.
//
// A cluster of two CTAs (rank 0 "leader", rank 1 "peer") owns one 256-row
// output tile. Each CTA holds its own 128 rows of A and one half (BN / 2 rows
// or columns) of B in shared memory; the tensor cores of the pair exchange the
// B halves, so each SM loads and stores 32 KB per 64-deep k-block instead of
// 48 KB. That leaves room for a 6-deep ring, which hides more memory latency.
// Each CTA's TMEM holds the fp32 accumulator of its own 128 rows (all BN
// columns), so the epilogues of ss_gemm.cuh run unchanged in both CTAs.
//
// Synchronisation (all waits bounded, as in ss_gemm.cuh):
//   full[s]   leader only: armed by the leader's producer for the bytes of
//             both CTAs; both producers' TMA loads complete on it.
//   empty[s]  both CTAs: the leader's commit arrives on both (multicast).
//   tfull[b]  both CTAs: the leader's commit arrives on both (multicast).
//   tempty[b] leader only: one arrival per epilogue warp of both CTAs.
// TMEM is allocated and freed collectively by both CTAs; a cluster barrier
// before the free keeps the leader's MMAs from outliving the peer's TMEM.
#pragma once

#include "ss_gemm.cuh"

namespace ss {

template <int BN, int STAGES, int EPI_BYTES>
struct Gemm2Smem {
  static constexpr int A_BYTES = BM * BK * 2;          // this CTA's 128 rows of A
  static constexpr int B_BYTES = (BN / 2) * BK * 2;    // this CTA's half of B
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int TILES_BYTES = STAGES * STAGE_BYTES;
  static constexpr int EPI_OFFSET = TILES_BYTES;
  static constexpr int CTRL_OFFSET = TILES_BYTES + EPI_BYTES;
  static constexpr int CTRL_BYTES = 256;
  static constexpr int TOTAL = CTRL_OFFSET + CTRL_BYTES + 1024;
  static_assert(TOTAL <= 232448, "shared memory per CTA");
};

// Units are (256-row tile, BN-column tile) pairs numbered m-major; the pair
// (cluster) index walks them round-robin. shp.m_tiles counts 256-row tiles.
// EPI_WARPS epilogue warps (4 or 8): with 8, two warps share each 32-lane
// quarter of TMEM and split the tile's columns between them.
template <int BN, int STAGES, bool A_MN, bool B_MN, class Epi, int EPI_WARPS>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(64 + 32 * EPI_WARPS, 1)
    k_gemm2(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
            GemmShape shp, const __grid_constant__ typename Epi::Params ep, int* status) {
  if (shp.late_wait) pdl_launch_dependents();
  else pdl_enter();
  static_assert(BN % 128 == 0 && BN >= 128 && BN <= 256, "BN");
  static_assert(STAGES >= 2 && STAGES <= 8, "STAGES");
  static_assert(EPI_WARPS == 4 || EPI_WARPS == 8, "EPI_WARPS");
  constexpr int NCG = EPI_WARPS / 4;  // column groups per row block
  using L = Gemm2Smem<BN, STAGES, Epi::kStageBytes>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_go;

  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  GemmCtrl* ctrl = reinterpret_cast<GemmCtrl*>(smem + L::CTRL_OFFSET);
  const uint32_t tiles = smem_u32(smem);
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;

  // Both CTAs must take the same decision: each reads the status word, then
  // each combines its own answer with the peer's after a cluster barrier.
  if (threadIdx.x == 0)
    s_go = read_status(status) == 0 && (shp.gate == nullptr || read_status(shp.gate) != 0);
  cluster_sync_all();
  if (threadIdx.x == 0) s_go = s_go && ld_shared_cluster_u32(mapa_shared(smem_u32(&s_go), rank ^ 1u));
  cluster_sync_all();  // the peer has read this CTA's s_go before it changes
  if (!s_go) return;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&ctrl->full[s], 1);
      mbar_init(&ctrl->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&ctrl->tfull[b], 1);
      mbar_init(&ctrl->tempty[b], 2 * EPI_WARPS);
    }
    mbar_init(&ctrl->drain, 1);
    ctrl->abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_map(&tmA);
    tma_prefetch_map(&tmB);
  }
  if (warp == 1) {
    tmem_alloc_pair(&ctrl->tmem_base, 2 * BN);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();  // barriers of both CTAs initialised, TMEM allocated
  tc_fence_after();
  const uint32_t tmem_base = ctrl->tmem_base;
  volatile int* abort_flag = &ctrl->abort_flag;
  const int num_units = shp.m_tiles * (shp.n_tiles - shp.n_begin);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0, issued = 0, issued_ph = 0;
      bool ok = true;
      for (int u = pair; ok && u < num_units; u += npairs) {
        int mt, nt;
        unit_tile(shp, u, mt, nt);
        const int m0 = mt * 2 * BM + static_cast<int>(rank) * BM;   // this CTA's A rows
        const int n0 = nt * BN + static_cast<int>(rank) * (BN / 2);  // this CTA's half of B
        for (int kb = 0; kb < shp.k_blocks; ++kb) {
          if (!mbar_wait(&ctrl->empty[s], ph ^ 1u, abort_flag, status)) {
            ok = false;
            break;
          }
          const uint32_t fb_local = smem_u32(&ctrl->full[s]);
          if (rank == 0) mbar_arrive_expect_tx(&ctrl->full[s], 2 * L::STAGE_BYTES);
          const uint32_t fb = rank == 0 ? fb_local : mapa_shared(fb_local, 0);
          const uint32_t a_dst = tiles + s * L::STAGE_BYTES;
          const uint32_t b_dst = a_dst + L::A_BYTES;
          if (A_MN) {
#pragma unroll
            for (int i = 0; i < BM / 64; ++i)
              tma_load_2d_pair(a_dst + i * 8192, &tmA, fb, m0 + 64 * i, kb * BK);
          } else {
            tma_load_2d_pair(a_dst, &tmA, fb, kb * BK, m0);
          }
          // B is re-read by every row tile: keep it in L2
          const uint64_t keep = l2_evict_last();
          if (B_MN) {
#pragma unroll
            for (int i = 0; i < BN / 128; ++i)
              tma_load_2d_pair_hint(b_dst + i * 8192, &tmB, fb, n0 + 64 * i, kb * BK, keep);
          } else {
            tma_load_2d_pair_hint(b_dst, &tmB, fb, kb * BK, n0, keep);
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
        // every copy of both CTAs that the leader armed must land
        for (int i = 0; i < STAGES; ++i)
          if ((issued >> i) & 1u) mbar_drain(&ctrl->full[i], (issued_ph >> i) & 1u, status);
      } else if (!ok) {
        // aborted: the peer cannot observe the leader's barriers; give its
        // copies in flight a bounded moment to land before shared memory goes
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 200000ull) {
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer (leader)
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(2 * BM, BN, A_MN, B_MN);
      int s = 0, b = 0;
      uint32_t ph = 0, aph = 0;
      bool ok = true;
      for (int u = pair; ok && u < num_units; u += npairs) {
        if (!mbar_wait(&ctrl->tempty[b], aph ^ 1u, abort_flag, status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * BN);
        for (int kb = 0; kb < shp.k_blocks; ++kb) {
          if (!mbar_wait(&ctrl->full[s], ph, abort_flag, status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = tiles + s * L::STAGE_BYTES;
          const uint32_t b_addr = a_addr + L::A_BYTES;
#pragma unroll
          for (int k = 0; k < BK / UMMA_K; ++k) {
            const uint64_t ad = A_MN ? sdesc_sw128(a_addr + k * 2048, 8192, 1024)
                                     : sdesc_sw128(a_addr + k * 32, 16, 1024);
            const uint64_t bd = B_MN ? sdesc_sw128(b_addr + k * 2048, 8192, 1024)
                                     : sdesc_sw128(b_addr + k * 32, 16, 1024);
            mma_bf16_pair(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
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
    const int q = warp & 3;          // TMEM lane quarter this warp may access
    const int cg = (warp - 2) / 4;   // column group
    const int row = q * 32 + lane;
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    EpiState es{tiles + L::EPI_OFFSET, static_cast<int>(threadIdx.x) - 64, 0u, 0.f};
    if (shp.late_wait == 1) pdl_wait();
    Epi::begin(ep, es);
    int b = 0;
    uint32_t aph = 0;
    for (int u = pair; u < num_units; u += npairs) {
      const bool ok = mbar_wait(&ctrl->tfull[b], aph, abort_flag, status);
      bool go = __all_sync(0xffffffffu, ok);
      if constexpr (Epi::kStageBytes > 0) {
        if (lane == 0) ctrl->vote[(u / npairs) & 1][warp - 2] = go ? 1 : 0;
        named_bar_sync(2, 32 * EPI_WARPS);
        const int* v = ctrl->vote[(u / npairs) & 1];
        int all = 1;
#pragma unroll
        for (int i = 0; i < EPI_WARPS; ++i) all &= v[i];
        go = all != 0;
      }
      if (!go) break;
      tc_fence_after();
      int mt, nt;
      unit_tile(shp, u, mt, nt);
      auto release = [&] {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          const uint32_t te = smem_u32(&ctrl->tempty[b]);
          if (rank == 0) mbar_arrive(&ctrl->tempty[b]);
          else mbar_arrive_cluster(mapa_shared(te, 0));
        }
      };
      const int mrow = mt * 2 + static_cast<int>(rank);
      const uint32_t acc = lane_addr + static_cast<uint32_t>(b * BN);
      if constexpr (EpiSelfRelease<Epi>::value) {
        Epi::template apply<BN, NCG>(ep, mrow, nt, row, acc, es, cg, release);
      } else {
        Epi::template apply<BN, NCG>(ep, mrow, nt, row, acc, es, cg);
        release();
      }
      if (++b == 2) {
        b = 0;
        aph ^= 1u;
      }
    }
    Epi::finish(ep, es);
    if (shp.late_wait == 2) pdl_wait();  // the kernel before this one has finished
  }
  __syncthreads();
  cluster_sync_all();  // the leader's MMAs are drained before either CTA frees TMEM
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, 2 * BN);
  }
}

// Host-side launcher: grid = 2 x min(units, SMs / 2), one CTA per SM.
template <int BN, int STAGES, bool A_MN, bool B_MN, class Epi, int EPI_WARPS>
cudaError_t launch_gemm2(const CUtensorMap& tA, const CUtensorMap& tB, GemmShape shp,
                         const typename Epi::Params& ep, int* status, int num_sms,
                         cudaStream_t stream) {
  auto kern = k_gemm2<BN, STAGES, A_MN, B_MN, Epi, EPI_WARPS>;
  constexpr int smem = Gemm2Smem<BN, STAGES, Epi::kStageBytes>::TOTAL;
  const int units = shp.m_tiles * (shp.n_tiles - shp.n_begin);
  if (units <= 0) return cudaSuccess;
  if (shp.gate != nullptr && shp.late_wait) return cudaErrorInvalidValue;  // the gate needs the wait
  const int pairs = units < num_sms / 2 ? units : num_sms / 2;
  return launch_pdl(kern, dim3(2 * pairs), dim3(64 + 32 * EPI_WARPS), smem, stream, tA, tB, shp, ep,
                    status);
}

}  // namespace ss
