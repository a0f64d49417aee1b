// ss_gemm_grads.cu -- the two gradient GEMMs of the backward pass in one
// persistent, stream-K scheduled kernel:
//   dH   = G . W_c          (M = T, N = D, K = C)        "dH tiles"
//   dW_c = G^T . H          (M = C, N = D, K = T)        "dW tiles", scattered
//                                                        into dW[cand[j]]
// G is read in place in both: K-major for dH, MN-major (transposed through the
// MMA's operand descriptor) for dW, so no transposed copy is ever made.
//
// Scheduling. The CTAs form n_nt groups, one per 256-wide column slice of D.
// Every group walks the same tile list -- all dW tiles, then all dH tiles, by
// row tile -- for its own slice, so the CTAs that share a row tile of G read it
// at the same moment (L2 reuse). Inside a group the list is cut into equal
// contiguous ranges of k-blocks, one per CTA (stream-K), which removes the
// idle tail a whole-tile schedule leaves on 152 SMs. A tile cut by a range
// boundary is finished by the CTA that holds its first k-block ("owner"): the
// other CTAs write their fp32 partial accumulators to the workspace and raise
// a flag; the owner waits for those flags (bounded), adds the partials in CTA
// order (deterministic) and runs the epilogue. A non-owner piece is always the
// first piece of its CTA, which never waits on anything, so the waits cannot
// form a cycle; the launch is cooperative, so every CTA is resident.
#include "ss_gemm.cuh"
#include "ss_internal.h"

namespace ss {

namespace {

constexpr int kStagesGrad = 4;
constexpr int BNG = kBnGrad;  // 256
using LG = GemmSmem<BNG, kStagesGrad, 0>;

struct GradParams {
  int T, C, D, V, accumulate;
  int n_nt;          // column slices of D (BNG wide) = CTA groups
  int n_cm, n_tm;    // row tiles of dW (C / 128) and of dH (T / 128)
  int kb_dw, kb_dh;  // k-blocks per tile: T / 64 and C / 64 (rounded up)
  int group_ctas;    // CTAs per group
  const int32_t* cand;
  uint16_t* dH;
  float* dW;
  float* partial;    // [grid][128][BNG] fp32
  int* flags;        // [grid], zero at launch
  int* status;
};

struct Seg {
  int tile;  // index in the group's list: [0, n_cm) dW, then [n_cm, n_cm + n_tm) dH
  int kb0, kb1, len;
};

__device__ __forceinline__ long long tile_start(const GradParams& p, int u) {
  return u < p.n_cm ? static_cast<long long>(u) * p.kb_dw
                    : static_cast<long long>(p.n_cm) * p.kb_dw +
                          static_cast<long long>(u - p.n_cm) * p.kb_dh;
}

__device__ __forceinline__ long long group_total(const GradParams& p) {
  return static_cast<long long>(p.n_cm) * p.kb_dw + static_cast<long long>(p.n_tm) * p.kb_dh;
}

// First k-block of CTA i's range within its group.
__device__ __forceinline__ long long range_begin(const GradParams& p, int i) {
  return group_total(p) * i / p.group_ctas;
}

struct SegIter {
  long long it, end;
  __device__ SegIter(const GradParams& p, int i) : it(range_begin(p, i)), end(range_begin(p, i + 1)) {}
  __device__ bool next(const GradParams& p, Seg& s) {
    if (it >= end) return false;
    const long long dw_total = static_cast<long long>(p.n_cm) * p.kb_dw;
    int u;
    if (it < dw_total) u = static_cast<int>(it / p.kb_dw);
    else u = p.n_cm + static_cast<int>((it - dw_total) / p.kb_dh);
    const long long us = tile_start(p, u);
    const int len = u < p.n_cm ? p.kb_dw : p.kb_dh;
    const long long ue = us + len;
    const long long stop = ue < end ? ue : end;
    s.tile = u;
    s.kb0 = static_cast<int>(it - us);
    s.kb1 = static_cast<int>(stop - us);
    s.len = len;
    it = stop;
    return true;
  }
};

__device__ __forceinline__ bool flag_wait(const int* flag, volatile int* abort_flag, int* status) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t k = 0;; ++k) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
    if (v != 0) return true;
    if ((k & 31u) == 31u) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        set_status(status, SS_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void flag_release(int* flag) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(flag), "r"(1) : "memory");
}

// Epilogue of one segment for this thread's row. The hand-off between CTAs is
// per warp: warp q of a non-owner writes rows [32q, 32q + 32) of its partial
// and raises flags[cta * 4 + q]; warp q of the owner waits for that flag of
// each other piece, so no barrier spans warps. Returns false if a wait gave up.
__device__ bool grad_epilogue(const GradParams& p, const Seg& s, int nt, int cta, int gi, int q,
                              int lane, int row, uint32_t taddr, volatile int* abort_flag) {
  const bool is_dw = s.tile < p.n_cm;
  const int mt = is_dw ? s.tile : s.tile - p.n_cm;
  const int n0 = nt * BNG;
  const int ncols = min(BNG, p.D - n0);

  if (s.kb0 > 0) {
    // non-owner: hand the fp32 accumulator to the owner
    float* my_part = p.partial + (static_cast<size_t>(cta) * BM + row) * BNG;
#pragma unroll 1
    for (int c = 0; c < BNG / 32; ++c) {
      const int jc = c * 32;
      if (jc >= ncols) break;
      uint32_t r[32];
      tmem_ld32(taddr + jc, r);
      tmem_ld_wait();
      float4* dst = reinterpret_cast<float4*>(my_part + jc);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        dst[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                             __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
    }
    __threadfence();
    __syncwarp();
    if (lane == 0) flag_release(p.flags + cta * 4 + q);
    return true;
  }

  // owner or whole tile: CTAs gi+1 .. j_end-1 of the group hold the rest of it
  int j_end = gi + 1;
  if (s.kb1 < s.len) {
    const long long ue = tile_start(p, s.tile) + s.len;
    while (j_end < p.group_ctas && range_begin(p, j_end) < ue) ++j_end;
    int ok = 1;
    if (lane == 0) {
      for (int j = gi + 1; j < j_end && ok; ++j)
        if (range_begin(p, j) < range_begin(p, j + 1))  // an empty range holds nothing
          ok = flag_wait(p.flags + (j * p.n_nt + nt) * 4 + q, abort_flag, p.status) ? 1 : 0;
    }
    __syncwarp();  // orders lane 0's acquire before the other lanes' reads of the partials
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) return false;
  }

  int v = 0;
  bool valid;
  if (is_dw) {
    const int j = mt * BM + row;
    valid = j < p.C;
    if (valid) {
      v = __ldg(p.cand + j);
      if (static_cast<unsigned>(v) >= static_cast<unsigned>(p.V)) {
        set_status(p.status, SS_ERR_INDEX);
        valid = false;
      }
    }
  } else {
    valid = mt * BM + row < p.T;
  }
#pragma unroll 1
  for (int c = 0; c < BNG / 32; ++c) {
    const int jc = c * 32;
    if (jc >= ncols) break;
    uint32_t r[32];
    tmem_ld32(taddr + jc, r);
    tmem_ld_wait();
    float x[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(r[i]);
    for (int j = gi + 1; j < j_end; ++j) {
      if (range_begin(p, j) >= range_begin(p, j + 1)) continue;
      const float4* src = reinterpret_cast<const float4*>(
          p.partial + (static_cast<size_t>(j * p.n_nt + nt) * BM + row) * BNG + jc);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 w = __ldcg(src + i);
        x[4 * i] += w.x;
        x[4 * i + 1] += w.y;
        x[4 * i + 2] += w.z;
        x[4 * i + 3] += w.w;
      }
    }
    if (!valid) continue;
    if (is_dw) {
      float4* dst = reinterpret_cast<float4*>(p.dW + static_cast<size_t>(v) * p.D + n0 + jc);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float4 o = make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
        if (p.accumulate) {
          const float4 old = dst[i];
          o.x += old.x;
          o.y += old.y;
          o.z += old.z;
          o.w += old.w;
        }
        dst[i] = o;
      }
    } else {
      uint4* dst = reinterpret_cast<uint4*>(p.dH + static_cast<size_t>(mt * BM + row) * p.D + n0 + jc);
#pragma unroll
      for (int w = 0; w < 4; ++w)
        dst[w] = make_uint4(pack_bf16x2(x[8 * w], x[8 * w + 1]), pack_bf16x2(x[8 * w + 2], x[8 * w + 3]),
                            pack_bf16x2(x[8 * w + 4], x[8 * w + 5]),
                            pack_bf16x2(x[8 * w + 6], x[8 * w + 7]));
    }
  }
  return true;
}

__device__ __forceinline__ void release_all_flags(const GradParams& p, int cta) {
  for (int q = 0; q < 4; ++q) flag_release(p.flags + cta * 4 + q);
}

__global__ void __launch_bounds__(GEMM_THREADS, 1)
    k_grad(const __grid_constant__ CUtensorMap tmGk, const __grid_constant__ CUtensorMap tmWcMn,
           const __grid_constant__ CUtensorMap tmGmn, const __grid_constant__ CUtensorMap tmHmn,
           const __grid_constant__ GradParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_go;
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  GemmCtrl* ctrl = reinterpret_cast<GemmCtrl*>(smem + LG::CTRL_OFFSET);
  const uint32_t tiles = smem_u32(smem);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int cta = blockIdx.x;
  const int nt = cta % p.n_nt;  // column slice of this CTA's group
  const int gi = cta / p.n_nt;  // index inside the group

  if (threadIdx.x == 0) s_go = (read_status(p.status) == 0);
  __syncthreads();
  if (!s_go) {
    // publish the flags anyway, so that no owner of this launch waits on us
    if (threadIdx.x == 0) release_all_flags(p, cta);
    return;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesGrad; ++s) {
      mbar_init(&ctrl->full[s], 1);
      mbar_init(&ctrl->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&ctrl->tfull[b], 1);
      mbar_init(&ctrl->tempty[b], 4 * 32);
    }
    mbar_init(&ctrl->drain, 1);
    ctrl->abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_map(&tmGk);
    tma_prefetch_map(&tmWcMn);
    tma_prefetch_map(&tmGmn);
    tma_prefetch_map(&tmHmn);
  }
  if (warp == 1) {
    tmem_alloc(&ctrl->tmem_base, 2 * BNG);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ctrl->tmem_base;
  volatile int* abort_flag = &ctrl->abort_flag;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0, issued = 0, issued_ph = 0;
      bool ok = true;
      SegIter segs(p, gi);
      Seg g;
      while (ok && segs.next(p, g)) {
        const bool is_dw = g.tile < p.n_cm;
        const int mt = is_dw ? g.tile : g.tile - p.n_cm;
        for (int kb = g.kb0; kb < g.kb1; ++kb) {
          if (!mbar_wait(&ctrl->empty[s], ph ^ 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          uint64_t* fb = &ctrl->full[s];
          mbar_arrive_expect_tx(fb, LG::STAGE_BYTES);
          const uint32_t a_dst = tiles + s * LG::STAGE_BYTES;
          const uint32_t b_dst = a_dst + LG::A_BYTES;
          if (is_dw) {  // A = G columns (MN-major), B = H (MN-major); K = tokens
            tma_load_2d(a_dst, &tmGmn, fb, mt * BM, kb * BK);
            tma_load_2d(a_dst + 8192, &tmGmn, fb, mt * BM + 64, kb * BK);
#pragma unroll
            for (int i = 0; i < BNG / 64; ++i)
              tma_load_2d(b_dst + i * 8192, &tmHmn, fb, nt * BNG + 64 * i, kb * BK);
          } else {      // A = G rows (K-major), B = W_c (MN-major); K = candidates
            tma_load_2d(a_dst, &tmGk, fb, kb * BK, mt * BM);
#pragma unroll
            for (int i = 0; i < BNG / 64; ++i)
              tma_load_2d(b_dst + i * 8192, &tmWcMn, fb, nt * BNG + 64 * i, kb * BK);
          }
          issued |= 1u << s;
          issued_ph = (issued_ph & ~(1u << s)) | (ph << s);
          if (++s == kStagesGrad) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      for (int i = 0; i < kStagesGrad; ++i)
        if ((issued >> i) & 1u) mbar_drain(&ctrl->full[i], (issued_ph >> i) & 1u, p.status);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_dw = idesc_bf16_f32(BM, BNG, true, true);
      constexpr uint32_t idesc_dh = idesc_bf16_f32(BM, BNG, false, true);
      int s = 0, b = 0;
      uint32_t ph = 0, aph = 0;
      bool ok = true;
      SegIter segs(p, gi);
      Seg g;
      while (ok && segs.next(p, g)) {
        const bool is_dw = g.tile < p.n_cm;
        if (!mbar_wait(&ctrl->tempty[b], aph ^ 1u, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * BNG);
        for (int kb = g.kb0; kb < g.kb1; ++kb) {
          if (!mbar_wait(&ctrl->full[s], ph, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = tiles + s * LG::STAGE_BYTES;
          const uint32_t b_addr = a_addr + LG::A_BYTES;
#pragma unroll
          for (int k = 0; k < BK / UMMA_K; ++k) {
            const uint64_t ad = is_dw ? sdesc_sw128(a_addr + k * 2048, 8192, 1024)
                                      : sdesc_sw128(a_addr + k * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(b_addr + k * 2048, 8192, 1024);
            mma_bf16(d_tmem, ad, bd, is_dw ? idesc_dw : idesc_dh,
                     (kb > g.kb0 || k > 0) ? 1u : 0u);
          }
          mma_commit(&ctrl->empty[s]);
          if (++s == kStagesGrad) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(&ctrl->tfull[b]);
        if (++b == 2) {
          b = 0;
          aph ^= 1u;
        }
      }
      mma_commit(&ctrl->drain);
      mbar_drain(&ctrl->drain, 0, p.status);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    // Each warp decides on its own (no barrier spans the epilogue warps).
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    int b = 0;
    uint32_t aph = 0;
    SegIter segs(p, gi);
    Seg g;
    while (segs.next(p, g)) {
      const bool ok = mbar_wait(&ctrl->tfull[b], aph, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      if (!grad_epilogue(p, g, nt, cta, gi, q, lane, row,
                         lane_addr + static_cast<uint32_t>(b * BNG), abort_flag))
        break;
      tc_fence_before();
      mbar_arrive(&ctrl->tempty[b]);
      if (++b == 2) {
        b = 0;
        aph ^= 1u;
      }
    }
  }
  __syncthreads();
  // A CTA that aborted before handing over its partials still releases its
  // flags (its owner then reads stale data, but the status word says so).
  if (threadIdx.x == 0 && *abort_flag) release_all_flags(p, cta);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 2 * BNG);
  }
}

}  // namespace

size_t grad_partial_bytes() { return static_cast<size_t>(kMaxGradCtas) * BM * BNG * sizeof(float); }
size_t grad_flag_bytes() { return static_cast<size_t>(kMaxGradCtas) * 4 * sizeof(int); }

cudaError_t launch_grads(const CUtensorMap& tG_kmaj, const CUtensorMap& tWc_mn,
                         const CUtensorMap& tG_mn, const CUtensorMap& tH_mn, int T, int C, int D,
                         int V, int accumulate, const int32_t* cand, uint16_t* dH, float* dW,
                         float* partial, int* flags, int* status, int num_sms,
                         cudaStream_t stream) {
  GradParams p;
  p.T = T;
  p.C = C;
  p.D = D;
  p.V = V;
  p.accumulate = accumulate;
  p.n_nt = (D + BNG - 1) / BNG;
  p.n_cm = (C + BM - 1) / BM;
  p.n_tm = (T + BM - 1) / BM;
  p.kb_dw = (T + BK - 1) / BK;
  p.kb_dh = (C + BK - 1) / BK;
  const int ctas = num_sms < kMaxGradCtas ? num_sms : kMaxGradCtas;
  p.group_ctas = ctas / p.n_nt;
  if (p.group_ctas < 1) return cudaErrorInvalidConfiguration;
  p.cand = cand;
  p.dH = dH;
  p.dW = dW;
  p.partial = partial;
  p.flags = flags;
  p.status = status;
  const int grid = p.group_ctas * p.n_nt;
  cudaError_t e = cudaMemsetAsync(flags, 0, static_cast<size_t>(grid) * 4 * sizeof(int), stream);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k_grad, cudaFuncAttributeMaxDynamicSharedMemorySize, LG::TOTAL);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(GEMM_THREADS);
  cfg.dynamicSmemBytes = LG::TOTAL;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_grad, tG_kmaj, tWc_mn, tG_mn, tH_mn, p);
}

}  // namespace ss
