// ss_gemm.cuh -- persistent, warp-specialised bf16 GEMM on the 5th-generation
// tensor cores of sm_103a, with the sampled-softmax epilogues fused in.
//
// One CTA per SM walks a static round-robin list of 128 x BN output tiles
// ("units"). Roles:
//   warp 0, one lane : TMA producer -- loads 128 x 64 A and BN x 64 B blocks
//                      (128-byte swizzle) into a STAGES-deep ring.
//   warp 1, one lane : MMA issuer  -- tcgen05.mma 128 x BN x 16 into one of two
//                      TMEM accumulators (2 x BN fp32 columns), commits to
//                      mbarriers to free ring slots and to hand tiles over.
//   warps 2-5        : epilogue    -- tcgen05.ld the accumulator (warp w owns
//                      TMEM lanes 32*(w%4)..+31, one output row per thread),
//                      apply the fused epilogue, release the accumulator.
// The epilogue of tile i overlaps the MMAs of tile i+1.
//
// Operand layouts (A is M x K, B is N x K in the MMA's terms):
//   K-major : the K index is contiguous in memory; one TMA box of 64 (K) x rows.
//   MN-major: the M/N index is contiguous; boxes of 64 (M/N) x 64 (K), one per
//             64-wide M/N chunk, laid out 8 KB apart.
// Out-of-range rows/columns of a box are zero-filled by TMA, so ragged M, N
// and K edges need no special casing in the main loop.
#pragma once

#include <string.h>

#include <math.h>

#include <type_traits>

#include "ss_internal.h"
#include "ss_ptx.cuh"

namespace ss {

constexpr int BM = 128;          // tile rows = TMEM lanes
constexpr int BK = 64;           // 64 bf16 = one 128-byte swizzle row
constexpr int UMMA_K = 16;       // K of one tcgen05.mma kind::f16
constexpr int GEMM_THREADS = 192;
constexpr float kLog2e = 1.4426950408889634f;

template <int BN, int STAGES, int EPI_BYTES>
struct GemmSmem {
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int TILES_BYTES = STAGES * STAGE_BYTES;
  static constexpr int EPI_OFFSET = TILES_BYTES;              // epilogue staging (1024-aligned)
  static constexpr int CTRL_OFFSET = TILES_BYTES + EPI_BYTES;
  static constexpr int CTRL_BYTES = 256;
  static constexpr int TOTAL = CTRL_OFFSET + CTRL_BYTES + 1024;  // + 1024-byte alignment slack
  static_assert(TOTAL <= 232448, "shared memory per CTA");
};

// Per-thread state the epilogue keeps across tiles.
struct EpiState {
  uint32_t stage;   // shared address of the epilogue staging region
  int ep_tid;       // index among the epilogue threads
  uint32_t rounds;  // staging buffers used so far
  float f0;         // a per-launch constant an epilogue computes in begin() (FP8 scales)
};

struct GemmCtrl {
  uint64_t full[8];
  uint64_t empty[8];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int vote[2][8];  // per-tile vote of the epilogue warps (alternating halves)
};

// Units are (m_tile, n_tile) pairs numbered m-major: u = m_tile * n_tiles + n_tile.
struct GemmShape {
  int m_tiles;
  int n_tiles;
  int k_blocks;
  // 1: the operands are older than the kernel just before this one in the
  // stream, and only the epilogue reads what that kernel writes. The producer
  // and MMA warps then start at once; the epilogue waits before its first
  // tile.
  // 2 (k_gemm2): nothing this kernel reads or writes is touched by the kernel
  // just before it, whose own wait covers everything older: no part waits
  // before the work, and the kernel's CTAs take SMs as that kernel's last
  // tiles free them; each CTA waits for it before exiting, so that the kernels
  // after this one, which wait for this one, also find that one finished.
  int late_wait;
  // the units cover the column tiles [n_begin, n_tiles) (0: all)
  int n_begin;
  // non-null: the kernel does its work only if *gate != 0, read once the
  // kernels before it have completed (no late_wait); else every CTA returns
  int* gate;
  // > 0: the units walk groups of group_m row tiles column tile by column
  // tile (the B tile of a column is reused by the group's rows while it is in
  // L2, and the group's A rows stay in L2 across the columns); 0: row by row
  int group_m;
};

// Unit u -> (row tile, column tile) of a GemmShape (column tiles
// [n_begin, n_tiles)), in the order group_m asks for.
__device__ __forceinline__ void unit_tile(const GemmShape& shp, int u, int& mt, int& nt) {
  const int n_cols = shp.n_tiles - shp.n_begin;
  if (shp.group_m <= 0) {
    mt = u / n_cols;
    nt = shp.n_begin + u % n_cols;
    return;
  }
  const int per = shp.group_m * n_cols;
  const int g = u / per, w = u % per;
  const int gm = min(shp.group_m, shp.m_tiles - g * shp.group_m);
  mt = g * shp.group_m + w % gm;
  nt = shp.n_begin + w / gm;
}

// ----------------------------------------------------------------- epilogues

// Runs fn(r, i) over the 32-column chunks [c_begin, c_begin + n) of this
// thread's TMEM row, with the load of chunk i + 1 in flight while chunk i is
// processed. on_loaded() runs once, as soon as the last chunk is in registers
// (before fn processes it): an epilogue that owns its accumulator release
// hands the TMEM buffer back to the MMA warp there.
template <int N, class F, class G>
__device__ __forceinline__ void for_tmem_chunks(uint32_t taddr, int c_begin, F&& fn,
                                                G&& on_loaded) {
  uint32_t ra[32], rb[32];
  tmem_ld32(taddr + c_begin * 32, ra);
#pragma unroll
  for (int i = 0; i < N; i += 2) {
    tmem_ld_wait(ra);
    if (i + 1 < N) tmem_ld32(taddr + (c_begin + i + 1) * 32, rb);
    if (i + 1 == N) on_loaded();
    fn(ra, i);
    if (i + 1 < N) {
      tmem_ld_wait(rb);
      if (i + 2 < N) tmem_ld32(taddr + (c_begin + i + 2) * 32, ra);
      if (i + 2 == N) on_loaded();
      fn(rb, i + 1);
    }
  }
}
template <int N, class F>
__device__ __forceinline__ void for_tmem_chunks(uint32_t taddr, int c_begin, F&& fn) {
  for_tmem_chunks<N>(taddr, c_begin, static_cast<F&&>(fn), [] {});
}

// Epilogues with `static constexpr bool kSelfRelease = true` take a release()
// functor as the last argument of apply() and call it once, after their last
// TMEM load of the tile and before their global stores: the MMA warp may then
// start the tile after next in that buffer while the stores are in flight, and
// the release-ordered mbarrier arrive does not wait for those stores.
template <class E, class = void>
struct EpiSelfRelease : std::false_type {};
template <class E>
struct EpiSelfRelease<E, std::void_t<decltype(E::kSelfRelease)>>
    : std::integral_constant<bool, E::kSelfRelease> {};

// x[off & 31]: a five-level select tree on the bits of off (31 selects,
// where comparing every index with off takes 32 compares and 32 selects)
template <class Tv>
__device__ __forceinline__ Tv select32(const Tv (&x)[32], int off) {
  Tv a[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) a[i] = (off & 1) ? x[2 * i + 1] : x[2 * i];
#pragma unroll
  for (int i = 0; i < 8; ++i) a[i] = (off & 2) ? a[2 * i + 1] : a[2 * i];
#pragma unroll
  for (int i = 0; i < 4; ++i) a[i] = (off & 4) ? a[2 * i + 1] : a[2 * i];
#pragma unroll
  for (int i = 0; i < 2; ++i) a[i] = (off & 8) ? a[2 * i + 1] : a[2 * i];
  return (off & 16) ? a[1] : a[0];
}

// The capped head: z = cap / (1 + exp(-s / tau)) = cap * 1 / (1 + 2^(-s k1)),
// k1 = log2(e) / tau, and dz/ds = z (cap - z) icap_tau, icap_tau = 1 / (cap tau).
__device__ __forceinline__ float head_z(float s, const HeadCap& h) {
  return h.cap * rcp_approx(1.f + ex2_approx(-s * h.k1));
}
__device__ __forceinline__ float head_dz(float z, const HeadCap& h) {
  return z * (h.cap - z) * h.icap_tau;
}

// amax[0] = max |H|, amax[1] = max |W_c|: the scale that turns the e4m3
// accumulator back into logits
__device__ __forceinline__ float e4m3_logit_scale(const float* amax) {
  return exp2i(-(e4m3_exponent(__ldcg(amax)) + e4m3_exponent(__ldcg(amax + 1))));
}

// Forward: per-row softmax partials of one 128 x BN logit tile.
//   With NCG column groups per tile (NCG epilogue warps per row block), group
//   cg covers columns [cg * BN / NCG, (cg + 1) * BN / NCG) of the tile and
//   writes part[nt * NCG + cg][t] = (max_j S[t,j], sum_j exp(S[t,j] - max))
//   over its valid columns, or (-inf, 0) if it has none; tgt[t] = S[t, slot[t]]
//   comes from the group that holds slot[t].
template <bool CAP, int KMAX = 1, bool F8 = false>
struct EpiFwdT {
  static constexpr int kStageBytes = 0;
  static constexpr bool kKeepOperands = false;
  struct Params {
    int T, C;
    const int32_t* slot;
    float2* part;
    float* tgt;    // [K * T]: the logit (z when CAP) of each target
    int* status;
    HeadCap head;  // used when CAP: the partials and the target logit are of z
    Targets tg;    // used when KMAX > 1
    const float* amax;  // used when F8: logits = accumulator * e4m3_logit_scale(amax)
  };
  // F8: the logit scale, the same for every tile, loaded once per launch
  __device__ static void begin(const Params& p, EpiState& es) {
    if constexpr (F8) es.f0 = e4m3_logit_scale(p.amax);
  }
  __device__ static void finish(const Params&, EpiState&) {}
  template <int BN, int NCG>
  __device__ static void apply(const Params& p, int mt, int nt, int row, uint32_t taddr,
                               EpiState& es, int cg) {
    constexpr int CPG = BN / 32 / NCG;  // chunks per group
    const int t = mt * BM + row;
    const bool valid = t < p.T;
    const int K = KMAX > 1 ? p.tg.K : 1;
    int sl[KMAX];
#pragma unroll
    for (int k = 0; k < KMAX; ++k)
      sl[k] = (valid && k < K) ? __ldg(p.slot + static_cast<size_t>(k) * p.T + t) : -1;
    const int j0 = nt * BN + cg * CPG * 32;  // first column of this group
    const int ncols = min(CPG * 32, p.C - j0);
    float s = 0.f, tg[KMAX];
    uint32_t has_t = 0u;  // bit k: target k lies in this group's columns
    float sig = 1.f;
    if constexpr (F8) sig = es.f0;
    // capped head: the e4m3 scale folds into the cap's exponent constant, and
    // z < cap, so (for cap <= 64, where exp(z - cap) stays normal) cap itself
    // is the softmax offset and no running max is needed
    HeadCap hz = p.head;
    if constexpr (CAP && F8) hz.k1 *= sig;
    const bool fixed = CAP && p.head.cap <= 64.f;  // uniform
    float m = fixed && ncols > 0 ? p.head.cap : -INFINITY;
    // Plain head: v holds the raw accumulator and the logit is v * vs (the
    // FP8 scale is a power of two, so it commutes exactly with the max and
    // folds into the exponent's constant); capped head: v = z, vs = 1.
    const float vs = CAP ? 1.f : sig;
    const float k2 = vs * kLog2e;
    if (ncols > 0) {  // uniform: depends on the tile only
      for_tmem_chunks<CPG>(taddr, cg * CPG, [&](const uint32_t(&r)[32], int i) {
        const int jc = i * 32;
        const int nv = min(32, ncols - jc);
        if (nv <= 0) return;
        float v[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const float acc = __uint_as_float(r[k]);
          v[k] = CAP ? head_z(acc, hz) : acc;
        }
        float cm = -INFINITY;
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
        float nm;
        if (CAP && fixed) {  // offset cap: no max, no rescale
          nm = m;
          const float nm2 = nm * kLog2e;
#pragma unroll
          for (int k = 0; k < 32; k += 4) {
            if (nv == 32 || k + 0 < nv) a0 += ex2_approx(fmaf(v[k + 0], kLog2e, -nm2));
            if (nv == 32 || k + 1 < nv) a1 += ex2_approx(fmaf(v[k + 1], kLog2e, -nm2));
            if (nv == 32 || k + 2 < nv) a2 += ex2_approx(fmaf(v[k + 2], kLog2e, -nm2));
            if (nv == 32 || k + 3 < nv) a3 += ex2_approx(fmaf(v[k + 3], kLog2e, -nm2));
          }
        } else if (nv == 32) {  // a full chunk (all but a ragged tail): no per-column predicates
#pragma unroll
          for (int k = 0; k < 32; ++k) cm = fmaxf(cm, v[k]);
          nm = fmaxf(m, cm * vs);
          const float nm2 = nm * kLog2e;
#pragma unroll
          for (int k = 0; k < 32; k += 4) {
            a0 += ex2_approx(fmaf(v[k + 0], k2, -nm2));
            a1 += ex2_approx(fmaf(v[k + 1], k2, -nm2));
            a2 += ex2_approx(fmaf(v[k + 2], k2, -nm2));
            a3 += ex2_approx(fmaf(v[k + 3], k2, -nm2));
          }
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k)
            if (k < nv) cm = fmaxf(cm, v[k]);
          nm = fmaxf(m, cm * vs);
          const float nm2 = nm * kLog2e;
#pragma unroll
          for (int k = 0; k < 32; k += 4) {
            if (k + 0 < nv) a0 += ex2_approx(fmaf(v[k + 0], k2, -nm2));
            if (k + 1 < nv) a1 += ex2_approx(fmaf(v[k + 1], k2, -nm2));
            if (k + 2 < nv) a2 += ex2_approx(fmaf(v[k + 2], k2, -nm2));
            if (k + 3 < nv) a3 += ex2_approx(fmaf(v[k + 3], k2, -nm2));
          }
        }
        if (CAP && fixed) {
          s += (a0 + a1) + (a2 + a3);
        } else {
          s = s * ex2_approx((m - nm) * kLog2e) + ((a0 + a1) + (a2 + a3));
          m = nm;
        }
#pragma unroll
        for (int k = 0; k < KMAX; ++k) {
          if (k >= K) break;  // uniform
          const int off = sl[k] - j0 - jc;
          const bool hit = static_cast<unsigned>(off) < static_cast<unsigned>(nv);
          // a target falls in a given 32-column chunk for a few rows of a warp
          // at most: skip the selection unless one does
          if (__any_sync(0xffffffffu, hit)) {
            if (hit) {
              tg[k] = select32(v, off) * vs;
              has_t |= 1u << k;
            }
          }
        }
      });
    }
    if (valid) {
      p.part[static_cast<size_t>(nt * NCG + cg) * p.T + t] = make_float2(m, s);
#pragma unroll
      for (int k = 0; k < KMAX; ++k)
        if ((has_t >> k) & 1u) p.tgt[static_cast<size_t>(k) * p.T + t] = tg[k];
    }
  }
};
using EpiFwd = EpiFwdT<false>;

// Backward, step 1: G[t, j] = scale * (exp(S[t,j] - lse[t]) - [j == slot[t]]), bf16.
// Folded form: scale * exp(x - lse) = sign(scale) * 2^(x*log2e - (lse*log2e - log2|scale|)).
// Each 64-column quarter of the tile is written into a 16 KB shared-memory
// buffer in the 128-byte-swizzled layout of the G tensor map (two buffers,
// alternating) and stored with one TMA bulk tensor store, so the global
// writes leave as full lines instead of 32 rows per warp instruction. The
// one-hot term touches one element per row: it is recomputed in fp32 and
// patched into the staged tile.
template <bool CAP, int KMAX = 1, bool F8 = false>
struct EpiGT {
  // 16 KB staging buffers, split between the column groups: two (bf16), or
  // four with the e4m3 operands, whose tiles take half as long, so that a
  // group never waits for its last store to have read the buffer
  static constexpr int kStageBytes = (F8 ? 4 : 2) * 16384;
  // G streams through L2 once; the H and W_c tiles are re-read by every CTA
  static constexpr bool kKeepOperands = true;
  static constexpr bool kSelfRelease = true;
  struct Params {
    CUtensorMap tmG;  // G [T, C] bf16 (row pitch ldG), box 64 x 128, 128-byte swizzle
    int T, C;
    const int32_t* slot;
    const float* lse;
    float scale;       // d(objective)/d(loss)
    float log2_scale;  // log2|scale| (-inf for 0)
    int* status;
    HeadCap head;      // used when CAP: G = scale * (P(z) - Y) * dz/ds
    Targets tg;        // the targets' weights: G = scale (W P - sum_k w[k] Y_k), W = sum_k w[k]
                       // (one target: W = w[0], 1 for the single-target loss); log2_scale is
                       // log2(|scale| W)
    const float* amax;  // used when F8: logits = accumulator * e4m3_logit_scale(amax)
    // non-null: the stored-probability step's fallback also resets, for each
    // row t (in its first column tile), fix_Hs[t, :] = fix_H[t, :] and
    // fix_rowfac[t] = fix_scale (D columns, bf16)
    const uint16_t* fix_H;
    uint16_t* fix_Hs;
    float* fix_rowfac;
    float fix_scale;
    int D;
  };
  __device__ static void begin(const Params& p, EpiState& es) {
    if constexpr (F8) es.f0 = e4m3_logit_scale(p.amax);
  }
  __device__ static void finish(const Params&, EpiState& es) {
    if ((es.ep_tid & 127) == 0) bulk_wait<0>();
  }
  // Column group cg of NCG (four warps each) covers quarters
  // [cg * 4 / NCG, (cg + 1) * 4 / NCG) of the tile with its own staging
  // buffer(s), named barrier (1 + 2 * cg) and storing thread.
  template <int BN, int NCG, class Rel>
  __device__ static void apply(const Params& p, int mt, int nt, int row, uint32_t taddr,
                               EpiState& es, int cg, Rel&& release) {
    static_assert(NCG == 1 || NCG == 2, "column groups");
    const int bar = 1 + 2 * cg;
    const bool leader = (es.ep_tid & 127) == 0;
    const int t = mt * BM + row;
    const bool valid = t < p.T;
    const int K = KMAX > 1 ? p.tg.K : 1;
    int sl[KMAX];
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
      sl[k] = (valid && k < K) ? __ldg(p.slot + static_cast<size_t>(k) * p.T + t) : -1;
      if (valid && k < K && nt == 0 && static_cast<unsigned>(sl[k]) >= static_cast<unsigned>(p.C))
        set_status(p.status, SS_ERR_INDEX);
    }
    if (p.fix_H != nullptr && nt == 0 && cg == 0 && valid) {
      const uint4* src = reinterpret_cast<const uint4*>(p.fix_H + static_cast<size_t>(t) * p.D);
      uint4* dst = reinterpret_cast<uint4*>(p.fix_Hs + static_cast<size_t>(t) * p.D);
      for (int i = 0; i < p.D / 8; ++i) dst[i] = __ldg(src + i);
      p.fix_rowfac[t] = p.fix_scale;
    }
    const float asc = fabsf(p.scale);
    float sig = 1.f;
    if constexpr (F8) sig = es.f0;
    const float k2 = sig * kLog2e;
    HeadCap hz = p.head;  // capped: the e4m3 scale folded into the exponent constant
    if constexpr (CAP && F8) hz.k1 *= sig;
    const uint32_t sgn = p.scale < 0.f ? 0x80008000u : 0u;
    const float off2 = valid ? fmaf(__ldg(p.lse + t), kLog2e, -p.log2_scale) : 0.f;
    const int j0 = nt * BN;
    const int ncols = min(BN, p.C - j0);
    const uint32_t r7 = static_cast<uint32_t>(row & 7);
    // the last 32-column chunk this group loads from TMEM: the accumulator is
    // handed back right after it (a group with no columns hands it back now)
    const int q_begin = cg * (BN / 64) / NCG, q_end = (cg + 1) * (BN / 64) / NCG;
    const int c_end = min(q_end * 64, ncols);
    const int jc_last = c_end > q_begin * 64 ? (c_end - 1) / 32 * 32 : -1;
    if (jc_last < 0) release();
#pragma unroll 1
    for (int q = q_begin; q < q_end; ++q) {
      const int qc = q * 64;
      if (qc >= ncols) break;  // uniform: depends on the tile only
      constexpr uint32_t kBufs = kStageBytes / 16384 / NCG;  // buffers per column group
      const uint32_t buf = es.stage + static_cast<uint32_t>(cg) * 16384u * kBufs +
                           (es.rounds % kBufs) * 16384u;
      // the store that last used this buffer must have read it
      if (es.rounds >= kBufs && leader) bulk_wait_read<static_cast<int>(kBufs) - 1>();
      named_bar_sync(bar, 128);
      const uint32_t rowbase = buf + static_cast<uint32_t>(row) * 128u;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int jc = qc + 32 * h;
        if (jc >= ncols) break;
        uint32_t r[32];
        tmem_ld32(taddr + jc, r);
        tmem_ld_wait(r);
        if (jc == jc_last) release();
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float g0, g1;
          if constexpr (CAP) {
            const float z0 = head_z(__uint_as_float(r[2 * i]), hz);
            const float z1 = head_z(__uint_as_float(r[2 * i + 1]), hz);
            g0 = ex2_approx(fmaf(z0, kLog2e, -off2)) * head_dz(z0, p.head);
            g1 = ex2_approx(fmaf(z1, kLog2e, -off2)) * head_dz(z1, p.head);
          } else {  // sig (a power of two) folded into the constant: the same value
            g0 = ex2_approx(fmaf(__uint_as_float(r[2 * i]), k2, -off2));
            g1 = ex2_approx(fmaf(__uint_as_float(r[2 * i + 1]), k2, -off2));
          }
          pk[i] = pack_bf16x2(g0, g1) ^ sgn;
        }
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const uint32_t ci = static_cast<uint32_t>(h * 4 + v);
          st_shared_v4(rowbase + ((ci ^ r7) << 4), pk[4 * v], pk[4 * v + 1], pk[4 * v + 2],
                       pk[4 * v + 3]);
        }
#pragma unroll
        for (int k = 0; k < KMAX; ++k) {
          if (k >= K) break;  // uniform
          const int off = sl[k] - j0 - jc;
          const bool has = static_cast<unsigned>(off) < 32u;
          if (__any_sync(0xffffffffu, has)) {
            float xt = __uint_as_float(select32(r, off));  // used where has
            if constexpr (F8 && !CAP) xt *= sig;  // capped: hz carries the scale
            if (has) {
              // the one-hot weight of this column: every target k2 that falls on it
              // (one target: its own weight, 1 for the single-target loss)
              float wt = 0.f;
#pragma unroll
              for (int k2 = 0; k2 < KMAX; ++k2) wt += (sl[k2] == sl[k]) ? p.tg.w[k2] : 0.f;
              float gt;
              if constexpr (CAP) {
                const float zt = head_z(xt, hz);
                gt = (ex2_approx(fmaf(zt, kLog2e, -off2)) - asc * wt) * head_dz(zt, p.head);
              } else {
                gt = ex2_approx(fmaf(xt, kLog2e, -off2)) - asc * wt;
              }
              const uint16_t bits = bf16_bits(gt) ^ static_cast<uint16_t>(sgn & 0xffffu);
              const uint32_t cc = static_cast<uint32_t>(32 * h + off);
              st_shared_b16(rowbase + (((cc >> 3) ^ r7) << 4) + (cc & 7u) * 2u, bits);
            }
          }
        }
      }
      fence_proxy_async_smem();
      named_bar_sync(bar, 128);
      if (leader) {
        tma_store_2d_hint(&p.tmG, buf, j0 + qc, mt * BM, l2_evict_first());
        bulk_commit();
      }
      ++es.rounds;
    }
  }
};
using EpiG = EpiGT<false>;

// Forward that keeps the probabilities for the backward (plain bf16 head, one
// target per token). Besides the per-row softmax partials and the target
// logit of EpiFwdT, it writes
//   Pt[t, j] = exp(S[t,j] - r[t])  (bf16, every column of the tile),
// with r[t] a per-row reference fixed before the tiles after the first: the
// row's largest logit over the first logit tile. PRE: this launch covers that
// tile only, finds r[t] itself (every thread of a row reads the row's whole
// tile from TMEM, so both column groups find the same value) and stores it;
// otherwise r[t] is read back. Once lse is known,
//   G[t,j] = scale (P - Y) = scale exp(r - lse) (Pt - Y exp(lse - r)),
// so the backward needs no second pass over the logits (the merge patches
// the target column and supplies the per-row factor).
// The partial's reference is r as well: per logit one FMA and one exp give
// both Pt and the partial's term. Only if a 32-column chunk's sum could
// overflow (a logit some 59 above r) does that thread move the partial to a
// running max, as EpiFwdT keeps it; Pt is then out of range, which the merge
// detects (lse - r too large) and answers with the recompute.
// The staging and the TMA stores are those of EpiGT; two column groups, two
// partials per row per tile, part[(nt * 2 + cg) * T + t].
// CAP: the capped head z = cap / (1 + exp(-s / tau)). Since z < cap, the
// reference is r = cap for every row (no first launch; exp(z - cap) stays a
// normal number for cap <= 64), the partials are of exp(z - cap), and
//   Pt[t, j] = exp(z[t,j] - cap) dz/ds[t,j],
// so that G = scale (P - Y) dz/ds = scale exp(cap - lse) (Pt - Y exp(lse - cap) dz/ds);
// the target logit stored is z.
template <bool PRE, int NBUF = 1, bool CAP = false, int KMAX = 1>
struct EpiFwdP {
  static_assert(!(PRE && CAP), "the capped head's reference is cap: no first launch");
  // NBUF 16 KB staging buffers per column group: with two, a group fills one
  // while the store of the other is still reading it
  static_assert(NBUF == 1 || NBUF == 2, "staging buffers per column group");
  static constexpr int kStageBytes = 2 * NBUF * 16384;
  // Pt streams through L2 once; the H and W_c tiles are re-read by every CTA
  static constexpr bool kKeepOperands = true;
  static constexpr bool kSelfRelease = true;
  struct Params {
    CUtensorMap tmP;  // Pt [T, C] bf16 (row pitch ldG), box 64 x 128, 128-byte swizzle
    int T, C;
    const int32_t* slot;  // [K, T]
    float2* part;
    float* tgt;        // [K, T]: S[t, slot[k T + t]] (z with CAP)
    float* ref;        // [T]: r[t] (PRE writes it, the later tiles read it); not used with CAP
    int* clear_word;   // PRE: set to 0 once (the merge's fallback flag), or null
    int* status;
    HeadCap head;      // used when CAP
    int K;             // targets per token (KMAX > 1; 1 otherwise)
  };
  __device__ static void begin(const Params& p, EpiState& es) {
    if constexpr (PRE)
      if (p.clear_word && blockIdx.x == 0 && es.ep_tid == 0) *p.clear_word = 0;
  }
  __device__ static void finish(const Params&, EpiState& es) {
    if ((es.ep_tid & 127) == 0) bulk_wait<0>();
  }
  template <int BN, int NCG, class Rel>
  __device__ static void apply(const Params& p, int mt, int nt, int row, uint32_t taddr,
                               EpiState& es, int cg, Rel&& release) {
    static_assert(NCG == 2 && BN == 256, "two column groups of two 64-column quarters");
    constexpr int CPG = BN / 32 / NCG;  // 32-column chunks per group
    const int bar = 1 + 2 * cg;
    const bool leader = (es.ep_tid & 127) == 0;
    const int t = mt * BM + row;
    const bool valid = t < p.T;
    const int K = KMAX > 1 ? p.K : 1;
    int sl[KMAX];
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
      sl[k] = valid && k < K ? __ldg(p.slot + static_cast<size_t>(k) * p.T + t) : -1;
      if (valid && k < K && nt == 0 && static_cast<unsigned>(sl[k]) >= static_cast<unsigned>(p.C))
        set_status(p.status, SS_ERR_INDEX);
    }
    const int j0 = nt * BN;
    const int ncols = min(BN, p.C - j0);
    float r;
    if constexpr (PRE) {  // the largest logit of the row over this (first) tile
      r = -INFINITY;
      for_tmem_chunks<BN / 32>(taddr, 0, [&](const uint32_t(&v)[32], int i) {
        const int nv = min(32, ncols - i * 32);
        if (nv <= 0) return;
        if (nv == 32) {
#pragma unroll
          for (int k = 0; k < 32; ++k) r = fmaxf(r, __uint_as_float(v[k]));
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k)
            if (k < nv) r = fmaxf(r, __uint_as_float(v[k]));
        }
      });
      if (valid && cg == 0) p.ref[t] = r;
    } else if constexpr (CAP) {
      r = p.head.cap;
    } else {
      r = valid ? __ldcg(p.ref + t) : 0.f;
    }
    const float r2 = r * kLog2e;
    const uint32_t r7 = static_cast<uint32_t>(row & 7);
    const uint32_t gbuf = es.stage + static_cast<uint32_t>(cg) * (16384u * NBUF);
    // partial (m, s): sum of exp(S - m) over this group's columns, m = r
    // unless a chunk moved it up
    float m = cg * CPG * 32 < ncols ? r : -INFINITY, s = 0.f, tg[KMAX];
    uint32_t has_t = 0u;  // bit k: target k lies in this group's columns
    for_tmem_chunks<CPG>(taddr, cg * CPG, [&](const uint32_t(&v)[32], int i) {
      const int jc = (cg * CPG + i) * 32;  // column of the tile
      if (jc >= ncols) return;             // uniform: depends on the tile only
      const int h = i & 1;                 // half of the 64-column quarter
      const uint32_t buf = gbuf + (es.rounds % NBUF) * 16384u;
      const uint32_t rowbase = buf + static_cast<uint32_t>(row) * 128u;
      if (h == 0) {
        // the store that last used this buffer must have read it
        if (es.rounds >= NBUF && leader) bulk_wait_read<NBUF - 1>();
        named_bar_sync(bar, 128);
      }
      const int nv = min(32, ncols - jc);
      float e[32];
      float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
      if constexpr (CAP) {
        // with w = 1 / (1 + exp(-s / tau)): z = cap w, z - cap = cap (w - 1)
        // and dz/ds = (cap / tau) w (1 - w); x = exp(z - cap) <= 1 enters the
        // partial, x dz/ds goes to Pt (two logits per packed operation)
        const float k1 = p.head.k1, cl2 = r2;  // r = cap
        const float ct = p.head.cap * p.head.cap * p.head.icap_tau;  // cap / tau
        const uint64_t nk1 = f32x2(-k1, -k1), one = f32x2(1.f, 1.f), mone = f32x2(-1.f, -1.f);
        const uint64_t cl = f32x2(cl2, cl2), ncl = f32x2(-cl2, -cl2), ctt = f32x2(ct, ct);
        uint64_t acc = f32x2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < 32; k += 2) {
          float t0, t1;
          f32x2_split(mul_f32x2(f32x2_bits(v[k], v[k + 1]), nk1), t0, t1);
          float q0, q1;
          f32x2_split(add_f32x2(f32x2(ex2_approx(t0), ex2_approx(t1)), one), q0, q1);
          const uint64_t w = f32x2(rcp_approx(q0), rcp_approx(q1));
          float y0, y1;
          f32x2_split(fma_f32x2(w, cl, ncl), y0, y1);
          float x0 = ex2_approx(y0), x1 = ex2_approx(y1);
          if (nv < 32) {
            if (k >= nv) x0 = 0.f;
            if (k + 1 >= nv) x1 = 0.f;
          }
          const uint64_t x = f32x2(x0, x1);
          acc = add_f32x2(acc, x);
          // x (cap / tau) w (1 - w)
          const uint64_t g = mul_f32x2(mul_f32x2(x, ctt), mul_f32x2(w, fma_f32x2(w, mone, one)));
          f32x2_split(g, e[k], e[k + 1]);
        }
        f32x2_split(acc, a0, a1);
      } else if (nv == 32) {  // every chunk but a ragged tail: no per-column predicates
        // two logits per FMA and per add (packed fp32 pairs)
        const uint64_t k2 = f32x2(kLog2e, kLog2e), nr2 = f32x2(-r2, -r2);
        uint64_t s01 = f32x2(0.f, 0.f), s23 = s01;
#pragma unroll
        for (int k = 0; k < 32; k += 4) {
          float y0, y1, y2, y3;
          f32x2_split(fma_f32x2(f32x2_bits(v[k], v[k + 1]), k2, nr2), y0, y1);
          f32x2_split(fma_f32x2(f32x2_bits(v[k + 2], v[k + 3]), k2, nr2), y2, y3);
          e[k + 0] = ex2_approx(y0);
          e[k + 1] = ex2_approx(y1);
          e[k + 2] = ex2_approx(y2);
          e[k + 3] = ex2_approx(y3);
          s01 = add_f32x2(s01, f32x2(e[k + 0], e[k + 1]));
          s23 = add_f32x2(s23, f32x2(e[k + 2], e[k + 3]));
        }
        f32x2_split(s01, a0, a1);
        f32x2_split(s23, a2, a3);
      } else {
#pragma unroll
        for (int k = 0; k < 32; k += 4) {
          e[k + 0] = k + 0 < nv ? ex2_approx(fmaf(__uint_as_float(v[k + 0]), kLog2e, -r2)) : 0.f;
          e[k + 1] = k + 1 < nv ? ex2_approx(fmaf(__uint_as_float(v[k + 1]), kLog2e, -r2)) : 0.f;
          e[k + 2] = k + 2 < nv ? ex2_approx(fmaf(__uint_as_float(v[k + 2]), kLog2e, -r2)) : 0.f;
          e[k + 3] = k + 3 < nv ? ex2_approx(fmaf(__uint_as_float(v[k + 3]), kLog2e, -r2)) : 0.f;
          a0 += e[k + 0];
          a1 += e[k + 1];
          a2 += e[k + 2];
          a3 += e[k + 3];
        }
      }
      const float a = (a0 + a1) + (a2 + a3);
      if (CAP || (a <= 0x1p86f && m == r)) {
        s += a;
      } else {  // rare: the partial takes a running max (robust lse for the fallback)
        float cm = -INFINITY;
#pragma unroll
        for (int k = 0; k < 32; ++k)
          if (nv == 32 || k < nv) cm = fmaxf(cm, __uint_as_float(v[k]));
        const float nm = fmaxf(m, cm);
        const float nm2 = nm * kLog2e;
        float b = 0.f;
#pragma unroll
        for (int k = 0; k < 32; ++k)
          if (nv == 32 || k < nv) b += ex2_approx(fmaf(__uint_as_float(v[k]), kLog2e, -nm2));
        s = s * ex2_approx((m - nm) * kLog2e) + b;
        m = nm;
      }
      uint32_t pk[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) pk[k] = pack_bf16x2(e[2 * k], e[2 * k + 1]);
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const uint32_t ci = static_cast<uint32_t>(h * 4 + w);
        st_shared_v4(rowbase + ((ci ^ r7) << 4), pk[4 * w], pk[4 * w + 1], pk[4 * w + 2],
                     pk[4 * w + 3]);
      }
      // the target logits: a target falls in a given 32-column chunk for a
      // few rows of a warp at most
#pragma unroll
      for (int k = 0; k < KMAX; ++k) {
        if (k >= K) break;  // uniform
        const int off = sl[k] - j0 - jc;
        const bool hit = static_cast<unsigned>(off) < static_cast<unsigned>(nv);
        if (__any_sync(0xffffffffu, hit)) {
          const float x = __uint_as_float(select32(v, off));
          if (hit) {
            tg[k] = CAP ? head_z(x, p.head) : x;
            has_t |= 1u << k;
          }
        }
      }
      if (h == 1 || jc + 32 >= ncols) {  // the quarter is complete: store it
        fence_proxy_async_smem();
        named_bar_sync(bar, 128);
        if (leader) {
          tma_store_2d_hint(&p.tmP, buf, j0 + jc - 32 * h, mt * BM, l2_evict_first());
          bulk_commit();
        }
        ++es.rounds;
      }
    }, release);
    if (valid) {
      p.part[static_cast<size_t>(nt * 2 + cg) * p.T + t] = make_float2(m, s);
#pragma unroll
      for (int k = 0; k < KMAX; ++k)
        if ((has_t >> k) & 1u) p.tgt[static_cast<size_t>(k) * p.T + t] = tg[k];
    }
  }
};

// FP8 gradients: G (before `scale`) is scaled by 2^g8e, the largest power of
// two that keeps its bound -- |P - Y| <= 1, times dz/ds <= cap / (4 tau) with
// the capped head -- within e5m2's largest finite value (57344) (g8e = 15 for
// the plain head), and rounded to e5m2; the scale and the operand's e4m3
// exponent come back out of the gradient GEMMs' fp32 accumulators.
__device__ __forceinline__ float fp8_grad_alpha(float scale, int g8e, const float* amax_b) {
  return scale * exp2i(-(g8e + e4m3_exponent(__ldcg(amax_b))));
}

// Backward, step 1 with FP8 gradients (e4m3 logit operands):
//   G8[t, j] = e5m2(2^g8e (exp(z[t,j] - lse[t]) - [j == slot[t]]) dz/ds)
// (z = S and dz/ds = 1 for the plain head),
// written twice through TMA bulk tensor stores: row-major G8 [T, C] (the
// K-major A operand of dH = G W_c) and transposed G8t [C, T] (the K-major A
// operand of dW_c = G^T H). Each 64-column quarter is staged as a 128 x 64-byte
// tile in the 64-byte-swizzled layout of G8's map and a 64 x 128-byte tile in
// the 128-byte-swizzled layout of G8t's map (16 KB per column group).
template <bool CAP>
struct EpiG8T {
  static constexpr int kStageBytes = 4 * 16384;  // two 16 KB buffers per column group
  static constexpr bool kKeepOperands = true;
  struct Params {
    CUtensorMap tmG;   // G8 [T, C] (row pitch ldG bytes), box 64 x 128, 64-byte swizzle
    CUtensorMap tmGt;  // G8t [C, T] (row pitch ldT bytes), box 128 x 64, 128-byte swizzle
    int T, C;
    const int32_t* slot;
    const float* lse;
    int* status;
    const float* amax;  // logits = accumulator * e4m3_logit_scale(amax)
    HeadCap head;       // used when CAP
    int g8e;            // G8 = e5m2(2^g8e (P - Y) dz/ds)
  };
  // the plain head folds the e4m3 scale into the exponent's constant; the
  // capped head needs the logit itself
  __device__ static void begin(const Params& p, EpiState& es) {
    es.f0 = e4m3_logit_scale(p.amax) * (CAP ? 1.f : kLog2e);
  }
  __device__ static void finish(const Params&, EpiState& es) {
    if ((es.ep_tid & 127) == 0) bulk_wait<0>();
  }
  template <int BN, int NCG>
  __device__ static void apply(const Params& p, int mt, int nt, int row, uint32_t taddr,
                               EpiState& es, int cg) {
    static_assert(NCG == 1 || NCG == 2, "column groups");
    const int bar = 1 + 2 * cg;
    const bool leader = (es.ep_tid & 127) == 0;
    const int t = mt * BM + row;
    const bool valid = t < p.T;
    const int sl = valid ? __ldg(p.slot + t) : -1;
    if (valid && nt == 0 && static_cast<unsigned>(sl) >= static_cast<unsigned>(p.C))
      set_status(p.status, SS_ERR_INDEX);
    const float k2 = es.f0;  // plain: scale * log2e; capped: the logit scale
    HeadCap hz = p.head;     // capped: the logit scale folded into the exponent constant
    if constexpr (CAP) hz.k1 *= k2;
    // 2^g8e exp(z - lse) = 2^(z log2e - (lse log2e - g8e))
    const float off2 = valid ? fmaf(__ldg(p.lse + t), kLog2e, -static_cast<float>(p.g8e)) : 0.f;
    const float one_hot = exp2i(p.g8e);
    const int j0 = nt * BN;
    const int ncols = min(BN, p.C - j0);
    // this thread's byte in row jj of the transposed tile: 16-byte chunk
    // (row / 16) ^ (jj % 8) of the 128-byte row, byte row % 16
    uint32_t toff[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
      toff[k] = ((static_cast<uint32_t>(row >> 4) ^ static_cast<uint32_t>(k)) << 4) |
                static_cast<uint32_t>(row & 15);
    const uint32_t r64 = static_cast<uint32_t>((row >> 1) & 3);  // 64-byte swizzle of this row
#pragma unroll 1
    for (int q = cg * (BN / 64) / NCG; q < (cg + 1) * (BN / 64) / NCG; ++q) {
      const int qc = q * 64;
      if (qc >= ncols) break;  // uniform: depends on the tile only
      constexpr uint32_t kBufs = kStageBytes / 16384 / NCG;
      const uint32_t buf = es.stage + static_cast<uint32_t>(cg) * 16384u * kBufs +
                           (es.rounds % kBufs) * 16384u;
      const uint32_t rbuf = buf, tbuf = buf + 8192u;
      if (es.rounds >= kBufs && leader) bulk_wait_read<static_cast<int>(kBufs) - 1>();
      named_bar_sync(bar, 128);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int jc = qc + 32 * h;
        if (jc >= ncols) break;
        uint32_t r[32];
        tmem_ld32(taddr + jc, r);
        tmem_ld_wait();
        const int off = sl - j0 - jc;
        float g[32];
        if constexpr (CAP) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float z = head_z(__uint_as_float(r[i]), hz);
            const float y = i == off ? one_hot : 0.f;
            g[i] = (ex2_approx(fmaf(z, kLog2e, -off2)) - y) * head_dz(z, p.head);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) g[i] = ex2_approx(fmaf(__uint_as_float(r[i]), k2, -off2));
          if (__any_sync(0xffffffffu, static_cast<unsigned>(off) < 32u)) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (i == off) g[i] -= one_hot;
          }
        }
        uint16_t pr[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) pr[i] = e5m2x2(g[2 * i], g[2 * i + 1]);
        // row-major tile: 32 bytes = 16-byte chunks 2h, 2h + 1 of this row
#pragma unroll
        for (int v = 0; v < 2; ++v) {
          const uint32_t c = static_cast<uint32_t>(2 * h + v);
          const uint16_t* w = pr + 8 * v;
          st_shared_v4(rbuf + static_cast<uint32_t>(row) * 64u + ((c ^ r64) << 4),
                       w[0] | (static_cast<uint32_t>(w[1]) << 16),
                       w[2] | (static_cast<uint32_t>(w[3]) << 16),
                       w[4] | (static_cast<uint32_t>(w[5]) << 16),
                       w[6] | (static_cast<uint32_t>(w[7]) << 16));
        }
        // transposed tile: column jj = 32h + i is row jj of it
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const uint16_t b = (i & 1) ? static_cast<uint16_t>(pr[i >> 1] >> 8) : pr[i >> 1];
          st_shared_u8(tbuf + static_cast<uint32_t>(32 * h + i) * 128u + toff[i & 7], b);
        }
      }
      fence_proxy_async_smem();
      named_bar_sync(bar, 128);
      if (leader) {
        const uint64_t pol = l2_evict_first();
        tma_store_2d_hint(&p.tmG, rbuf, j0 + qc, mt * BM, pol);
        tma_store_2d_hint(&p.tmGt, tbuf, mt * BM, j0 + qc, pol);
        bulk_commit();
      }
      ++es.rounds;
    }
  }
};

using EpiG8 = EpiG8T<false>;

// Backward, step 2: dH tile -> bf16 (column group cg of NCG). F8G: the
// accumulator is of e5m2 G and e4m3 W_c, times fp8_grad_alpha.
template <bool F8G = false>
struct EpiDhT {
  static constexpr int kStageBytes = 0;
  static constexpr bool kKeepOperands = false;
  struct Params {
    int T, D;
    uint16_t* dH;
    float scale;         // used when F8G
    const float* amax;   // used when F8G: max |W_c|
    int g8e;             // used when F8G: G8's power of two
    const float* rowfac;  // bf16: null, or a factor per row of dH (the accumulator times it)
  };
  __device__ static void begin(const Params& p, EpiState& es) {
    if constexpr (F8G) es.f0 = fp8_grad_alpha(p.scale, p.g8e, p.amax);
  }
  __device__ static void finish(const Params&, EpiState&) {}
  template <int BN, int NCG>
  __device__ static void apply(const Params& p, int mt, int nt, int row, uint32_t taddr,
                               EpiState& es, int cg) {
    constexpr int CPG = BN / 32 / NCG;
    const int t = mt * BM + row;
    const bool valid = t < p.T;
    const int n0 = nt * BN + cg * CPG * 32;
    const int ncols = min(CPG * 32, p.D - n0);
    if (ncols <= 0) return;
    uint16_t* drow = p.dH + static_cast<size_t>(valid ? t : 0) * p.D + n0;
    float al = 1.f;
    if constexpr (F8G) al = es.f0;
    const bool rf = !F8G && p.rowfac != nullptr;  // uniform
    if (rf) al = valid ? __ldg(p.rowfac + t) : 0.f;
    for_tmem_chunks<CPG>(taddr, cg * CPG, [&](const uint32_t(&r)[32], int i) {
      const int jc = i * 32;
      if (jc >= ncols || !valid) return;
      uint4* dst = reinterpret_cast<uint4*>(drow + jc);
      auto x = [&](int k) {
        return (F8G || rf) ? __uint_as_float(r[k]) * al : __uint_as_float(r[k]);
      };
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const uint32_t q0 = pack_bf16x2(x(8 * v + 0), x(8 * v + 1));
        const uint32_t q1 = pack_bf16x2(x(8 * v + 2), x(8 * v + 3));
        const uint32_t q2 = pack_bf16x2(x(8 * v + 4), x(8 * v + 5));
        const uint32_t q3 = pack_bf16x2(x(8 * v + 6), x(8 * v + 7));
        dst[v] = make_uint4(q0, q1, q2, q3);
      }
    });
  }
};
using EpiDh = EpiDhT<false>;

// Backward, step 3: dW_c tile scattered into the owning rows dW[cand[j]]
// (= or +=), column group cg of NCG. Candidate ids are distinct, so no two
// threads write one row. F8G: as for EpiDhT, with H's e4m3 exponent.
template <bool F8G = false>
struct EpiDwT {
  static constexpr int kStageBytes = 0;
  static constexpr bool kKeepOperands = false;
  struct Params {
    int C, D, V, accumulate;
    const int32_t* cand;
    float* dW;
    int* status;
    float scale;         // F8G: the gradient's scale; bf16 with out_scale: the factor
    const float* amax;   // used when F8G: max |H|
    int g8e;             // used when F8G: G8's power of two
    int out_scale;       // bf16: 1 if the accumulator is multiplied by `scale`
  };
  __device__ static void begin(const Params& p, EpiState& es) {
    if constexpr (F8G) es.f0 = fp8_grad_alpha(p.scale, p.g8e, p.amax);
    else es.f0 = p.out_scale ? p.scale : 1.f;
  }
  __device__ static void finish(const Params&, EpiState&) {}
  template <int BN, int NCG>
  __device__ static void apply(const Params& p, int mt, int nt, int row, uint32_t taddr,
                               EpiState& es, int cg) {
    constexpr int CPG = BN / 32 / NCG;
    const int j = mt * BM + row;
    bool valid = j < p.C;
    const int v = valid ? __ldg(p.cand + j) : 0;
    if (valid && static_cast<unsigned>(v) >= static_cast<unsigned>(p.V)) {
      if (cg == 0) set_status(p.status, SS_ERR_INDEX);
      valid = false;
    }
    const int n0 = nt * BN + cg * CPG * 32;
    const int ncols = min(CPG * 32, p.D - n0);
    if (ncols <= 0) return;
    float* drow = p.dW + static_cast<size_t>(valid ? v : 0) * p.D + n0;
    const float al = es.f0;
    const bool sc = F8G || p.out_scale;  // uniform
    for_tmem_chunks<CPG>(taddr, cg * CPG, [&](const uint32_t(&r)[32], int i) {
      const int jc = i * 32;
      if (jc >= ncols || !valid) return;
      float4* dst = reinterpret_cast<float4*>(drow + jc);
      auto x = [&](int k) { return sc ? __uint_as_float(r[k]) * al : __uint_as_float(r[k]); };
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        float4 o = make_float4(x(4 * k), x(4 * k + 1), x(4 * k + 2), x(4 * k + 3));
        if (p.accumulate) {
          const float4 old = dst[k];
          o.x += old.x;
          o.y += old.y;
          o.z += old.z;
          o.w += old.w;
        }
        dst[k] = o;
      }
    });
  }
};
using EpiDw = EpiDwT<false>;

// -------------------------------------------------------------------- kernel

// F8: e4m3 operands (kind::f8f6f4, K-major only): the same 128-byte
// swizzled rows then hold 128 elements, so a k-block covers 128 of K.
template <int BN, int STAGES, bool A_MN, bool B_MN, class Epi, int EPI_WARPS = 4, bool F8 = false>
__global__ void __launch_bounds__(64 + 32 * EPI_WARPS, 1)
    k_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
           GemmShape shp, const __grid_constant__ typename Epi::Params ep, int* status) {
  if (shp.late_wait) pdl_launch_dependents();
  else pdl_enter();
  static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "BN");
  static_assert(STAGES >= 2 && STAGES <= 8, "STAGES");
  static_assert(EPI_WARPS == 4 || EPI_WARPS == 8, "EPI_WARPS");
  static_assert(!F8 || (!A_MN && !B_MN), "e4m3 operands are K-major");
  constexpr int KB = F8 ? 2 * BK : BK;  // elements of K per k-block
  constexpr int NCG = EPI_WARPS / 4;
  using L = GemmSmem<BN, STAGES, Epi::kStageBytes>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_go;

  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  GemmCtrl* ctrl = reinterpret_cast<GemmCtrl*>(smem + L::CTRL_OFFSET);
  const uint32_t tiles = smem_u32(smem);
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  // An earlier error of this batch, or a gate that is shut: do nothing
  // (decided once for the CTA).
  if (threadIdx.x == 0)
    s_go = read_status(status) == 0 && (shp.gate == nullptr || read_status(shp.gate) != 0);
  __syncthreads();
  if (!s_go) return;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&ctrl->full[s], 1);
      mbar_init(&ctrl->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&ctrl->tfull[b], 1);
      mbar_init(&ctrl->tempty[b], EPI_WARPS * 32);
    }
    mbar_init(&ctrl->drain, 1);
    ctrl->abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_map(&tmA);
    tma_prefetch_map(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(&ctrl->tmem_base, 2 * BN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ctrl->tmem_base;
  volatile int* abort_flag = &ctrl->abort_flag;
  const int n_cols = shp.n_tiles - shp.n_begin;  // column tiles per row block
  const int num_units = shp.m_tiles * n_cols;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0, issued = 0, issued_ph = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < num_units; u += gridDim.x) {
        int mt, nt;
        unit_tile(shp, u, mt, nt);
        for (int kb = 0; kb < shp.k_blocks; ++kb) {
          if (!mbar_wait(&ctrl->empty[s], ph ^ 1u, abort_flag, status)) {
            ok = false;
            break;
          }
          uint64_t* fb = &ctrl->full[s];
          mbar_arrive_expect_tx(fb, L::STAGE_BYTES);
          const uint32_t a_dst = tiles + s * L::STAGE_BYTES;
          const uint32_t b_dst = a_dst + L::A_BYTES;
          if constexpr (Epi::kKeepOperands) {
            static_assert(!A_MN && !B_MN, "cache-hinted loads are K-major");
            const uint64_t pol = l2_evict_last();
            tma_load_2d_hint(a_dst, &tmA, fb, kb * KB, mt * BM, pol);
            tma_load_2d_hint(b_dst, &tmB, fb, kb * KB, nt * BN, pol);
          } else {
            if (A_MN) {
#pragma unroll
              for (int i = 0; i < BM / 64; ++i)
                tma_load_2d(a_dst + i * 8192, &tmA, fb, mt * BM + 64 * i, kb * BK);
            } else {
              tma_load_2d(a_dst, &tmA, fb, kb * KB, mt * BM);
            }
            if (B_MN) {
#pragma unroll
              for (int i = 0; i < BN / 64; ++i)
                tma_load_2d(b_dst + i * 8192, &tmB, fb, nt * BN + 64 * i, kb * BK);
            } else {
              tma_load_2d(b_dst, &tmB, fb, kb * KB, nt * BN);
            }
          }
          issued |= 1u << s;
          issued_ph = (issued_ph & ~(1u << s)) | (ph << s);
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      // Every issued copy must land before the CTA may exit.
      for (int i = 0; i < STAGES; ++i)
        if ((issued >> i) & 1u) mbar_drain(&ctrl->full[i], (issued_ph >> i) & 1u, status);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = F8 ? idesc_e4m3_f32(BM, BN) : idesc_bf16_f32(BM, BN, A_MN, B_MN);
      int s = 0, b = 0;
      uint32_t ph = 0, aph = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < num_units; u += gridDim.x) {
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
            if constexpr (F8) mma_e4m3(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
            else mma_bf16(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
          }
          mma_commit(&ctrl->empty[s]);
          if (++s == STAGES) {
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
      // Every issued MMA must finish before TMEM is released.
      mma_commit(&ctrl->drain);
      mbar_drain(&ctrl->drain, 0, status);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;         // TMEM lane quarter this warp may access
    const int cg = (warp - 2) / 4;  // column group
    const int row = q * 32 + lane;
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    EpiState es{tiles + L::EPI_OFFSET, static_cast<int>(threadIdx.x) - 64, 0u, 0.f};
    if (shp.late_wait) pdl_wait();
    Epi::begin(ep, es);
    int b = 0;
    uint32_t aph = 0;
    for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
      const bool ok = mbar_wait(&ctrl->tfull[b], aph, abort_flag, status);
      bool go = __all_sync(0xffffffffu, ok);
      if constexpr (Epi::kStageBytes > 0) {
        // This epilogue synchronises its warps with named barriers, so they
        // must leave the loop together: vote every tile.
        if (lane == 0) ctrl->vote[(u / gridDim.x) & 1][warp - 2] = go ? 1 : 0;
        named_bar_sync(2, 32 * EPI_WARPS);
        const int* v = ctrl->vote[(u / gridDim.x) & 1];
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
        mbar_arrive(&ctrl->tempty[b]);
      };
      const uint32_t acc = lane_addr + static_cast<uint32_t>(b * BN);
      if constexpr (EpiSelfRelease<Epi>::value) {
        Epi::template apply<BN, NCG>(ep, mt, nt, row, acc, es, cg, release);
      } else {
        Epi::template apply<BN, NCG>(ep, mt, nt, row, acc, es, cg);
        release();
      }
      if (++b == 2) {
        b = 0;
        aph ^= 1u;
      }
    }
    Epi::finish(ep, es);  // outstanding stores from shared memory complete before exit
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 2 * BN);
  }
}

// Host-side launcher: grid = min(units, SMs), one CTA per SM.
template <int BN, int STAGES, bool A_MN, bool B_MN, class Epi, int EPI_WARPS = 4, bool F8 = false>
cudaError_t launch_gemm(const CUtensorMap& tA, const CUtensorMap& tB, GemmShape shp,
                        const typename Epi::Params& ep, int* status, int num_sms,
                        cudaStream_t stream) {
  auto kern = k_gemm<BN, STAGES, A_MN, B_MN, Epi, EPI_WARPS, F8>;
  constexpr int smem = GemmSmem<BN, STAGES, Epi::kStageBytes>::TOTAL;
  const int units = shp.m_tiles * (shp.n_tiles - shp.n_begin);
  if (units <= 0) return cudaSuccess;
  if (shp.gate != nullptr && shp.late_wait) return cudaErrorInvalidValue;  // the gate needs the wait
  const int grid = units < num_sms ? units : num_sms;
  return launch_pdl(kern, dim3(grid), dim3(64 + 32 * EPI_WARPS), smem, stream, tA, tB, shp, ep,
                    status);
}

}  // namespace ss
