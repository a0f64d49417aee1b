// ss_candidates.cu -- build the shared candidate set of one batch on the GPU.
//
// The pages' method scores every token that occurs in the batch and fills the
// rest of a fixed-size candidate set with other vocabulary ids ("KellerJordan/
// modded-nanogpt" README, technique list: one candidate set shared by the
// batch; the record tweet quoted on the airebao page: in-batch tokens are
// always scored, absent ones only sometimes). Here:
//   cand[0, U)   = the distinct targets, ascending;
//   cand[U, C)   = the C - U non-target ids with the smallest keys
//                  key(v) = hash(seed, v) * 2^32 + v, in ascending id order,
//                  hash(seed, v) = high 32 bits of SplitMix64 output number v
//                  (Steele, Lea and Flood, OOPSLA 2014): a uniform sample
//                  without replacement when the hash behaves as random;
//   slot[t]      = rank of targets[t] among the distinct targets.
//
// One thread-block cluster of 8 CTAs x 1024 threads. CTA r owns a contiguous
// slice of the vocabulary bitmap in its shared memory; peers reach it through
// distributed shared memory (DSMEM):
//   1. mark targets in a CTA-local bitmap of the whole vocabulary (range-
//      checked shared-memory atomics), then OR the eight local bitmaps into
//      each owner's slice;
//   2. popcounts + block scans + cluster prefix -> U, per-word target prefix;
//   3. radix-select the (C-U)-th smallest key among non-targets with 12-bit
//      digits over the 32-bit hash: per-CTA histograms, reduce-scattered over
//      the cluster (CTA r sums one eighth of the bins); as soon as the
//      selected bin holds at most kTieCap ids they are
//      ranked exactly by (hash, id); at the last digit, equal hashes are
//      taken in id order. Selected ids go into a second bitmap;
//   4. compaction: popcount scans over the two bitmaps -> cand;
//   5. slot[t] = word prefix + popcount of the lower bits of its word, from
//      local copies of the whole bitmap and prefix array.
// The whole vocabulary is hashed twice in the common case.
#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ss.h"
#include "ss_internal.h"
#include "ss_ptx.cuh"

namespace cg = cooperative_groups;

namespace ss {

namespace {

constexpr int kClusterCtas = 8;
constexpr int kCandThreads = 1024;
constexpr int kWarps = kCandThreads / 32;
constexpr int kBins = 4096;   // 12-bit digits (the last digit has 8 bits)
#ifndef SS_TIE_CAP
#define SS_TIE_CAP 1024
#endif
constexpr int kTieCap = SS_TIE_CAP;  // ranked exactly when the selected bin is this small
// tie-list entries allocated: at least 2 and even, so that the arrays after it
// stay 16-byte aligned for vector access
constexpr int kTieSlots = 2 * (((kTieCap > 2 ? kTieCap : 2) + 1) & ~1);  // own list + all lists

__device__ __forceinline__ uint32_t negative_hash(uint64_t seed, uint32_t v) {
  uint64_t z = seed + (static_cast<uint64_t>(v) + 1ull) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  z ^= z >> 31;
  return static_cast<uint32_t>(z >> 32);
}

// Exclusive scan of one value per thread over the block; *total = block sum.
__device__ __forceinline__ uint32_t block_scan(uint32_t x, uint32_t* ws, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) ws[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const uint32_t w = ws[lane];
    uint32_t wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    ws[lane] = wi - w;
    if (lane == 31) ws[32] = wi;
  }
  __syncthreads();
  const uint32_t r = ws[warp] + incl - x;
  *total = ws[32];
  __syncthreads();
  return r;
}

// Warp 0: lane q < 8 fetches value q of the cluster (one DSMEM load each, in
// parallel); returns (sum over q < r, total) on every lane of warp 0.
template <class F>
__device__ __forceinline__ void cluster_prefix(F&& fetch, int r, uint32_t* before, uint32_t* total) {
  const int lane = threadIdx.x & 31;
  const uint32_t x = lane < kClusterCtas ? fetch(lane) : 0u;
  uint32_t incl = x;
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  *total = __shfl_sync(0xffffffffu, incl, kClusterCtas - 1);
  *before = r > 0 ? __shfl_sync(0xffffffffu, incl, r - 1) : 0u;
}

struct Shared {
  uint32_t scan[33];
  int err;
  uint32_t U_r, S_r, E_r;     // this CTA's targets, selected negatives, final-digit ties
  uint32_t ntie;              // entries in this CTA's tie list
  uint32_t slice_sum;         // sum of this CTA's slice of the cluster histogram
  uint32_t b, rem, cnt;       // selected bin, remaining rank inside it, its size
  uint32_t U, Uoff, Soff, Eoff, any_err, s_slice, s_rem;  // broadcast values
};

// All peer scalars are read by one thread and broadcast through shared memory:
// distributed shared memory is limited by its request rate, so no phase lets
// every thread of a CTA fetch the same remote word.
__global__ void __cluster_dims__(kClusterCtas, 1, 1) __launch_bounds__(kCandThreads, 1)
    k_build_candidates(const int32_t* __restrict__ targets, int T, int V, int C, uint64_t seed,
                       int32_t* __restrict__ cand, int32_t* __restrict__ slot, int* hdr, int wpc) {
  pdl_enter();
  cg::cluster_group cluster = cg::this_cluster();
  const int r = static_cast<int>(cluster.block_rank());
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  extern __shared__ __align__(16) uint32_t dyn[];
  __shared__ Shared sh;
  const int nW = (V + 31) >> 5;
  const int nWp = (nW + 3) & ~3;   // padded to whole uint4
  uint32_t* bm = dyn;              // [wpc] targets (this CTA's slice); wpc % 4 == 0
  uint32_t* sel = bm + wpc;        // [wpc] selected negatives
  uint32_t* eqb = sel + wpc;       // [wpc] final-digit ties
  uint32_t* wpre = eqb + wpc;      // [wpc] targets in all words before this one
  uint32_t* hist = wpre + wpc;     // [kBins] this CTA's histogram
  uint32_t* hsl = hist + kBins;    // [kBins / 8] cluster totals of this CTA's slice of bins
  uint64_t* tie = reinterpret_cast<uint64_t*>(hsl + kBins / kClusterCtas);  // [kTieCap]
  uint32_t* local = reinterpret_cast<uint32_t*>(tie + kTieSlots);  // [nWp]
  uint32_t* fwpre = local + nWp;   // [nWp] word prefixes of the whole vocabulary (for slots)

  const int w0 = r * wpc;
  const int nw = max(0, min(wpc, nW - w0));  // words owned by this CTA
  if (r == 0 && tid == 0) hdr[0] = 0;        // a new batch: clear the status word
  for (int i = tid; i < wpc; i += kCandThreads) sel[i] = eqb[i] = 0u;
  for (int i = tid; i < nWp; i += kCandThreads) local[i] = 0u;
  if (tid == 0) {
    sh.err = 0;
    sh.ntie = 0;
  }
  __syncthreads();

  // 1. mark this CTA's share of the targets in a CTA-local bitmap of the whole
  //    vocabulary (shared-memory atomics, skipped when the bit is already set)
  for (int t = r * kCandThreads + tid; t < T; t += kClusterCtas * kCandThreads) {
    const int v = __ldg(targets + t);
    if (static_cast<unsigned>(v) >= static_cast<unsigned>(V)) {
      sh.err = 1;
      continue;
    }
    const uint32_t bit = 1u << (v & 31);
    if (!(local[v >> 5] & bit)) atomicOr(&local[v >> 5], bit);
  }
  cluster.sync();  // S1: local bitmaps complete
  // this CTA's slice of the union bitmap = OR of the eight local bitmaps
  for (int i = 4 * tid; i < wpc; i += 4 * kCandThreads) {
    uint4 o = make_uint4(0u, 0u, 0u, 0u);
    if (w0 + i < nWp) {
#pragma unroll
      for (int q = 0; q < kClusterCtas; ++q) {
        const uint4 x = *reinterpret_cast<const uint4*>(cluster.map_shared_rank(local, q) + w0 + i);
        o.x |= x.x;
        o.y |= x.y;
        o.z |= x.z;
        o.w |= x.w;
      }
    }
    *reinterpret_cast<uint4*>(bm + i) = o;
  }
  if (warp == 0) {
    uint32_t before, total;
    cluster_prefix([&](int q) { return static_cast<uint32_t>(cluster.map_shared_rank(&sh, q)->err); },
                   r, &before, &total);
    if (lane == 0) sh.any_err = total;
  }
  __syncthreads();
  if (sh.any_err) {
    if (r == 0 && tid == 0) {
      set_status(hdr, SS_ERR_TARGET_RANGE);
      hdr[1] = -1;
    }
    cluster.sync();  // no CTA exits while a peer may still read its shared memory
    return;
  }

  // 2. per-CTA target count (contiguous word chunk per thread) and the
  //    first-digit histogram of the non-targets' hashes; one cluster barrier
  const int wpt = (wpc + kCandThreads - 1) / kCandThreads;
  const int c0 = min(tid * wpt, nw), c1 = min(c0 + wpt, nw);
  uint32_t tcnt = 0;
  for (int i = c0; i < c1; ++i) tcnt += __popc(bm[i]);
  uint32_t U_r;
  const uint32_t t_excl = block_scan(tcnt, sh.scan, &U_r);
  if (tid == 0) sh.U_r = U_r;
  for (int i = tid; i < kBins; i += kCandThreads) hist[i] = 0u;
  __syncthreads();
  for (int i = warp; i < nw; i += kWarps) {
    const int v = (w0 + i) * 32 + lane;
    if (v < V && !((bm[i] >> lane) & 1u))
      atomicAdd(&hist[negative_hash(seed, static_cast<uint32_t>(v)) >> 20], 1u);
  }
  cluster.sync();  // S2: target counts and histograms complete
  if (warp == 0) {
    uint32_t before, total;
    cluster_prefix([&](int q) { return cluster.map_shared_rank(&sh, q)->U_r; }, r, &before, &total);
    if (lane == 0) {
      sh.U = total;
      sh.Uoff = before;
    }
  }
  __syncthreads();
  const uint32_t U = sh.U, Uoff = sh.Uoff;
  {
    uint32_t run = Uoff + t_excl;
    for (int i = c0; i < c1; ++i) {
      wpre[i] = run;
      run += __popc(bm[i]);
    }
  }
  if (static_cast<int>(U) > C) {
    if (r == 0 && tid == 0) {
      set_status(hdr, SS_ERR_CAPACITY);
      hdr[1] = static_cast<int>(U);
    }
    cluster.sync();
    return;
  }
  const uint32_t k = static_cast<uint32_t>(C) - U;
  const uint32_t n_non = static_cast<uint32_t>(V) - U;

  // 3. select the k non-targets with the smallest keys
  if (k == n_non) {
    for (int i = tid; i < nw; i += kCandThreads) {
      const int vbase = (w0 + i) * 32;
      const uint32_t valid = (V - vbase >= 32) ? 0xffffffffu : ((1u << (V - vbase)) - 1u);
      sel[i] = ~bm[i] & valid;
    }
  } else if (k > 0) {
    uint32_t prefix = 0, mask = 0, rem = k;
    int level = 0;
    for (;; ++level) {
      const int shift = level == 0 ? 20 : (level == 1 ? 8 : 0);
      const int nb = level == 2 ? 256 : kBins;
      const bool last = level == 2;
      if (level > 0) {  // level 0's histogram was built before the U exchange
        for (int i = tid; i < nb; i += kCandThreads) hist[i] = 0u;
        __syncthreads();
        for (int i = warp; i < nw; i += kWarps) {
          const int v = (w0 + i) * 32 + lane;
          if (v < V && !((bm[i] >> lane) & 1u)) {
            const uint32_t h = negative_hash(seed, static_cast<uint32_t>(v));
            if ((h & mask) == prefix) atomicAdd(&hist[(h >> shift) & (nb - 1)], 1u);
          }
        }
        cluster.sync();
      }
      // reduce-scatter: CTA r sums bins [r*nb/8, (r+1)*nb/8) over the cluster
      const int sl = nb / kClusterCtas;  // 512 or 32 bins, a multiple of 4
      uint32_t part = 0;
      if (4 * tid < sl) {
        uint4 s4 = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int q = 0; q < kClusterCtas; ++q) {
          const uint4 x =
              *reinterpret_cast<const uint4*>(cluster.map_shared_rank(hist, q) + r * sl + 4 * tid);
          s4.x += x.x;
          s4.y += x.y;
          s4.z += x.z;
          s4.w += x.w;
        }
        *reinterpret_cast<uint4*>(hsl + 4 * tid) = s4;
        part = s4.x + s4.y + s4.z + s4.w;
      }
      uint32_t ssum;
      (void)block_scan(part, sh.scan, &ssum);
      if (tid == 0) sh.slice_sum = ssum;
      cluster.sync();  // slice totals complete (and peers are done with our histogram)
      // every CTA: which slice holds rank rem, then which bin inside it
      if (warp == 0) {
        // lane q < 8 holds slice q's total; find the slice where rank rem falls
        const uint32_t x = lane < kClusterCtas ? cluster.map_shared_rank(&sh, lane)->slice_sum : 0u;
        uint32_t incl = x;
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const unsigned hit = __ballot_sync(0xffffffffu, lane < kClusterCtas && rem <= incl);
        const int s = hit ? __ffs(hit) - 1 : kClusterCtas - 1;
        const uint32_t cum = __shfl_sync(0xffffffffu, incl - x, s);
        if (lane == 0) {
          sh.s_slice = static_cast<uint32_t>(s);
          sh.s_rem = rem - cum;
        }
      }
      __syncthreads();
      const uint32_t s = sh.s_slice, srem = sh.s_rem;
      uint32_t b4[4] = {0u, 0u, 0u, 0u};
      uint32_t psum = 0;
      if (4 * tid < sl) {
        const uint4 x = *reinterpret_cast<const uint4*>(cluster.map_shared_rank(hsl, s) + 4 * tid);
        b4[0] = x.x;
        b4[1] = x.y;
        b4[2] = x.z;
        b4[3] = x.w;
        psum = x.x + x.y + x.z + x.w;
      }
      uint32_t tot;
      const uint32_t before = block_scan(psum, sh.scan, &tot);
      if (4 * tid < sl && before < srem && srem <= before + psum) {
        uint32_t cum = before;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (srem <= cum + b4[j]) {
            sh.b = s * sl + static_cast<uint32_t>(4 * tid + j);
            sh.rem = srem - cum;
            sh.cnt = b4[j];
            break;
          }
          cum += b4[j];
        }
      }
      __syncthreads();
      const uint32_t b = sh.b, cnt = sh.cnt;
      const bool collect = last || cnt <= static_cast<uint32_t>(kTieCap);
      // another level rebuilds the histograms: peers must be done reading hsl
      if (!collect) cluster.sync();
      for (int i = warp; i < nw; i += kWarps) {
        const int v = (w0 + i) * 32 + lane;
        bool below = false, in_bin = false;
        uint32_t h = 0;
        if (v < V && !((bm[i] >> lane) & 1u)) {
          h = negative_hash(seed, static_cast<uint32_t>(v));
          if ((h & mask) == prefix) {
            const uint32_t d = (h >> shift) & static_cast<uint32_t>(nb - 1);
            below = d < b;
            in_bin = d == b;
          }
        }
        const uint32_t bw = __ballot_sync(0xffffffffu, below);
        if (lane == 0 && bw) sel[i] |= bw;
        if (collect) {
          if (last) {
            const uint32_t ew = __ballot_sync(0xffffffffu, in_bin);
            if (lane == 0) eqb[i] = ew;
          } else if (in_bin) {
            const uint32_t at = atomicAdd(&sh.ntie, 1u);
            tie[at] = (static_cast<uint64_t>(h) << 32) | static_cast<uint32_t>(v);
          }
        }
      }
      prefix |= b << shift;
      mask |= static_cast<uint32_t>(nb - 1) << shift;
      rem = sh.rem;
      if (collect) break;
    }
    if (level < 2) {
      // The selected bin is small: copy every CTA's list of its ids into
      // local shared memory (after this CTA's own list), then rank this
      // CTA's ids exactly by (hash, id).
      cluster.sync();
      uint64_t* all = tie + sh.ntie;  // room: the bin holds at most kTieCap ids in total
      __shared__ uint32_t s_off[kClusterCtas + 1];
      if (warp == 0) {
        const uint32_t n = lane < kClusterCtas ? cluster.map_shared_rank(&sh, lane)->ntie : 0u;
        uint32_t incl = n;
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        if (lane < kClusterCtas) s_off[lane] = incl - n;
        if (lane == kClusterCtas - 1) s_off[kClusterCtas] = incl;
      }
      __syncthreads();
      const uint32_t ntot = s_off[kClusterCtas];
      for (uint32_t i = tid; i < ntot; i += kCandThreads) {
        int q = 0;
        while (q + 1 < kClusterCtas && s_off[q + 1] <= i) ++q;
        all[i] = cluster.map_shared_rank(tie, q)[i - s_off[q]];
      }
      __syncthreads();
      const uint32_t mine = sh.ntie;
      for (uint32_t i = tid; i < mine; i += kCandThreads) {
        const uint64_t key = tie[i];
        uint32_t rank = 0;
        for (uint32_t j = 0; j < ntot; ++j) rank += all[j] < key;
        if (rank < rem) {
          const int v = static_cast<int>(key & 0xffffffffu);
          atomicOr(&sel[(v >> 5) - w0], 1u << (v & 31));
        }
      }
    } else {
      // all 32 hash bits equal: take the first `rem` of them in id order
      uint32_t ecnt = 0;
      for (int i = c0; i < c1; ++i) ecnt += __popc(eqb[i]);
      uint32_t E_r;
      const uint32_t e_excl = block_scan(ecnt, sh.scan, &E_r);
      if (tid == 0) sh.E_r = E_r;
      cluster.sync();
      if (warp == 0) {
        uint32_t before, total;
        cluster_prefix([&](int q) { return cluster.map_shared_rank(&sh, q)->E_r; }, r, &before,
                       &total);
        if (lane == 0) sh.Eoff = before;
      }
      __syncthreads();
      uint32_t e = sh.Eoff + e_excl;
      for (int i = c0; i < c1; ++i) {
        uint32_t bits = eqb[i];
        while (bits) {
          const int j = __ffs(bits) - 1;
          bits &= bits - 1;
          if (e < rem) sel[i] |= 1u << j;
          ++e;
        }
      }
    }
  }
  __syncthreads();

  // 4. compaction: targets into [0, U), selected negatives into [U, C)
  uint32_t scnt = 0;
  for (int i = c0; i < c1; ++i) scnt += __popc(sel[i]);
  uint32_t S_r;
  const uint32_t s_excl = block_scan(scnt, sh.scan, &S_r);
  if (tid == 0) sh.S_r = S_r;
  cluster.sync();  // S_r and every slice's word prefixes complete
  if (warp == 0) {
    uint32_t before, total;
    cluster_prefix([&](int q) { return cluster.map_shared_rank(&sh, q)->S_r; }, r, &before, &total);
    if (lane == 0) sh.Soff = before;
  }
  // replicate the whole vocabulary's bitmap and word prefixes for the slots
  // (`local` is free: peers finished reading it before the second barrier)
  for (int i = 4 * tid; i < nWp; i += 4 * kCandThreads) {
    const int q = i / wpc;
    const int li = i - q * wpc;
    *reinterpret_cast<uint4*>(local + i) =
        *reinterpret_cast<const uint4*>(cluster.map_shared_rank(bm, q) + li);
    *reinterpret_cast<uint4*>(fwpre + i) =
        *reinterpret_cast<const uint4*>(cluster.map_shared_rank(wpre, q) + li);
  }
  __syncthreads();
  {
    uint32_t ti = Uoff + t_excl, si = U + sh.Soff + s_excl;
    for (int i = c0; i < c1; ++i) {
      const int vbase = (w0 + i) * 32;
      uint32_t tb = bm[i], sb = sel[i];
      while (tb) {
        cand[ti++] = vbase + __ffs(tb) - 1;
        tb &= tb - 1;
      }
      while (sb) {
        cand[si++] = vbase + __ffs(sb) - 1;
        sb &= sb - 1;
      }
    }
  }

  // 5. slots from the local copies
  for (int t = r * kCandThreads + tid; t < T; t += kClusterCtas * kCandThreads) {
    const int v = __ldg(targets + t);
    const int w = v >> 5;
    slot[t] = static_cast<int32_t>(fwpre[w] + __popc(local[w] & ((1u << (v & 31)) - 1u)));
  }
  if (r == 0 && tid == 0) hdr[1] = static_cast<int>(U);
  cluster.sync();  // keep every CTA's shared memory alive until all peers are done
}

// words of the bitmap per CTA, a multiple of 4 (whole uint4 vectors)
int words_per_cta(int64_t V) {
  const int64_t nW = (V + 31) / 32;
  const int64_t w = (nW + kClusterCtas - 1) / kClusterCtas;
  return static_cast<int>((w + 3) / 4 * 4);
}

}  // namespace

size_t build_candidates_smem_bytes(int64_t V) {
  const size_t nWp = static_cast<size_t>(((V + 31) / 32 + 3) / 4 * 4);
  return static_cast<size_t>(words_per_cta(V)) * 4 * sizeof(uint32_t) +
         (kBins + kBins / kClusterCtas) * sizeof(uint32_t) +
         kTieSlots * sizeof(uint64_t) + 2 * nWp * sizeof(uint32_t);
}

cudaError_t launch_build_candidates(const int32_t* targets, int T, int V, int C, uint64_t seed,
                                    int32_t* cand, int32_t* slot, int* hdr,
                                    cudaStream_t stream) {
  const size_t smem = build_candidates_smem_bytes(V);
  cudaError_t e = cudaFuncSetAttribute(k_build_candidates,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_pdl(k_build_candidates, dim3(kClusterCtas), dim3(kCandThreads), smem, stream, targets,
                    T, V, C, seed, cand, slot, hdr, words_per_cta(V));
}

}  // namespace ss
