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
// One thread-block cluster of 8 CTAs x 1024 threads. Every CTA ends up with a
// bitmap of all targets over the whole vocabulary in its own shared memory
// (marking all targets itself, or an eighth of them merged with the others'
// through distributed shared memory, DSMEM), so U, the word prefixes (for the
// compaction and the slots) and range errors need no further exchange. The
// non-targets are split in eight contiguous id slices, one per CTA, and the
// selection exchanges only histograms and tie lists:
//   1. mark (and merge); popcount scan of the whole bitmap -> U, prefixes;
//   2. radix-select the (C-U)-th smallest key among the non-targets, 8-bit
//      digits over the 32-bit hash: each CTA histograms its slice, every CTA
//      reads all eight histograms and finds the digit and, for each CTA, how
//      many of its ids fall below it; as soon as the selected bin holds at
//      most kTieCap ids, every CTA gathers all CTAs' lists of them and ranks
//      them exactly by (hash, id) with one more digit and a few comparisons;
//      at the last digit, equal hashes are taken in id order;
//   3. each CTA knows every CTA's selected count, hence its own output
//      offset; compaction of its slice into cand, slots of 1/8 of the tokens.
// Cluster barriers: two after a split marking, one per radix level, one
// before the tie exchange, and a split one whose wait is the kernel's last
// step (no CTA leaves while a peer may still read its shared memory).
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
constexpr int kBins = 256;  // 8-bit digits, four levels over the 32-bit hash
#ifndef SS_TIE_CAP
#define SS_TIE_CAP 512
#endif
constexpr int kTieCap = SS_TIE_CAP;  // ranked exactly when the selected bin is this small
constexpr int kTieSlots = 2 * (kTieCap > 1 ? kTieCap : 1);  // own list + all lists
static_assert(kBins + 2 * kTieCap <= kClusterCtas * kBins,
              "the tie ranking reuses the gathered histograms' shared memory");
// Up to this vocabulary size each CTA keeps its slice's hashes in shared
// memory for the passes after the first.
constexpr int kSmallV = 131072;

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

__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

struct Shared {
  uint32_t scan[33];
  int err, any_err;
  uint32_t ntie;                   // entries in this CTA's tie list
  uint32_t b, rem, cnt;            // selected bin, remaining rank inside it, its size
  uint32_t below[kClusterCtas];    // per CTA: its ids selected at earlier digits / below b
  uint32_t at_b[kClusterCtas];     // per CTA: its ids in the selected bin
  uint32_t tsel[kClusterCtas];     // per CTA: its ids taken from the selected bin
  uint32_t toff[kClusterCtas + 1]; // tie-list offsets in the gathered list
  uint32_t wsum[kBins / 32];        // per-warp sums of the bin scan
  uint32_t b2, rem2, m2;            // tie ranking: sub-bin, rank left in it, its size
};

// Words of the bitmap per CTA slice, a multiple of 4 (whole uint4 vectors).
__host__ __device__ inline int slice_words(int V) {
  const int nW = (V + 31) / 32;
  const int w = (nW + kClusterCtas - 1) / kClusterCtas;
  return (w + 3) / 4 * 4;
}

__global__ void __cluster_dims__(kClusterCtas, 1, 1) __launch_bounds__(kCandThreads, 1)
    k_build_candidates(const int32_t* __restrict__ targets, int T, int V, int C, uint64_t seed,
                       int32_t* __restrict__ cand, int32_t* __restrict__ slot, int* hdr) {
  pdl_enter();
  cg::cluster_group cluster = cg::this_cluster();
  const int r = static_cast<int>(cluster.block_rank());
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  extern __shared__ __align__(16) uint32_t dyn[];
  __shared__ Shared sh;
  const int nW = (V + 31) >> 5;
  const int nWp = (nW + 4) & ~3;   // room for the total after the last word
  const int wpc = slice_words(V);
  uint64_t* tie = reinterpret_cast<uint64_t*>(dyn);  // [kTieCap] own list, then all lists
  uint32_t* mine = reinterpret_cast<uint32_t*>(tie + kTieSlots);  // [nWp] this CTA's share
  uint32_t* full = mine + nWp;     // [nWp] all targets, whole vocabulary
  uint32_t* fpre = full + nWp;     // [nWp] targets in all words before word i; fpre[nW] = U
  uint32_t* sel = fpre + nWp;      // [wpc] selected negatives of this CTA's slice
  uint32_t* eqb = sel + wpc;       // [wpc] last-digit ties of the slice
  uint32_t* hist = eqb + wpc;      // [2][kBins] this CTA's histograms (alternating levels)
  uint32_t* gat = hist + 2 * kBins;  // [kClusterCtas][kBins] all CTAs' histograms of a level
  const bool small_v = V <= kSmallV;
  uint32_t* hs = gat + kClusterCtas * kBins;  // small_v: [wpc * 32] hashes of the slice

  const int w0 = r * wpc;
  const int nw = max(0, min(wpc, nW - w0));  // words of this CTA's slice
  if (r == 0 && tid == 0) hdr[0] = 0;        // a new batch: clear the status word
  for (int i = tid; i < wpc; i += kCandThreads) sel[i] = eqb[i] = 0u;
  for (int i = tid; i < nWp; i += kCandThreads) {
    mine[i] = 0u;
    full[i] = 0u;
  }
  if (tid < kClusterCtas) sh.below[tid] = sh.tsel[tid] = 0u;
  if (tid == 0) {
    sh.err = 0;
    sh.ntie = 0;
  }
  __syncthreads();

  // 1. the targets into a bitmap of the whole vocabulary (range-checked
  //    shared atomics, skipped when the bit is set already; targets read four
  //    at a time once aligned). Few targets per vocabulary word: every CTA
  //    marks all of them in `full` (no exchange; each CTA sees every range
  //    error). Otherwise each CTA marks an eighth in `mine`, then CTA q ORs
  //    slice q of the eight bitmaps (reduce-scatter) and every CTA copies the
  //    other slices from their owners (all-gather): a cluster barrier each.
  //    Distributed shared memory costs per request, so every CTA reading all
  //    eight whole bitmaps would be slower than both.
  const bool all_t = T <= 14 * nW;
  {
    uint32_t* bits = all_t ? full : mine;
    auto mark = [&](int v) {
      if (static_cast<unsigned>(v) >= static_cast<unsigned>(V)) {
        sh.err = 1;
        return;
      }
      const uint32_t bit = 1u << (v & 31);
      if (!(bits[v >> 5] & bit)) atomicOr(&bits[v >> 5], bit);
    };
    const int per = all_t ? T : (T + kClusterCtas - 1) / kClusterCtas;
    const int tb = all_t ? 0 : min(T, r * per), te = min(T, tb + per);
    const int32_t* tg = targets + tb;
    const int n = te - tb;
    const uintptr_t addr = reinterpret_cast<uintptr_t>(tg);
    const int head = min(n, static_cast<int>(((16u - (addr & 15u)) & 15u) >> 2));
    if (tid < head) mark(__ldg(tg + tid));
    const int n4 = (n - head) / 4;
    const int4* t4 = reinterpret_cast<const int4*>(tg + head);
    for (int i = tid; i < n4; i += kCandThreads) {
      const int4 x = __ldg(t4 + i);
      mark(x.x);
      mark(x.y);
      mark(x.z);
      mark(x.w);
    }
    for (int t = head + 4 * n4 + tid; t < n; t += kCandThreads) mark(__ldg(tg + t));
  }
  if (all_t) {
    __syncthreads();
    if (sh.err) {  // no shared memory of a peer has been touched: CTAs may leave
      if (r == 0 && tid == 0) {
        set_status(hdr, SS_ERR_TARGET_RANGE);
        hdr[1] = -1;
      }
      return;
    }
  } else {
    cluster.sync();  // every CTA's share is marked
    // reduce-scatter: this CTA's slice [w0, min(w0 + wpc, nWp)) of the union
    const int s1 = min(w0 + wpc, nWp);
    for (int i = w0 + 4 * tid; i < s1; i += 4 * kCandThreads) {
      uint4 o = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int q = 0; q < kClusterCtas; ++q) {
        const uint4 x = *reinterpret_cast<const uint4*>(cluster.map_shared_rank(mine, q) + i);
        o.x |= x.x;
        o.y |= x.y;
        o.z |= x.z;
        o.w |= x.w;
      }
      *reinterpret_cast<uint4*>(full + i) = o;
    }
    if (warp == 0) {
      const int e = lane < kClusterCtas ? cluster.map_shared_rank(&sh, lane)->err : 0;
      const unsigned any = __ballot_sync(0xffffffffu, e != 0);
      if (lane == 0) sh.any_err = any != 0u;
    }
    cluster.sync();  // every slice of the union is complete
    if (sh.any_err) {
      if (r == 0 && tid == 0) {
        set_status(hdr, SS_ERR_TARGET_RANGE);
        hdr[1] = -1;
      }
      cluster.sync();  // no CTA leaves while a peer may still read its shared memory
      return;
    }
    // all-gather: the other slices from their owners
    for (int i = 4 * tid; i < nWp; i += 4 * kCandThreads) {
      const int q = i / wpc;  // words past the last slice are >= nW: zero already
      if (q != r && q < kClusterCtas)
        *reinterpret_cast<uint4*>(full + i) =
            *reinterpret_cast<const uint4*>(cluster.map_shared_rank(full, q) + i);
    }
    __syncthreads();
  }
  // popcount scan over the whole bitmap: a contiguous chunk of words per thread
  {
    const int wpt = (nW + kCandThreads - 1) / kCandThreads;
    const int c0 = min(tid * wpt, nW), c1 = min(c0 + wpt, nW);
    uint32_t cnt = 0;
    for (int i = c0; i < c1; ++i) cnt += __popc(full[i]);
    uint32_t tot;
    uint32_t run = block_scan(cnt, sh.scan, &tot);
    for (int i = c0; i < c1; ++i) {
      fpre[i] = run;
      run += __popc(full[i]);
    }
    if (tid == 0) fpre[nW] = tot;
  }
  __syncthreads();
  const uint32_t U = fpre[nW];
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

  // 2. select the k non-targets with the smallest keys
  if (k == n_non) {
    for (int i = tid; i < nw; i += kCandThreads) {
      const int vbase = (w0 + i) * 32;
      const uint32_t valid = (V - vbase >= 32) ? 0xffffffffu : ((1u << (V - vbase)) - 1u);
      sel[i] = ~full[w0 + i] & valid;
    }
    if (tid < kClusterCtas) {  // every slice's non-target count, from the local prefixes
      const int q0 = min(tid * wpc, nW), q1 = min(q0 + wpc, nW);
      const int ids = max(0, min(V, q1 * 32) - q0 * 32);
      sh.below[tid] = static_cast<uint32_t>(ids) - (fpre[q1] - fpre[q0]);
    }
  } else if (k > 0) {
    uint32_t prefix = 0, mask = 0, rem = k;
    for (int level = 0;; ++level) {
      const int shift = 24 - 8 * level;
      const bool last = level == 3;
      uint32_t* hb = hist + (level & 1) * kBins;
      for (int i = tid; i < kBins; i += kCandThreads) hb[i] = 0u;
      __syncthreads();
      for (int i = warp; i < nw; i += kWarps) {
        const int v = (w0 + i) * 32 + lane;
        if (v < V && !((full[w0 + i] >> lane) & 1u)) {
          uint32_t h;
          if (small_v && level > 0) {
            h = hs[i * 32 + lane];
          } else {
            h = negative_hash(seed, static_cast<uint32_t>(v));
            if (small_v) hs[i * 32 + lane] = h;
          }
          if ((h & mask) == prefix) atomicAdd(&hb[(h >> shift) & (kBins - 1)], 1u);
        }
      }
      cluster.sync();  // every CTA's histogram of this level is complete
      // gather the eight histograms into gat[q][bin]
      for (int i = tid; i < kClusterCtas * kBins / 4; i += kCandThreads) {
        const int q = i / (kBins / 4), j = i % (kBins / 4);
        reinterpret_cast<uint4*>(gat)[i] =
            reinterpret_cast<const uint4*>(cluster.map_shared_rank(hb, q))[j];
      }
      __syncthreads();
      // bin search: thread i < kBins holds bin i's cluster total; a scan over
      // the kBins threads finds the bin where rank rem falls
      uint32_t tb = 0;
      if (tid < kBins) {
#pragma unroll
        for (int q = 0; q < kClusterCtas; ++q) tb += gat[q * kBins + tid];
      }
      const uint32_t incl = warp_incl_scan(tb);
      if (lane == 31 && warp < kBins / 32) sh.wsum[warp] = incl;
      __syncthreads();
      if (tid < kBins) {
        uint32_t excl = incl - tb;
        for (int w = 0; w < warp; ++w) excl += sh.wsum[w];
        if (excl < rem && rem <= excl + tb) {  // exactly one bin
          sh.b = static_cast<uint32_t>(tid);
          sh.rem = rem - excl;
          sh.cnt = tb;
        }
      }
      __syncthreads();
      // warp q: CTA q's ids below the bin (selected) and in it
      if (warp < kClusterCtas) {
        const int bb = static_cast<int>(sh.b);
        uint32_t s = 0;
        for (int i = lane; i < bb; i += 32) s += gat[warp * kBins + i];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) {
          sh.below[warp] += s;
          sh.at_b[warp] = gat[warp * kBins + bb];
        }
      }
      __syncthreads();
      const uint32_t b = sh.b, cnt = sh.cnt;
      const bool collect = last || cnt <= static_cast<uint32_t>(kTieCap);
      const bool eq_path = last && cnt > static_cast<uint32_t>(kTieCap);
      for (int i = warp; i < nw; i += kWarps) {
        const int v = (w0 + i) * 32 + lane;
        bool below = false, in_bin = false;
        uint32_t h = 0;
        if (v < V && !((full[w0 + i] >> lane) & 1u)) {
          h = small_v ? hs[i * 32 + lane] : negative_hash(seed, static_cast<uint32_t>(v));
          if ((h & mask) == prefix) {
            const uint32_t d = (h >> shift) & static_cast<uint32_t>(kBins - 1);
            below = d < b;
            in_bin = d == b;
          }
        }
        const uint32_t bw = __ballot_sync(0xffffffffu, below);
        if (lane == 0 && bw) sel[i] |= bw;
        if (collect) {
          if (eq_path) {
            const uint32_t ew = __ballot_sync(0xffffffffu, in_bin);
            if (lane == 0) eqb[i] = ew;
          } else if (in_bin) {
            const uint32_t at = atomicAdd(&sh.ntie, 1u);
            tie[at] = (static_cast<uint64_t>(h) << 32) | static_cast<uint32_t>(v);
          }
        }
      }
      prefix |= b << shift;
      mask |= static_cast<uint32_t>(kBins - 1) << shift;
      rem = sh.rem;
      if (!collect) continue;
      if (eq_path) {
        // all 32 hash bits equal: the first `rem` ids of the bin in id order;
        // CTA q's ids of the bin come after those of CTAs 0..q-1
        uint32_t before = 0;
        for (int q = 0; q < r; ++q) before += sh.at_b[q];
        if (tid < kClusterCtas) {
          uint32_t bq = 0;
          for (int q = 0; q < tid; ++q) bq += sh.at_b[q];
          sh.tsel[tid] = rem > bq ? min(rem - bq, sh.at_b[tid]) : 0u;
        }
        const int wpt = (nw + kCandThreads - 1) / kCandThreads;
        const int c0 = min(tid * wpt, nw), c1 = min(c0 + wpt, nw);
        uint32_t ecnt = 0;
        for (int i = c0; i < c1; ++i) ecnt += __popc(eqb[i]);
        uint32_t etot;
        uint32_t e = before + block_scan(ecnt, sh.scan, &etot);
        for (int i = c0; i < c1; ++i) {
          uint32_t bits = eqb[i];
          while (bits) {
            const int j = __ffs(bits) - 1;
            bits &= bits - 1;
            if (e < rem) sel[i] |= 1u << j;
            ++e;
          }
        }
      } else {
        // The selected bin is small: gather every CTA's list of its ids after
        // this CTA's own list, rank all of them exactly by (hash, id), keep
        // this CTA's ranks below rem, and count every CTA's selections.
        cluster.sync();  // tie lists complete
        uint64_t* all = tie + kTieCap;
        if (warp == 0) {
          const uint32_t n = lane < kClusterCtas ? cluster.map_shared_rank(&sh, lane)->ntie : 0u;
          const uint32_t incl = warp_incl_scan(n);
          if (lane < kClusterCtas) sh.toff[lane] = incl - n;
          if (lane == kClusterCtas - 1) sh.toff[kClusterCtas] = incl;
        }
        __syncthreads();
        const uint32_t ntot = sh.toff[kClusterCtas];
        for (uint32_t i = tid; i < ntot; i += kCandThreads) {
          int q = 0;
          while (q + 1 < kClusterCtas && sh.toff[q + 1] <= i) ++q;
          all[i] = cluster.map_shared_rank(tie, q)[i - sh.toff[q]];
        }
        __syncthreads();
        // One more radix digit, locally (every CTA holds the whole list): the
        // entries agree on the hash bits above `shift`; count them by key bits
        // [24 + shift, 32 + shift) (the next 8 hash bits; id bits when all hash
        // bits are fixed), find the sub-bin where rank rem falls, take the
        // entries below it, and rank the sub-bin's few entries exactly, a warp
        // per entry.
        const int dshift = 24 + shift;
        uint32_t* lcnt = gat;                  // [kBins]
        uint32_t* tflag = gat + kBins;         // [ntot] taken or not
        uint32_t* sub = tflag + kTieCap;       // [ntot] entries of the sub-bin
        if (tid < kBins) lcnt[tid] = 0u;
        if (tid == 0) sh.m2 = 0u;
        __syncthreads();
        for (uint32_t i = tid; i < ntot; i += kCandThreads)
          atomicAdd(&lcnt[static_cast<uint32_t>(all[i] >> dshift) & (kBins - 1)], 1u);
        __syncthreads();
        {
          const uint32_t c = tid < kBins ? lcnt[tid] : 0u;
          const uint32_t incl = warp_incl_scan(c);
          if (lane == 31 && warp < kBins / 32) sh.wsum[warp] = incl;
          __syncthreads();
          if (tid < kBins) {
            uint32_t excl = incl - c;
            for (int w = 0; w < warp; ++w) excl += sh.wsum[w];
            if (excl < rem && rem <= excl + c) {  // exactly one sub-bin
              sh.b2 = static_cast<uint32_t>(tid);
              sh.rem2 = rem - excl;
            }
          }
          __syncthreads();
        }
        const uint32_t b2 = sh.b2, rem2 = sh.rem2;
        const uint32_t own0 = sh.toff[r], own1 = sh.toff[r + 1];
        for (uint32_t i = tid; i < ntot; i += kCandThreads) {
          const uint64_t key = all[i];
          const uint32_t d = static_cast<uint32_t>(key >> dshift) & (kBins - 1);
          tflag[i] = d < b2 ? 1u : 0u;
          if (d < b2 && i >= own0 && i < own1) {
            const int v = static_cast<int>(key & 0xffffffffu);
            atomicOr(&sel[(v >> 5) - w0], 1u << (v & 31));
          }
          if (d == b2) sub[atomicAdd(&sh.m2, 1u)] = i;
        }
        __syncthreads();
        const uint32_t m2 = sh.m2;
        for (uint32_t s2 = warp; s2 < m2; s2 += kWarps) {
          const uint32_t i = sub[s2];
          const uint64_t key = all[i];
          uint32_t rank = 0;
          for (uint32_t j = lane; j < ntot; j += 32) {
            const uint64_t o = all[j];
            rank += ((static_cast<uint32_t>(o >> dshift) & (kBins - 1)) == b2) && o < key;
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) rank += __shfl_xor_sync(0xffffffffu, rank, o);
          if (lane == 0) {
            const bool take = rank < rem2;
            tflag[i] = take ? 1u : 0u;
            if (take && i >= own0 && i < own1) {
              const int v = static_cast<int>(key & 0xffffffffu);
              atomicOr(&sel[(v >> 5) - w0], 1u << (v & 31));
            }
          }
        }
        __syncthreads();
        // warp q counts CTA q's taken entries (its contiguous range of the list)
        if (warp < kClusterCtas) {
          uint32_t c = 0;
          for (uint32_t i = sh.toff[warp] + lane; i < sh.toff[warp + 1]; i += 32) c += tflag[i];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
          if (lane == 0) sh.tsel[warp] = c;
        }
      }
      break;
    }
  }
  // the last reads of peers' shared memory are done: arrive now, wait at the end
  cluster_arrive();
  __syncthreads();

  // 3. compaction: targets of the slice into [0, U), its selected negatives
  //    into [U + offset of this CTA, ...); a warp per word, a lane per bit
  uint32_t soff = U;
  for (int q = 0; q < r; ++q) soff += sh.below[q] + sh.tsel[q];
  {
    const int wpt = (nw + kCandThreads - 1) / kCandThreads;
    const int c0 = min(tid * wpt, nw), c1 = min(c0 + wpt, nw);
    uint32_t scnt = 0;
    for (int i = c0; i < c1; ++i) scnt += __popc(sel[i]);
    uint32_t stot;
    uint32_t run = block_scan(scnt, sh.scan, &stot);
    for (int i = c0; i < c1; ++i) {  // sel's words now hold their exclusive prefix in eqb
      eqb[i] = run;
      run += __popc(sel[i]);
    }
  }
  __syncthreads();
  const uint32_t below_mask = (1u << lane) - 1u;
  for (int i = warp; i < nw; i += kWarps) {
    const int v = (w0 + i) * 32 + lane;
    const uint32_t tw = full[w0 + i], sw = sel[i];
    if ((tw >> lane) & 1u) cand[fpre[w0 + i] + __popc(tw & below_mask)] = v;
    if ((sw >> lane) & 1u) cand[soff + eqb[i] + __popc(sw & below_mask)] = v;
  }

  // slots of one eighth of the tokens, from the local bitmap and prefixes
  for (int t = r * kCandThreads + tid; t < T; t += kClusterCtas * kCandThreads) {
    const int v = __ldg(targets + t);
    const int w = v >> 5;
    slot[t] = static_cast<int32_t>(fpre[w] + __popc(full[w] & ((1u << (v & 31)) - 1u)));
  }
  if (r == 0 && tid == 0) hdr[1] = static_cast<int>(U);
  cluster_wait();  // peers are done with this CTA's shared memory
}

}  // namespace

size_t build_candidates_smem_bytes(int64_t V) {
  const size_t nW = static_cast<size_t>((V + 31) / 32);
  const size_t nWp = (nW + 4) & ~static_cast<size_t>(3);
  const size_t wpc = static_cast<size_t>(slice_words(static_cast<int>(V)));
  size_t bytes = kTieSlots * sizeof(uint64_t) + 3 * nWp * sizeof(uint32_t) +
                 2 * wpc * sizeof(uint32_t) + (2 + kClusterCtas) * kBins * sizeof(uint32_t);
  if (V <= kSmallV) bytes += wpc * 32 * sizeof(uint32_t);  // the slice's hashes
  return bytes;
}

const void* build_candidates_kernel() { return reinterpret_cast<const void*>(k_build_candidates); }

cudaError_t launch_build_candidates(const int32_t* targets, int T, int V, int C, uint64_t seed,
                                    int32_t* cand, int32_t* slot, int* hdr,
                                    cudaStream_t stream) {
  const size_t smem = build_candidates_smem_bytes(V);
  return launch_pdl(k_build_candidates, dim3(kClusterCtas), dim3(kCandThreads), smem, stream, targets,
                    T, V, C, seed, cand, slot, hdr);
}

}  // namespace ss
