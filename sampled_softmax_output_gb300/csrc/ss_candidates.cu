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
// One CTA of 1024 threads does all of it with the vocabulary bitmap in shared
// memory (V bits; 6.3 KB at V = 50,304):
//   1. mark targets in the bitmap (range-checked);
//   2. popcount + block scan -> U and the per-word target prefix;
//   3. radix-select (4 passes of 8 bits) of the (C-U)-th smallest hash among
//      non-targets, ties broken by id;
//   4. block scans over the id range -> compaction into cand;
//   5. slot[t] = word prefix + popcount of the lower bits of its word.
#include <cuda_runtime.h>
#include <stdint.h>

#include "ss.h"
#include "ss_internal.h"
#include "ss_ptx.cuh"

namespace ss {

namespace {

constexpr int kCandThreads = 1024;

__device__ __forceinline__ uint32_t negative_hash(uint64_t seed, uint32_t v) {
  uint64_t z = seed + (static_cast<uint64_t>(v) + 1ull) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  z ^= z >> 31;
  return static_cast<uint32_t>(z >> 32);
}

// Exclusive scan of one value per thread over the 1024-thread block.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t x, uint32_t* warp_sums,
                                                         uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = warp_sums[lane];
    uint32_t wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    warp_sums[lane] = wi - w;  // exclusive prefix of warp totals
    if (lane == 31) warp_sums[32] = wi;
  }
  __syncthreads();
  const uint32_t r = warp_sums[warp] + incl - x;
  *total = warp_sums[32];
  __syncthreads();  // warp_sums may be reused by the caller's next scan
  return r;
}

__global__ void __launch_bounds__(kCandThreads, 1)
    k_build_candidates(const int32_t* __restrict__ targets, int T, int V, int C, uint64_t seed,
                       int32_t* __restrict__ cand, int32_t* __restrict__ slot, int* hdr) {
  extern __shared__ uint32_t sm[];
  __shared__ uint32_t warp_sums[33];
  __shared__ uint32_t hist[256];
  __shared__ int s_err;
  __shared__ uint32_t s_digit, s_rem;

  const int tid = threadIdx.x;
  const int nW = (V + 31) >> 5;
  uint32_t* bm = sm;         // [nW] target bitmap
  uint32_t* wpre = sm + nW;  // [nW] number of targets in words before w

  for (int w = tid; w < nW; w += kCandThreads) bm[w] = 0u;
  if (tid == 0) s_err = 0;
  __syncthreads();

  // 1. mark
  for (int t = tid; t < T; t += kCandThreads) {
    const int v = __ldg(targets + t);
    if (static_cast<unsigned>(v) >= static_cast<unsigned>(V)) {
      s_err = 1;
    } else {
      const uint32_t bit = 1u << (v & 31);
      if (!(bm[v >> 5] & bit)) atomicOr(&bm[v >> 5], bit);
    }
  }
  __syncthreads();
  if (s_err) {
    if (tid == 0) {
      set_status(hdr, SS_ERR_TARGET_RANGE);
      hdr[1] = -1;
    }
    return;
  }

  // 2. U and word prefixes; each thread owns a contiguous range of words
  const int wpt = (nW + kCandThreads - 1) / kCandThreads;
  const int w0 = min(tid * wpt, nW), w1 = min(w0 + wpt, nW);
  const int v0 = w0 * 32, v1 = min(w1 * 32, V);
  uint32_t cnt = 0;
  for (int w = w0; w < w1; ++w) cnt += __popc(bm[w]);
  uint32_t U;
  const uint32_t tbase = block_exclusive_scan(cnt, warp_sums, &U);
  {
    uint32_t run = tbase;
    for (int w = w0; w < w1; ++w) {
      wpre[w] = run;
      run += __popc(bm[w]);
    }
  }
  if (static_cast<int>(U) > C) {
    if (tid == 0) {
      set_status(hdr, SS_ERR_CAPACITY);
      hdr[1] = static_cast<int>(U);
    }
    return;
  }
  const uint32_t k = static_cast<uint32_t>(C) - U;

  // 3. radix-select the k-th smallest hash among non-targets
  uint32_t prefix = 0, pmask = 0, rem = k;
  if (k > 0) {
#pragma unroll 1
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      if (tid < 256) hist[tid] = 0u;
      __syncthreads();
      for (int v = v0; v < v1; ++v) {
        if (bm[v >> 5] & (1u << (v & 31))) continue;
        const uint32_t h = negative_hash(seed, static_cast<uint32_t>(v));
        if ((h & pmask) == prefix) atomicAdd(&hist[(h >> shift) & 255u], 1u);
      }
      __syncthreads();
      if (tid == 0) {
        uint32_t cum = 0, digit = 255;
        for (int d = 0; d < 256; ++d) {
          if (cum + hist[d] >= rem) {
            digit = static_cast<uint32_t>(d);
            break;
          }
          cum += hist[d];
        }
        s_digit = digit;
        s_rem = rem - cum;
      }
      __syncthreads();
      prefix |= s_digit << shift;
      pmask |= 255u << shift;
      rem = s_rem;
    }
  }
  // Selected negatives: hash < prefix, plus the first `rem` ids (ascending)
  // whose hash == prefix.

  // 4. compaction
  uint32_t nlt = 0, neq = 0;
  if (k > 0) {
    for (int v = v0; v < v1; ++v) {
      if (bm[v >> 5] & (1u << (v & 31))) continue;
      const uint32_t h = negative_hash(seed, static_cast<uint32_t>(v));
      nlt += (h < prefix);
      neq += (h == prefix);
    }
  }
  uint32_t eq_total, sel_total;
  const uint32_t eq_base = block_exclusive_scan(neq, warp_sums, &eq_total);
  const uint32_t take_eq = rem > eq_base ? min(rem - eq_base, neq) : 0u;
  const uint32_t sel_base = block_exclusive_scan(nlt + take_eq, warp_sums, &sel_total);
  {
    uint32_t ti = tbase, ni = U + sel_base, ei = eq_base;
    for (int v = v0; v < v1; ++v) {
      if (bm[v >> 5] & (1u << (v & 31))) {
        cand[ti++] = v;
      } else if (k > 0) {
        const uint32_t h = negative_hash(seed, static_cast<uint32_t>(v));
        if (h < prefix) {
          cand[ni++] = v;
        } else if (h == prefix) {
          if (ei < rem) cand[ni++] = v;
          ++ei;
        }
      }
    }
  }
  __syncthreads();  // wpre complete

  // 5. slots
  for (int t = tid; t < T; t += kCandThreads) {
    const int v = __ldg(targets + t);
    const int w = v >> 5;
    slot[t] = static_cast<int32_t>(wpre[w] + __popc(bm[w] & ((1u << (v & 31)) - 1u)));
  }
  if (tid == 0) hdr[1] = static_cast<int>(U);
}

}  // namespace

size_t build_candidates_smem_bytes(int64_t V) {
  return static_cast<size_t>((V + 31) / 32) * 2 * sizeof(uint32_t);
}

cudaError_t launch_build_candidates(const int32_t* targets, int T, int V, int C, uint64_t seed,
                                    int32_t* cand, int32_t* slot, int* hdr,
                                    cudaStream_t stream) {
  const size_t smem = build_candidates_smem_bytes(V);
  cudaError_t e = cudaFuncSetAttribute(k_build_candidates,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  k_build_candidates<<<1, kCandThreads, smem, stream>>>(targets, T, V, C, seed, cand, slot, hdr);
  return cudaGetLastError();
}

}  // namespace ss
