// ss_api.cu -- the C ABI declared in include/ss.h: argument checks, the
// workspace layout, TMA tensor maps, and the launch sequence of each call.
// Also holds the three small memory-bound kernels of the path: the candidate
// row gather W_c = W[cand], the log-sum-exp merge of the forward partials, and
// the zeroing of candidate rows for an empty batch.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <mutex>
#include <vector>

#include "ss.h"
#include "ss_internal.h"
#include "ss_ptx.cuh"

namespace ss {

// Kernels launched by this host thread (launch_pdl counts them).
thread_local int g_kernel_launches = 0;

namespace {

// ------------------------------------------------------------ workspace

struct Layout {
  size_t hdr, wc, part, tgt, g, g8t, h8, hq, h8t, w8, w8t, total;
  int64_t ldG, n_ct;
  int64_t ldT8, ldC8;  // row pitch (bytes) of the transposed e4m3 / e5m2 copies
};

constexpr size_t kHdrBytes = 1024;  // int32 status, int32 U, padding, FP8 amax words
constexpr size_t kHdrAmax = 64;     // byte offset of float amax[2] (max |H|, max |W_c|)
constexpr size_t kHdrBar = 72;      // uint32 bar[2] of k_h_prep_beside (arrivals, gave up)
constexpr size_t kHdrQuant = 80;    // ss_quantize_e4m3's own float amax + int32 status
constexpr size_t kHdrFallback = 96;  // int32: ss_step's stored-probability backward falls back

// The grid barrier of k_h_prep_beside waits for as many arrivals as its grid
// has blocks, for up to 4 s. A test builds a copy of the library with one
// more arrival than blocks and a 1 ms limit, so that the wait runs out (the
// timeout path, with no fault and nothing else in flight); the library
// itself is built with the defaults.
#ifndef SS_BESIDE_EXTRA_ARRIVALS
#define SS_BESIDE_EXTRA_ARRIVALS 0
#endif
#ifndef SS_BESIDE_WAIT_NS
#define SS_BESIDE_WAIT_NS 4000000000ull
#endif

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

Layout make_layout(int64_t T, int64_t C, int64_t D) {
  Layout L;
  L.ldG = (C + 63) / 64 * 64;
  L.n_ct = (C + kBnLogits - 1) / kBnLogits;
  size_t off = 0;
  L.hdr = off;
  off += kHdrBytes;
  L.wc = off;
  off = align_up(off + static_cast<size_t>(C) * D * 2, 1024);
  L.part = off;
  off = align_up(off + static_cast<size_t>(L.n_ct) * kFwdGroupsMax * T * sizeof(float2), 1024);
  L.tgt = off;  // target logits, up to kMaxTargets per token; then r and the row factors
  off = align_up(off + static_cast<size_t>(T) * (kMaxTargets + 2) * sizeof(float), 1024);
  L.ldT8 = (T + 15) / 16 * 16;
  L.ldC8 = (C + 15) / 16 * 16;
  // G in bf16, or (FP8 gradients) G8 [T, ldG] and G8^T [C, ldT8] in e5m2
  L.g = off;
  L.g8t = align_up(off + static_cast<size_t>(T) * L.ldG, 1024);
  off = align_up(std::max(off + static_cast<size_t>(T) * L.ldG * 2,
                          L.g8t + static_cast<size_t>(C) * L.ldT8),
                 1024);
  // the FP8 head's operands: H and W_c in e4m3; H rounded to the e4m3 grid in
  // bf16 (FP8 logits only) or, in the same place, H^T in e4m3 (FP8 gradients);
  // W_c^T in e4m3 (FP8 gradients)
  L.h8 = off;
  off = align_up(off + static_cast<size_t>(T) * D, 1024);
  L.hq = L.h8t = off;
  off = align_up(off + std::max(static_cast<size_t>(T) * D * 2, static_cast<size_t>(D) * L.ldT8),
                 1024);
  L.w8 = off;
  off = align_up(off + static_cast<size_t>(C) * D, 1024);
  L.w8t = off;
  off = align_up(off + static_cast<size_t>(D) * L.ldC8, 1024);
  L.total = off;
  return L;
}

ss_status check_sizes(int64_t T, int64_t V, int64_t C, int64_t D) {
  if (T < 0 || V <= 0 || C <= 0 || D <= 0 || C > V) return SS_ERR_INVALID;
  if (T >= (int64_t(1) << 31) || V > SS_MAX_V || D > SS_MAX_D || D % 64 != 0 || D < 64)
    return SS_ERR_UNSUPPORTED;
  return SS_OK;
}

bool aligned(const void* p, size_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

// ------------------------------------------------------------ device info

constexpr int kMaxDevices = 64;
std::atomic<int> g_num_sms[kMaxDevices];

int num_sms_current() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  int n = g_num_sms[dev].load(std::memory_order_relaxed);
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  g_num_sms[dev].store(n, std::memory_order_relaxed);
  return n;
}

// ------------------------------------------------------------ tensor maps

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Row-major bf16 matrix [outer, inner] with `row_bytes` between rows, read in
// boxes of box_outer rows x box_inner elements with the 128-byte swizzle (or
// another element type and swizzle).
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
              uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
              CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
              CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  return fn(m, dtype, 2, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ------------------------------------------------------------ small kernels

// max |x| over this thread's grid-stride slice of x (n8 groups of 8 bf16),
// four loads in flight, as bf16 magnitude bits
__device__ __forceinline__ uint32_t absmax_slice(const uint16_t* __restrict__ x, int64_t n8) {
  const uint4* v = reinterpret_cast<const uint4*>(x);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  uint32_t mx = 0u;
  for (; i + 3 * stride < n8; i += 4 * stride) {
    const uint4 a = __ldg(v + i), b = __ldg(v + i + stride), c = __ldg(v + i + 2 * stride),
                d = __ldg(v + i + 3 * stride);
    mx = max(mx, max(max(bf16x8_absmax_bits(a), bf16x8_absmax_bits(b)),
                     max(bf16x8_absmax_bits(c), bf16x8_absmax_bits(d))));
  }
  for (; i < n8; i += stride) mx = max(mx, bf16x8_absmax_bits(__ldg(v + i)));
  return mx;
}

// *amax = max(*amax, the warp's largest magnitude): an atomic max of the
// non-negative float's bits
__device__ __forceinline__ void warp_atomic_max(float* amax, uint32_t mx) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((threadIdx.x & 31) == 0 && mx) atomicMax(reinterpret_cast<unsigned*>(amax), mx << 16);
}

// W_c[j, :] = W[cand[j], :]; one warp per row, 16-byte vectors. AMAX (the FP8
// head): also max |W_c| into *amax and, over a second tensor x (n8 groups of
// 8), max |x| into *x_amax.
template <bool AMAX>
__global__ void __launch_bounds__(256) k_gather_rows(const uint16_t* __restrict__ W,
                                                     const int32_t* __restrict__ cand, int C,
                                                     int V, int D, uint16_t* __restrict__ Wc,
                                                     float* amax, const uint16_t* __restrict__ x,
                                                     int64_t x_n8, float* x_amax, int* status) {
  pdl_enter();
  if (read_status(status) != 0) return;
  const int lane = threadIdx.x & 31;
  const int n16 = D / 8;
  const int warps = gridDim.x * (blockDim.x / 32);
  uint32_t mx = 0u;  // AMAX: max |x| over the copied rows, as bf16 magnitude bits
  for (int j = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32; j < C; j += warps) {
    const int v = __ldg(cand + j);
    uint4* dst = reinterpret_cast<uint4*>(Wc + static_cast<size_t>(j) * D);
    if (static_cast<unsigned>(v) >= static_cast<unsigned>(V)) {
      if (lane == 0) set_status(status, SS_ERR_INDEX);
      for (int i = lane; i < n16; i += 32) dst[i] = make_uint4(0, 0, 0, 0);
      continue;
    }
    const uint4* src = reinterpret_cast<const uint4*>(W + static_cast<size_t>(v) * D);
    if constexpr (AMAX) {
      for (int i = lane; i < n16; i += 32) {
        const uint4 q = __ldg(src + i);
        dst[i] = q;
        mx = max(mx, bf16x8_absmax_bits(q));
      }
      continue;
    }
    // all of a lane's loads of the row (four at D <= 1024) in flight before
    // its stores (measured 15 -> 13 us for 10240 rows of 768; with the max
    // over the rows the single-load loop was faster)
    for (int i0 = lane; i0 < n16; i0 += 4 * 32) {
      uint4 q[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (i0 + 32 * u < n16) q[u] = __ldg(src + i0 + 32 * u);
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (i0 + 32 * u < n16) dst[i0 + 32 * u] = q[u];
    }
  }
  if constexpr (AMAX) {
    warp_atomic_max(amax, mx);
    if (x_amax) warp_atomic_max(x_amax, absmax_slice(x, x_n8));
  }
}

// amax[0] = max over x of |x| (n bf16 values, n % 8 == 0), as an atomic max of
// the non-negative float's bits
__global__ void __launch_bounds__(256) k_amax_bf16(const uint16_t* __restrict__ x, int64_t n8,
                                                   float* amax, int* status) {
  pdl_enter();
  if (read_status(status) != 0) return;
  warp_atomic_max(amax, absmax_slice(x, n8));
}

// The FP8 head's operands, two tensors in one launch (job 0: H, job 1: W_c):
// q = e4m3(x * 2^e) and xq = bf16(e4m3 value * 2^-e) (exact), e from the
// tensor's amax; xq may alias x.
struct QuantJob {
  const uint16_t* x;
  uint8_t* q;
  uint16_t* xq;
  const float* amax;
  int64_t n8;  // groups of 8 values
};
// Groups i0, i0 + stride, ... of job J (the row-major quantizer's work).
__device__ __forceinline__ void quantize_rows(const QuantJob& J, int64_t i0, int64_t stride) {
  const int e = e4m3_exponent(__ldcg(J.amax));
  const float up = exp2i(e), down = exp2i(-e);
  for (int64_t i = i0; i < J.n8; i += stride) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(J.x) + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t qw[2], out[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float lo = __uint_as_float(w[k] << 16) * up;
      const float hi = __uint_as_float(w[k] & 0xffff0000u) * up;
      const uint16_t c = e4m3x2(lo, hi);
      const uint32_t h2 = e4m3x2_to_f16x2(c);
      const float dlo = __half2float(__ushort_as_half(static_cast<uint16_t>(h2 & 0xffffu))) * down;
      const float dhi = __half2float(__ushort_as_half(static_cast<uint16_t>(h2 >> 16))) * down;
      out[k] = (__float_as_uint(dlo) >> 16) | (__float_as_uint(dhi) & 0xffff0000u);
      if (k & 1) qw[k >> 1] |= static_cast<uint32_t>(c) << 16;
      else qw[k >> 1] = c;
    }
    reinterpret_cast<uint2*>(J.q)[i] = make_uint2(qw[0], qw[1]);
    reinterpret_cast<uint4*>(J.xq)[i] = make_uint4(out[0], out[1], out[2], out[3]);
  }
}

// beside_fail (nullable): set when H's half, quantized beside the candidate
// build (k_h_prep_beside), gave up waiting; reported here as SS_ERR_TIMEOUT.
__global__ void __launch_bounds__(256) k_quantize_e4m3(QuantJob a, QuantJob b, int* status,
                                                       const uint32_t* beside_fail) {
  pdl_enter();
  if (read_status(status) != 0) return;
  if (beside_fail && __ldcg(beside_fail) != 0u) {
    if (blockIdx.x == 0 && threadIdx.x == 0) set_status(status, SS_ERR_TIMEOUT);
    return;
  }
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t i0 = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  quantize_rows(a, i0, stride);
  quantize_rows(b, i0, stride);
}

// FP8 gradients: x [R, D] bf16 (D % 64 == 0) to e4m3 codes twice, q [R, D]
// row-major (the logit GEMMs) and qt [D, ldR] transposed (the gradient GEMMs,
// which need K = R contiguous), e from the tensor's amax. One 64 x 64 tile per
// iteration, transposed through shared memory; two tensors in one launch.
struct QuantTJob {
  const uint16_t* x;
  uint8_t* q;
  uint8_t* qt;
  const float* amax;
  int R, D, ldR, tiles;  // tiles = ceil(R / 64) * (D / 64)
};
constexpr int kQtPitch = 72;  // bytes per row of the shared tile (64 + 8 against conflicts)
// Tile ti of job J, transposed through the shared tile; every thread of the
// block calls it (it synchronises the block).
__device__ __forceinline__ void quantize_t_tile(const QuantTJob& J, int ti, uint8_t* tile) {
  const int nct = J.D / 64;
  const int r0 = (ti / nct) * 64, c0 = (ti % nct) * 64;
  const float up = exp2i(e4m3_exponent(__ldcg(J.amax)));
  __syncthreads();  // the previous tile's transposed reads are done
  for (int v = threadIdx.x; v < 512; v += blockDim.x) {
    const int r = v >> 3, c8 = (v & 7) * 8;  // row r, columns c8 .. c8 + 7 of the tile
    uint32_t qw[2] = {0u, 0u};
    if (r0 + r < J.R) {
      const size_t at = static_cast<size_t>(r0 + r) * J.D + c0 + c8;
      const uint4 x = __ldg(reinterpret_cast<const uint4*>(J.x + at));
      const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint16_t c = e4m3x2(__uint_as_float(xw[k] << 16) * up,
                                  __uint_as_float(xw[k] & 0xffff0000u) * up);
        qw[k >> 1] |= static_cast<uint32_t>(c) << (16 * (k & 1));
      }
      *reinterpret_cast<uint2*>(J.q + at) = make_uint2(qw[0], qw[1]);
    }
    *reinterpret_cast<uint2*>(tile + r * kQtPitch + c8) = make_uint2(qw[0], qw[1]);
  }
  __syncthreads();
  for (int v = threadIdx.x; v < 512; v += blockDim.x) {
    const int c = v >> 3, rg = (v & 7) * 8;  // column c, rows rg .. rg + 7 of the tile
    const int nr = min(8, J.R - r0 - rg);
    if (nr <= 0) continue;
    uint32_t o[2] = {0u, 0u};
#pragma unroll
    for (int k = 0; k < 8; ++k)
      o[k >> 2] |= static_cast<uint32_t>(tile[(rg + k) * kQtPitch + c]) << (8 * (k & 3));
    uint8_t* dst = J.qt + static_cast<size_t>(c0 + c) * J.ldR + r0 + rg;
    if (nr == 8) {
      *reinterpret_cast<uint2*>(dst) = make_uint2(o[0], o[1]);
    } else {
      for (int k = 0; k < nr; ++k) dst[k] = static_cast<uint8_t>(o[k >> 2] >> (8 * (k & 3)));
    }
  }
}

// beside_fail: as for k_quantize_e4m3.
__global__ void __launch_bounds__(256) k_quantize_e4m3_t(QuantTJob a, QuantTJob b, int* status,
                                                         const uint32_t* beside_fail) {
  pdl_enter();
  if (read_status(status) != 0) return;
  if (beside_fail && __ldcg(beside_fail) != 0u) {
    if (blockIdx.x == 0 && threadIdx.x == 0) set_status(status, SS_ERR_TIMEOUT);
    return;
  }
  __shared__ __align__(16) uint8_t tile[64 * kQtPitch];
  for (int w = blockIdx.x; w < a.tiles + b.tiles; w += gridDim.x) {
    if (w < a.tiles) quantize_t_tile(a, w, tile);
    else quantize_t_tile(b, w - a.tiles, tile);
  }
}

// The FP8 head's H beside the candidate build, launched right after it: max
// |H| into *amax, then, after a barrier over this grid, H's e4m3 operands
// (mode 1: jr, as k_quantize_e4m3; mode 2: jt, as k_quantize_e4m3_t).
// - No wait at the start: this grid may start once every CTA of the build has
//   started, by which time everything the build waited for (H's producer
//   among it) is complete, and the build writes nothing this kernel reads.
// - The grid barrier can be waited on: the kernel after this one is launched
//   only once every block of this grid has started, so all of them are
//   resident together (the build holds 8 SMs). bar[0] counts arrivals up to
//   `arrivals` (the grid size); a block that has waited `wait_ns` (4 s) gives
//   up and sets bar[1], which the W_c quantizer reports as SS_ERR_TIMEOUT.
//   bar[0..1] and *amax are zero at launch.
// - It waits for the build before it exits, so that the kernels after it,
//   which wait for it, find the build's results. No status check: the build
//   clears the status word while this kernel may run.
__global__ void __launch_bounds__(256) k_h_prep_beside(int64_t n8, float* amax, uint32_t* bar,
                                                       uint32_t arrivals, uint64_t wait_ns,
                                                       QuantJob jr, QuantTJob jt, int mode) {
  pdl_launch_dependents();
  __shared__ __align__(16) uint8_t tile[64 * kQtPitch];
  __shared__ int s_go;
  warp_atomic_max(amax, absmax_slice(jr.x, n8));
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(bar, 1u);
    const uint64_t t0 = globaltimer_ns();
    int go = 1;
    while (ld_acquire_gpu(bar) < arrivals) {
      if (globaltimer_ns() - t0 > wait_ns) {
        atomicExch(bar + 1, 1u);
        go = 0;
        break;
      }
    }
    s_go = go;
  }
  __syncthreads();
  if (s_go) {
    if (mode == 2) {
      for (int w = blockIdx.x; w < jt.tiles; w += gridDim.x) quantize_t_tile(jt, w, tile);
    } else {
      quantize_rows(jr, blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x,
                    static_cast<int64_t>(gridDim.x) * blockDim.x);
    }
  }
  pdl_wait();
}

// lse[t] = log sum over tiles of s_c * exp(m_c); loss[t] = lse[t] - tgt[t].
// Eight threads per token: thread k folds tiles k, k + 8, ... online, then the
// eight (max, sum) pairs are combined with shuffles. (-inf, 0) marks a tile
// part without valid columns.
constexpr int kMergeLanes = 8;
static_assert(kMaxTargets <= kMergeLanes, "one lane of a token's group per target");

__device__ __forceinline__ void lse_fold(float& M, float& S, float m, float s) {
  if (m == -INFINITY) return;
  const float nm = fmaxf(M, m);
  S = S * expf(M - nm) + s * expf(m - nm);
  M = nm;
}

__global__ void __launch_bounds__(256) k_lse_merge(const float2* __restrict__ part,
                                                   const float* __restrict__ tgt,
                                                   const int32_t* __restrict__ slot, int T, int C,
                                                   int n_ct, Targets tg,
                                                   float* __restrict__ loss,
                                                   float* __restrict__ lse, int* status) {
  pdl_enter();
  if (read_status(status) != 0) return;
  // grid-stride over tokens, the same trip count for a whole block
  const int64_t lanes = static_cast<int64_t>(T) * kMergeLanes;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t g0 = static_cast<int64_t>(blockIdx.x) * blockDim.x; g0 < lanes; g0 += stride) {
    const int64_t gid = g0 + threadIdx.x;
    const int t = static_cast<int>(gid / kMergeLanes);
    const int k = static_cast<int>(gid % kMergeLanes);
    const bool valid = gid < lanes;  // whole groups of 8 lanes share a token
    // lane j < K of the group fetches target j's slot and logit along with the
    // partials (one memory round trip for all of them)
    int my_slot = 0;
    float my_tgt = 0.f;
    if (valid && k < tg.K) {
      my_slot = __ldg(slot + static_cast<size_t>(k) * T + t);
      my_tgt = __ldcg(tgt + static_cast<size_t>(k) * T + t);
    }
    float M = -INFINITY, S = 0.f;
    constexpr int kBatch = 8;  // loads a thread has in flight
    if (valid)
      for (int c0 = k; c0 < n_ct; c0 += kMergeLanes * kBatch) {
        float2 q[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
          const int c = c0 + i * kMergeLanes;
          q[i] = c < n_ct ? __ldcg(part + static_cast<size_t>(c) * T + t)
                          : make_float2(-INFINITY, 0.f);
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i) lse_fold(M, S, q[i].x, q[i].y);
      }
#pragma unroll
    for (int o = 1; o < kMergeLanes; o <<= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, M, o);
      const float s2 = __shfl_xor_sync(0xffffffffu, S, o);
      lse_fold(M, S, m2, s2);
    }
    const float l = M + logf(S);
    // sum over the targets of w[j] (lse - target logit), lanes 0..K-1 of the
    // group (one target: lse - tgt); a slot out of range is an error
    bool bad = valid && k < tg.K && static_cast<unsigned>(my_slot) >= static_cast<unsigned>(C);
    float acc = 0.f;
    const int base = (threadIdx.x & 31) & ~(kMergeLanes - 1);
    for (int j = 0; j < tg.K; ++j) {  // K <= kMergeLanes
      const float tj = __shfl_sync(0xffffffffu, my_tgt, base + j);
      acc += tg.w[j] * (l - tj);
    }
#pragma unroll
    for (int o = 1; o < kMergeLanes; o <<= 1) bad |= __shfl_xor_sync(0xffffffffu, bad, o) != 0;
    if (valid && k == 0) {
      if (bad) {
        set_status(status, SS_ERR_INDEX);
      } else {
        lse[t] = l;
        loss[t] = acc;
      }
    }
  }
}

// ss_step's merge when the forward kept the probabilities (EpiFwdP): lse and
// loss as k_lse_merge (two partials per row per logit tile), then, for the
// backward, per token t with alpha = exp(r[t] - lse[t]):
//   rowfac[t] = scale * alpha                        dH   = rowfac * (Pt' . W_c)
//   Pt[t, slot[t]] = bf16(exp(tgt - r) - exp(lse - r))   so Pt' = (P - Y) / alpha
//   Hs[t, :] = bf16(alpha * H[t, :])                 dW_c = scale * (Pt'^T . Hs)
// The target column is recomputed from the fp32 target logit, so (P - 1) keeps
// its precision when P is close to 1. A row whose lse exceeds r by more than
// kStoredSpan (or is not finite) raises *fallback: alpha and Pt' would then
// leave the range where bf16 holds them to full precision, and the backward
// recomputes G from the logits instead (the gated softmax-gradient GEMM,
// which then also resets Hs to H and the row factors to `scale`).
constexpr float kStoredSpan = 60.f;

// Partials relative to the row's reference r (the forward's usual case) add
// without exponentials; a partial with another maximum folds as lse_fold.
__device__ __forceinline__ void lse_fold_same(float& M, float& S, float m, float s) {
  if (m == M) {
    S += s;
    return;
  }
  lse_fold(M, S, m, s);
}

// One block per kMergeTokens consecutive tokens. Warp w folds the partial rows
// c = w, w + 8, ... (each row's kMergeTokens entries are contiguous: one
// 256-byte load per warp and row), the eight warps' (max, sum) pairs meet in
// shared memory, and then the block scales the tokens' H rows (one contiguous
// block of kMergeTokens * D values) into Hs.
constexpr int kMergeTokens = 32;

// CAP: the capped head's stored forward (EpiFwdP<false, NBUF, true>): the
// reference is cap for every row, tgt holds z at the target, and the patched
// target entry carries dz/ds there; lse - cap <= ln C, so no fallback.
template <bool CAP>
__global__ void __launch_bounds__(256) k_lse_merge_p(
    const float2* __restrict__ part, const float* __restrict__ tgt,
    const int32_t* __restrict__ slot, const float* __restrict__ ref, int T, int C, int n_parts,
    const uint16_t* __restrict__ H, int D, float scale, uint16_t* __restrict__ Pt, int64_t ldP,
    uint16_t* __restrict__ Hs, float* __restrict__ rowfac, int* fallback,
    float* __restrict__ loss, float* __restrict__ lse, int* status, HeadCap head, Targets tg) {
  static_assert(kMergeTokens == 32, "one lane per token");
  __shared__ float2 red[8][kMergeTokens];
  __shared__ float s_alpha[kMergeTokens];
  __shared__ int s_go;
  pdl_enter();
  // one decision per block: its threads meet at barriers below
  if (threadIdx.x == 0) s_go = read_status(status) == 0;
  __syncthreads();
  if (!s_go) return;
  const int warp = static_cast<int>(threadIdx.x) >> 5, lane = static_cast<int>(threadIdx.x) & 31;
  const int n8 = D / 8;
  for (int64_t t0 = static_cast<int64_t>(blockIdx.x) * kMergeTokens; t0 < T;
       t0 += static_cast<int64_t>(gridDim.x) * kMergeTokens) {
    const int t = static_cast<int>(t0) + lane;
    const bool valid = t < T;
    float M = -INFINITY, S = 0.f;
    constexpr int kBatch = 8;
    if (valid)
      for (int c0 = warp; c0 < n_parts; c0 += 8 * kBatch) {
        float2 q[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
          const int c = c0 + 8 * i;
          q[i] = c < n_parts ? __ldcs(part + static_cast<size_t>(c) * T + t)
                             : make_float2(-INFINITY, 0.f);
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i) lse_fold_same(M, S, q[i].x, q[i].y);
      }
    red[warp][lane] = make_float2(M, S);
    __syncthreads();
    if (warp == 0) {
#pragma unroll
      for (int w = 1; w < 8; ++w) lse_fold_same(M, S, red[w][lane].x, red[w][lane].y);
      const float l = M + logf(S);
      const float r = CAP ? head.cap : (valid ? __ldcg(ref + t) : 0.f);
      const float alpha = expf(r - l);
      // the targets: tg.K slots and logits (z with the cap) per token
      int sl[kMaxTargets];
      float x[kMaxTargets];
      bool bad = false;
      float wsum = 0.f, acc = 0.f;
      for (int k = 0; k < tg.K; ++k) {
        sl[k] = valid ? __ldg(slot + static_cast<size_t>(k) * T + t) : 0;
        x[k] = valid ? __ldcg(tgt + static_cast<size_t>(k) * T + t) : 0.f;
        bad |= valid && static_cast<unsigned>(sl[k]) >= static_cast<unsigned>(C);
        wsum += tg.w[k];
        acc += tg.w[k] * (l - x[k]);
      }
      // 0 marks a token whose H row is not scaled (beyond T, or a bad slot)
      s_alpha[lane] = valid && !bad ? alpha : 0.f;
      if (valid) {
        if (bad) {
          set_status(status, SS_ERR_INDEX);
        } else {
          lse[t] = l;
          loss[t] = acc;
          rowfac[t] = scale * wsum * alpha;
          if (!CAP && !(l - r <= kStoredSpan)) {
            *fallback = 1;
          } else {
            // each target column: exp(x - r) - (w / W) exp(lse - r), w the summed
            // weight of every target on that column (times dz/ds with the cap)
            const float el = expf(l - r);
            for (int k = 0; k < tg.K; ++k) {
              float wt = 0.f;
              for (int k2 = 0; k2 < tg.K; ++k2) wt += sl[k2] == sl[k] ? tg.w[k2] : 0.f;
              float g = expf(x[k] - r) - wt / wsum * el;
              if (CAP) g *= x[k] * (head.cap - x[k]) * head.icap_tau;
              Pt[static_cast<int64_t>(t) * ldP + sl[k]] = bf16_bits(g);
            }
          }
        }
      }
    }
    __syncthreads();
    // Hs rows of the block's tokens: 16-byte pieces p of the contiguous block
    const int nt = T - t0 < kMergeTokens ? static_cast<int>(T - t0) : kMergeTokens;
    const int pieces = nt * n8;
    const uint4* src = reinterpret_cast<const uint4*>(H + t0 * D);
    uint4* dst = reinterpret_cast<uint4*>(Hs + t0 * D);
    constexpr int kHB = 4;
    for (int p0 = static_cast<int>(threadIdx.x); p0 < pieces; p0 += 256 * kHB) {
      uint4 v[kHB];
#pragma unroll
      for (int i = 0; i < kHB; ++i) {
        const int p = p0 + 256 * i;
        if (p < pieces) v[i] = __ldg(src + p);
      }
#pragma unroll
      for (int i = 0; i < kHB; ++i) {
        const int p = p0 + 256 * i;
        if (p >= pieces) continue;
        const float alpha = s_alpha[p / n8];
        if (alpha == 0.f) continue;
        const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          o[j] = pack_bf16x2(__uint_as_float(w[j] << 16) * alpha,
                             __uint_as_float(w[j] & 0xffff0000u) * alpha);
        dst[p] = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
    __syncthreads();  // red and s_alpha are reused by the next group of tokens
  }
}

// dW[cand[j], :] = 0 (the gradient of an empty batch).
__global__ void __launch_bounds__(256) k_zero_rows(const int32_t* __restrict__ cand, int C, int V,
                                                   int D, float* __restrict__ dW, int* status) {
  pdl_enter();
  if (read_status(status) != 0) return;
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * (blockDim.x / 32);
  for (int j = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32; j < C; j += warps) {
    const int v = __ldg(cand + j);
    if (static_cast<unsigned>(v) >= static_cast<unsigned>(V)) {
      if (lane == 0) set_status(status, SS_ERR_INDEX);
      continue;
    }
    float4* dst = reinterpret_cast<float4*>(dW + static_cast<size_t>(v) * D);
    for (int i = lane; i < D / 4; i += 32) dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

int rows_grid(int64_t rows, int num_sms) {
  const int64_t want = (rows + 7) / 8;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  return static_cast<int>(want < cap ? (want > 0 ? want : 1) : cap);
}

// Detail of the last failing CUDA call on this host thread (ss_last_error).
thread_local char g_err[256] = "";

ss_status fail(const char* what, cudaError_t e) {
  snprintf(g_err, sizeof g_err, "%s: %s (%d)", what, cudaGetErrorString(e), static_cast<int>(e));
  return SS_ERR_CUDA;
}

ss_status cuda_status(cudaError_t e, const char* what) {
  return e == cudaSuccess ? SS_OK : fail(what, e);
}

// ------------------------------------------------------------ launch trace

struct Trace {
  bool on = false;
  bool failed = false;
  cudaEvent_t* events = nullptr;
  int capacity = 0;
  int count = 0;
  std::vector<const char*> names;  // one per recorded entry (host memory)
  std::vector<int> kernels;        // kernel launches inside each recorded entry
  int at_pre = 0;                  // g_kernel_launches when the open entry began
};
thread_local Trace g_trace;

void trace_pre(cudaStream_t s, const char* name) {
  Trace& t = g_trace;
  if (!t.on) return;
  if (t.count < t.capacity) {
    // A failed record must not leave a pending error for the launch checks.
    if (cudaEventRecord(t.events[2 * t.count], s) != cudaSuccess) {
      (void)cudaGetLastError();
      t.failed = true;
    }
    t.names.push_back(name);
  }
  t.at_pre = g_kernel_launches;
}

void trace_post(cudaStream_t s) {
  Trace& t = g_trace;
  if (!t.on) return;
  if (t.count < t.capacity) {
    if (cudaEventRecord(t.events[2 * t.count + 1], s) != cudaSuccess) {
      (void)cudaGetLastError();
      t.failed = true;
    }
    t.kernels.push_back(g_kernel_launches - t.at_pre);
  }
  ++t.count;
}

// ------------------------------------------------- allocation-free forward
// Scratch of ss_forward_noalloc, in the library's own device data: callers
// of that entry point pass no workspace. Host code must not use this name as
// an address -- on the host it is only a stand-in; the device address comes
// from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SS_NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mu;
// The array's device address, per device, together with the context it was
// looked up in: after cudaDeviceReset (or once the primary context is
// released and created again) the module is loaded anew and the address may
// change, so a different current context means a fresh lookup.
struct NoallocAddr {
  void* ctx;
  void* addr;
};
NoallocAddr g_noalloc_addr[kMaxDevices];

using CtxGetCurrentFn = int (*)(void**);  // cuCtxGetCurrent(CUcontext*), CUDA_SUCCESS = 0

CtxGetCurrentFn ctx_get_current_fn() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

// Device address of g_noalloc_scratch on the current device, looked up with
// that device current and cached per (device, context).
cudaError_t noalloc_scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  void* ctx = nullptr;
  CtxGetCurrentFn get_ctx = ctx_get_current_fn();
  if (!get_ctx || get_ctx(&ctx) != 0) return cudaErrorDeviceUninitialized;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoallocAddr& a = g_noalloc_addr[dev];
  if (ctx == nullptr || a.addr == nullptr || a.ctx != ctx) {
    // (the lookup makes the device's primary context current if no context
    // was yet)
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    if (ctx == nullptr && (get_ctx(&ctx) != 0 || ctx == nullptr)) return cudaErrorDeviceUninitialized;
    a.ctx = ctx;
    a.addr = p;
  }
  *out = a.addr;
  return cudaSuccess;
}

// ------------------------------------------------------- launch sequences

ss_status enqueue_gather(const uint16_t* W, const int32_t* cand, int64_t C, int64_t V, int64_t D,
                         uint16_t* Wc, int* status, int nsm, cudaStream_t s,
                         float* amax = nullptr, const uint16_t* x = nullptr, int64_t x_n8 = 0,
                         float* x_amax = nullptr) {
  trace_pre(s, "gather_rows");
  const cudaError_t e =
      amax ? launch_pdl(k_gather_rows<true>, dim3(rows_grid(C, nsm)), dim3(256), 0, s, W, cand,
                        static_cast<int>(C), static_cast<int>(V), static_cast<int>(D), Wc, amax, x,
                        x_n8, x_amax, status)
           : launch_pdl(k_gather_rows<false>, dim3(rows_grid(C, nsm)), dim3(256), 0, s, W, cand,
                        static_cast<int>(C), static_cast<int>(V), static_cast<int>(D), Wc, amax, x,
                        x_n8, x_amax, status);
  trace_post(s);
  return e == cudaSuccess ? SS_OK : fail("launch k_gather_rows", e);
}

// H's e4m3 jobs: mode 1 (h8 and the rounded bf16 copy hq), mode 2 (h8 and
// the transposed h8t); tiles = 0 / n8 = 0 give the empty job
QuantJob h_rows_job(const uint16_t* H, int64_t T, int64_t D, const Layout& L, char* ws,
                    bool empty) {
  return QuantJob{H, reinterpret_cast<uint8_t*>(ws + L.h8), reinterpret_cast<uint16_t*>(ws + L.hq),
                  reinterpret_cast<const float*>(ws + L.hdr + kHdrAmax), empty ? 0 : T * D / 8};
}
QuantTJob h_tiles_job(const uint16_t* H, int64_t T, int64_t D, const Layout& L, char* ws,
                      bool empty) {
  return QuantTJob{H, reinterpret_cast<uint8_t*>(ws + L.h8),
                   reinterpret_cast<uint8_t*>(ws + L.h8t),
                   reinterpret_cast<const float*>(ws + L.hdr + kHdrAmax), static_cast<int>(T),
                   static_cast<int>(D), static_cast<int>(L.ldT8),
                   empty ? 0 : static_cast<int>((T + 63) / 64 * (D / 64))};
}

// W_c = W[cand] and, for the FP8 head, the e4m3 operands: amax of W_c and of
// H (both in the gather's launch), then H -> (h8, hq) and W_c -> (w8, W_c
// rounded in place), or (FP8 gradients) the row-major and transposed codes.
// h_beside: max |H| and H's codes come from k_h_prep_beside (ss_step), which
// zeroed nothing itself: amax and its barrier words were cleared before it.
ss_status enqueue_gather_operands(const uint16_t* W, const int32_t* cand, const uint16_t* H,
                                  int64_t T, int64_t C, int64_t V, int64_t D, int fp8,
                                  const Layout& L, char* ws, int nsm, cudaStream_t s,
                                  bool h_beside = false) {
  int* status = reinterpret_cast<int*>(ws + L.hdr);
  uint16_t* Wc = reinterpret_cast<uint16_t*>(ws + L.wc);
  if (!fp8) return enqueue_gather(W, cand, C, V, D, Wc, status, nsm, s);
  float* amax = reinterpret_cast<float*>(ws + L.hdr + kHdrAmax);
  const uint32_t* beside_fail =
      h_beside ? reinterpret_cast<const uint32_t*>(ws + L.hdr + kHdrBar) + 1 : nullptr;
  cudaError_t e = cudaSuccess;
  if (!h_beside) {
    e = cudaMemsetAsync(amax, 0, 2 * sizeof(float), s);
    if (e != cudaSuccess) return fail("cudaMemsetAsync(amax)", e);
  }
  ss_status r = h_beside ? enqueue_gather(W, cand, C, V, D, Wc, status, nsm, s, amax + 1)
                         : enqueue_gather(W, cand, C, V, D, Wc, status, nsm, s, amax + 1, H,
                                          T * D / 8, amax);
  if (r != SS_OK) return r;
  if (fp8 == 2) {  // FP8 gradients: row-major and transposed codes, no bf16 copies
    if ((T + 63) / 64 * (D / 64) > INT32_MAX / 2) return SS_ERR_UNSUPPORTED;
    const QuantTJob th = h_tiles_job(H, T, D, L, ws, h_beside);
    const QuantTJob tw{Wc, reinterpret_cast<uint8_t*>(ws + L.w8),
                       reinterpret_cast<uint8_t*>(ws + L.w8t), amax + 1, static_cast<int>(C),
                       static_cast<int>(D), static_cast<int>(L.ldC8),
                       static_cast<int>((C + 63) / 64 * (D / 64))};
    trace_pre(s, "quantize_e4m3");
    e = launch_pdl(k_quantize_e4m3_t, dim3(nsm * 4), dim3(256), 0, s, th, tw, status,
                   beside_fail);
    trace_post(s);
    return e == cudaSuccess ? SS_OK : fail("launch k_quantize_e4m3_t", e);
  }
  const QuantJob jh = h_rows_job(H, T, D, L, ws, h_beside);
  const QuantJob jw{Wc, reinterpret_cast<uint8_t*>(ws + L.w8), Wc, amax + 1, C * D / 8};
  trace_pre(s, "quantize_e4m3");
  e = launch_pdl(k_quantize_e4m3, dim3(nsm * 4), dim3(256), 0, s, jh, jw, status, beside_fail);
  trace_post(s);
  return e == cudaSuccess ? SS_OK : fail("launch k_quantize_e4m3", e);
}

// forward GEMM (LSE partials, target logit) and the LSE merge, from W_c.
ss_status enqueue_forward(const uint16_t* H, const int32_t* slot, int64_t T, int64_t C, int64_t D,
                          float cap, float tau, const Targets& tg, int fp8, float* loss,
                          float* lse, const Layout& L, char* ws, int nsm, cudaStream_t s) {
  int* status = reinterpret_cast<int*>(ws + L.hdr);
  uint16_t* Wc = reinterpret_cast<uint16_t*>(ws + L.wc);
  float2* part = reinterpret_cast<float2*>(ws + L.part);
  float* tgt = reinterpret_cast<float*>(ws + L.tgt);
  CUtensorMap tH, tWc;
  const float* amax = nullptr;
  if (fp8) {  // e4m3 copies: 128 elements = 128 bytes per row of a k-block
    amax = reinterpret_cast<const float*>(ws + L.hdr + kHdrAmax);
    if (!make_map(&tH, ws + L.h8, D, T, D, 128, 128, CU_TENSOR_MAP_DATA_TYPE_UINT8) ||
        !make_map(&tWc, ws + L.w8, D, C, D, 128, kBnLogits, CU_TENSOR_MAP_DATA_TYPE_UINT8))
      return fail("cuTensorMapEncodeTiled", cudaErrorInvalidValue);
  } else if (!make_map(&tH, H, D, T, D * 2, 64, 128) ||
             !make_map(&tWc, Wc, D, C, D * 2, 64, kBnLogits)) {
    return fail("cuTensorMapEncodeTiled", cudaErrorInvalidValue);
  }
  trace_pre(s, "gemm_forward_lse");
  const cudaError_t e = launch_forward_logits(tH, tWc, static_cast<int>(T), static_cast<int>(C),
                                              static_cast<int>(D), slot, part, tgt, cap, tau,
                                              tg, amax, status, nsm, s);
  trace_post(s);
  if (e != cudaSuccess) return fail("launch gemm_forward_lse", e);
  const int blocks = static_cast<int>((T * kMergeLanes + 255) / 256);
  trace_pre(s, "lse_merge");
  const cudaError_t em =
      launch_pdl(k_lse_merge, dim3(blocks), dim3(256), 0, s, part, tgt, slot, static_cast<int>(T),
                 static_cast<int>(C), static_cast<int>(L.n_ct * fwd_groups(cap, fp8 != 0, tg.K)), tg, loss,
                 lse, status);
  trace_post(s);
  return cuda_status(em, "launch k_lse_merge");
}

// FP8 gradients: G8 and G8^T (e5m2) from the e4m3 logits, then both gradient
// GEMMs on e5m2 x e4m3, every operand K-major
// G8's power of two: the largest e with B 2^e <= 57344 (e5m2's largest finite
// value), B the bound of |(P - Y) dz/ds|: 1 for the plain head, cap / (4 tau)
// (the largest dz/ds) for the capped head
int g8_exponent(float cap, float tau) {
  const double B = cap > 0.f ? static_cast<double>(cap) / (4.0 * tau) : 1.0;
  int k;
  std::frexp(57344.0 / B, &k);  // 57344 / B in [2^(k-1), 2^k)
  return std::max(-100, std::min(100, k - 1));
}

ss_status enqueue_backward_fp8(const int32_t* cand, const int32_t* slot, const float* lse,
                               int64_t T, int64_t V, int64_t C, int64_t D, float cap, float tau,
                               float scale, int accumulate, uint16_t* dH, float* dW,
                               const Layout& L, char* ws, int nsm, cudaStream_t s) {
  const int g8e = g8_exponent(cap, tau);
  int* status = reinterpret_cast<int*>(ws + L.hdr);
  const float* amax = reinterpret_cast<const float*>(ws + L.hdr + kHdrAmax);
  const auto u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const uint64_t ldG = static_cast<uint64_t>(L.ldG), ldT = static_cast<uint64_t>(L.ldT8),
                 ldC = static_cast<uint64_t>(L.ldC8);
  CUtensorMap tH8, tW8, tG8s, tG8ts, tG8, tW8t, tG8t, tH8t;
  const bool ok =
      make_map(&tH8, ws + L.h8, D, T, D, 128, 128, u8) &&
      make_map(&tW8, ws + L.w8, D, C, D, 128, kBnLogits, u8) &&
      make_map(&tG8s, ws + L.g, C, T, ldG, 64, 128, u8, CU_TENSOR_MAP_SWIZZLE_64B) &&
      make_map(&tG8ts, ws + L.g8t, T, C, ldT, 128, 64, u8) &&
      make_map(&tG8, ws + L.g, C, T, ldG, 128, 128, u8) &&
      make_map(&tW8t, ws + L.w8t, C, D, ldC, 128, 128, u8) &&
      make_map(&tG8t, ws + L.g8t, T, C, ldT, 128, 128, u8) &&
      make_map(&tH8t, ws + L.h8t, T, D, ldT, 128, 128, u8);
  if (!ok) return fail("cuTensorMapEncodeTiled", cudaErrorInvalidValue);
  const int iT = static_cast<int>(T), iV = static_cast<int>(V), iC = static_cast<int>(C),
            iD = static_cast<int>(D);
  trace_pre(s, "gemm_softmax_grad");
  cudaError_t e = launch_softmax_grad_fp8(tH8, tW8, tG8s, tG8ts, iT, iC, iD, slot, lse, cap, tau,
                                          g8e, amax, status, nsm, s);
  trace_post(s);
  if (e != cudaSuccess) return fail("launch gemm_softmax_grad", e);
  trace_pre(s, "gemm_grads");
  e = launch_grads_fp8(tG8, tW8t, tG8t, tH8t, iT, iC, iD, iV, accumulate, cand, scale, g8e, amax,
                       dH, dW, status, nsm, s);
  trace_post(s);
  return e == cudaSuccess ? SS_OK : fail("launch gemm_grads", e);
}

// softmax-gradient GEMM and the two gradient GEMMs, from W_c.
ss_status enqueue_backward(const uint16_t* H, const int32_t* cand, const int32_t* slot,
                           const float* lse, int64_t T, int64_t V, int64_t C, int64_t D,
                           float cap, float tau, const Targets& tg, int fp8, float scale,
                           int accumulate, uint16_t* dH, float* dW, const Layout& L, char* ws,
                           int nsm, cudaStream_t s) {
  if (fp8 == 2)
    return enqueue_backward_fp8(cand, slot, lse, T, V, C, D, cap, tau, scale, accumulate, dH, dW,
                                L, ws, nsm, s);
  int* status = reinterpret_cast<int*>(ws + L.hdr);
  uint16_t* Wc = reinterpret_cast<uint16_t*>(ws + L.wc);
  uint16_t* G = reinterpret_cast<uint16_t*>(ws + L.g);
  const int iT = static_cast<int>(T), iV = static_cast<int>(V), iC = static_cast<int>(C),
            iD = static_cast<int>(D);
  CUtensorMap tH, tWc, tWc2, tGk, tWcMn, tGmn, tHmn;
  const uint64_t gRow = static_cast<uint64_t>(L.ldG) * 2;
  // the FP8 head: the logit recompute reads the e4m3 copies, the gradient
  // GEMMs the same rounded operands in bf16 (H rounded in hq, W_c in place)
  const uint16_t* Hg = fp8 ? reinterpret_cast<const uint16_t*>(ws + L.hq) : H;
  const float* amax = fp8 ? reinterpret_cast<const float*>(ws + L.hdr + kHdrAmax) : nullptr;
  bool ok = fp8 ? make_map(&tH, ws + L.h8, D, T, D, 128, 128, CU_TENSOR_MAP_DATA_TYPE_UINT8) &&
                      make_map(&tWc, ws + L.w8, D, C, D, 128, kBnLogits,
                               CU_TENSOR_MAP_DATA_TYPE_UINT8)
                : make_map(&tH, H, D, T, D * 2, 64, 128) &&
                      make_map(&tWc, Wc, D, C, D * 2, 64, kBnLogits);
  ok = ok && make_map(&tWc2, Wc, D, C, D * 2, 64, kBnLogits / 2) &&
       make_map(&tGk, G, C, T, gRow, 64, 128) && make_map(&tWcMn, Wc, D, C, D * 2, 64, 64) &&
       make_map(&tGmn, G, C, T, gRow, 64, 64) && make_map(&tHmn, Hg, D, T, D * 2, 64, 64);
  if (!ok) return fail("cuTensorMapEncodeTiled", cudaErrorInvalidValue);
  trace_pre(s, "gemm_softmax_grad");
  cudaError_t e =
      launch_softmax_grad(tH, tWc, tWc2, tGk, iT, iC, iD, slot, lse, scale, cap, tau, tg, amax,
                          status, nsm, s);
  trace_post(s);
  if (e != cudaSuccess) return fail("launch gemm_softmax_grad", e);
  trace_pre(s, "gemm_grads");
  e = launch_grads(tGk, tWcMn, tGmn, tHmn, iT, iC, iD, iV, accumulate, cand, dH, dW, status, nsm,
                   s);
  trace_post(s);
  return e == cudaSuccess ? SS_OK : fail("launch gemm_grads", e);
}

// ss_step with the plain bf16 head and one target: the forward keeps the
// probabilities exp(S - r) (EpiFwdP) and the gradient GEMMs read them, so
// the logits are computed once per step. The merge patches the target column
// and writes the per-row factors; the softmax-gradient GEMM (the recompute,
// G = P - Y) runs only if the merge raised the fallback flag, and then also
// sets Hs = H and the row factors to `scale`. The regions: Pt in G's
// place, r and the dH row factors after the target logits, Hs = alpha H in
// the place of the FP8 head's rounded H.
// hc: the capped head (cap <= kStoredCapMax), or cap 0 for the plain head;
// tg: the targets per token and their weights
ss_status enqueue_step_stored(const uint16_t* H, const int32_t* cand, const int32_t* slot,
                              int64_t T, int64_t V, int64_t C, int64_t D, const HeadCap& hc,
                              const Targets& tg, float scale, int accumulate, float* loss,
                              float* lse, uint16_t* dH, float* dW, const Layout& L, char* ws,
                              int nsm, cudaStream_t s) {
  const bool capped = hc.cap > 0.f;
  int* status = reinterpret_cast<int*>(ws + L.hdr);
  int* fallback = reinterpret_cast<int*>(ws + L.hdr + kHdrFallback);
  uint16_t* Wc = reinterpret_cast<uint16_t*>(ws + L.wc);
  uint16_t* P = reinterpret_cast<uint16_t*>(ws + L.g);
  float2* part = reinterpret_cast<float2*>(ws + L.part);
  float* tgt = reinterpret_cast<float*>(ws + L.tgt);  // [K, T]
  float* ref = tgt + kMaxTargets * T;
  float* rowfac = ref + T;
  uint16_t* Hs = reinterpret_cast<uint16_t*>(ws + L.hq);
  const int iT = static_cast<int>(T), iV = static_cast<int>(V), iC = static_cast<int>(C),
            iD = static_cast<int>(D);
  const uint64_t pRow = static_cast<uint64_t>(L.ldG) * 2;
  CUtensorMap tH, tWc, tWc2, tPk, tWcMn, tPmn, tHsMn;
  const bool ok = make_map(&tH, H, D, T, D * 2, 64, 128) &&
                  make_map(&tWc, Wc, D, C, D * 2, 64, kBnLogits) &&
                  make_map(&tWc2, Wc, D, C, D * 2, 64, kBnLogits / 2) &&
                  make_map(&tPk, P, C, T, pRow, 64, 128) &&
                  make_map(&tWcMn, Wc, D, C, D * 2, 64, 64) &&
                  make_map(&tPmn, P, C, T, pRow, 64, 64) &&
                  make_map(&tHsMn, Hs, D, T, D * 2, 64, 64);
  if (!ok) return fail("cuTensorMapEncodeTiled", cudaErrorInvalidValue);
  trace_pre(s, "gemm_forward_lse");
  cudaError_t e = launch_forward_stored(tH, tWc, tWc2, tPk, iT, iC, iD, slot, part, tgt, ref,
                                        fallback, hc, tg, status, nsm, s);
  trace_post(s);
  if (e != cudaSuccess) return fail("launch gemm_forward_lse", e);
  trace_pre(s, "lse_merge");
  const dim3 merge_grid(static_cast<unsigned>((T + kMergeTokens - 1) / kMergeTokens));
  e = capped ? launch_pdl(k_lse_merge_p<true>, merge_grid, dim3(256), 0, s, part, tgt, slot, ref,
                          iT, iC, static_cast<int>(L.n_ct * 2), H, iD, scale, P,
                          static_cast<int64_t>(L.ldG), Hs, rowfac, fallback, loss, lse, status,
                          hc, tg)
             : launch_pdl(k_lse_merge_p<false>, merge_grid, dim3(256), 0, s, part, tgt, slot, ref,
                          iT, iC, static_cast<int>(L.n_ct * 2), H, iD, scale, P,
                          static_cast<int64_t>(L.ldG), Hs, rowfac, fallback, loss, lse, status,
                          hc, tg);
  trace_post(s);
  if (e != cudaSuccess) return fail("launch k_lse_merge_p", e);
  // the capped head's lse lies within ln C of its reference: no fallback
  if (!capped) {
    trace_pre(s, "gemm_softmax_grad");
    e = launch_softmax_grad_gated(tH, tWc, tWc2, tPk, iT, iC, iD, slot, lse, fallback, H, Hs,
                                  rowfac, tg, scale, status, nsm, s);
    trace_post(s);
    if (e != cudaSuccess) return fail("launch gemm_softmax_grad", e);
  }
  trace_pre(s, "gemm_grads");
  // dW_c = scale W (Pt'^T . Hs), W the targets' summed weight
  float dw_scale = 0.f;
  for (int k = 0; k < tg.K; ++k) dw_scale += tg.w[k];
  dw_scale *= scale;
  e = launch_grads(tPk, tWcMn, tPmn, tHsMn, iT, iC, iD, iV, accumulate, cand, dH, dW, status, nsm,
                   s, rowfac, &dw_scale);
  trace_post(s);
  return e == cudaSuccess ? SS_OK : fail("launch gemm_grads", e);
}

ss_status enqueue_zero_rows(const int32_t* cand, int64_t C, int64_t V, int64_t D, float* dW,
                            int* status, int nsm, cudaStream_t s) {
  trace_pre(s, "zero_rows");
  const cudaError_t e = launch_pdl(k_zero_rows, dim3(rows_grid(C, nsm)), dim3(256), 0, s, cand,
                                   static_cast<int>(C), static_cast<int>(V), static_cast<int>(D),
                                   dW, status);
  trace_post(s);
  return cuda_status(e, "launch k_zero_rows");
}

constexpr Targets kOneTarget = {1, {1.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f}};

// The argument checks of ss_step (and of ss_step_graph_create).
ss_status step_args_status(const int32_t* targets, const uint16_t* H, const uint16_t* W,
                           int64_t T, int64_t V, int64_t C, int64_t D, int accumulate,
                           const int32_t* cand, const int32_t* slot, const float* loss,
                           const float* lse, const uint16_t* dH, const float* dW,
                           const void* workspace, size_t workspace_bytes) {
  const ss_status st = check_sizes(T, V, C, D);
  if (st != SS_OK) return st;
  if (!W || !cand || !dW || !workspace ||
      (T > 0 && (!targets || !H || !slot || !loss || !lse || !dH)))
    return SS_ERR_INVALID;
  if (!aligned(targets, 4) || !aligned(H, 16) || !aligned(W, 16) || !aligned(dH, 16) ||
      !aligned(dW, 16) || !aligned(workspace, 16) || !aligned(cand, 4) || !aligned(slot, 4) ||
      !aligned(loss, 4) || !aligned(lse, 4))
    return SS_ERR_INVALID;
  if (accumulate != 0 && accumulate != 1) return SS_ERR_INVALID;
  if (workspace_bytes < make_layout(T, C, D).total) return SS_ERR_WORKSPACE;
  return SS_OK;
}

}  // namespace

cudaError_t prepare_kernel(const void* kern, int dyn_smem_bytes) {
  struct Done {
    const void* kern;
    int dev, smem;
  };
  static std::mutex mu;
  static std::vector<Done> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  Done* d = nullptr;
  for (auto& x : done)
    if (x.kern == kern && x.dev == dev) d = &x;
  if (d && d->smem >= dyn_smem_bytes) return cudaSuccess;
  if (dyn_smem_bytes > 0) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_smem_bytes);
    if (e != cudaSuccess) return e;
  }
  if (d) {
    d->smem = dyn_smem_bytes;
    return cudaSuccess;
  }
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  done.push_back(Done{kern, dev, dyn_smem_bytes});
  return cudaSuccess;
}

}  // namespace ss

using namespace ss;

// A captured ss_step: the graph, its executable, and the candidate kernel's
// node with the argument values it is launched with (only `seed` changes).
struct ss_step_graph {
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  cudaGraphNode_t cand_node = nullptr;
  cudaKernelNodeParams base = {};
  const int32_t* targets = nullptr;
  int T = 0, V = 0, C = 0;
  uint64_t seed = 0;
  int32_t* cand = nullptr;
  int32_t* slot = nullptr;
  int* hdr = nullptr;
  void* args[8] = {};
};

extern "C" {

size_t ss_workspace_size(int64_t T, int64_t V, int64_t C, int64_t D) {
  if (check_sizes(T, V, C, D) != SS_OK) return 0;
  return make_layout(T, C, D).total;
}

ss_status ss_build_candidates(const int32_t* targets, int64_t T, int64_t V, int64_t C,
                              uint64_t seed, int32_t* cand, int32_t* slot, int32_t* U_host,
                              void* workspace, size_t workspace_bytes, ss_stream stream) {
  const ss_status st = check_sizes(T, V, C, 64);
  if (st != SS_OK) return st;
  if ((T > 0 && (!targets || !slot)) || !cand || !workspace) return SS_ERR_INVALID;
  if (!aligned(targets, 4) || !aligned(cand, 4) || !aligned(slot, 4) || !aligned(workspace, 16))
    return SS_ERR_INVALID;
  if (workspace_bytes < kHdrBytes) return SS_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* hdr = static_cast<int*>(workspace);
  // the kernel clears the status word before anything else
  trace_pre(s, "build_candidates");
  cudaError_t e = launch_build_candidates(targets, static_cast<int>(T), static_cast<int>(V),
                                                static_cast<int>(C), seed, cand, slot, hdr, s);
  trace_post(s);
  if (e != cudaSuccess) return fail("launch k_build_candidates", e);
  if (U_host) {
    int32_t h[2] = {0, 0};
    e = cudaMemcpyAsync(h, hdr, sizeof h, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return fail("read status after candidate build", e);
    *U_host = h[1];
    return static_cast<ss_status>(h[0]);
  }
  return SS_OK;
}

static ss_status forward_impl(const uint16_t* H, const uint16_t* W, const int32_t* cand,
                              const int32_t* slot, int64_t T, int64_t V, int64_t C, int64_t D,
                              float cap, float tau, const Targets& tg, int fp8, float* loss,
                              float* lse, void* workspace, size_t workspace_bytes,
                              ss_stream stream) {
  const ss_status st = check_sizes(T, V, C, D);
  if (st != SS_OK) return st;
  if (!W || !cand || !workspace || (T > 0 && (!H || !slot || !loss || !lse)))
    return SS_ERR_INVALID;
  if (!aligned(H, 16) || !aligned(W, 16) || !aligned(workspace, 16) || !aligned(cand, 4) ||
      !aligned(slot, 4) || !aligned(loss, 4) || !aligned(lse, 4))
    return SS_ERR_INVALID;
  const Layout L = make_layout(T, C, D);
  if (workspace_bytes < L.total) return SS_ERR_WORKSPACE;
  if (T == 0) return SS_OK;
  const int nsm = num_sms_current();
  if (nsm <= 0) return fail("cudaGetDevice/cudaDeviceGetAttribute", cudaGetLastError());
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  const ss_status sg = enqueue_gather_operands(W, cand, H, T, C, V, D, fp8, L, ws, nsm, s);
  if (sg != SS_OK) return sg;
  return enqueue_forward(H, slot, T, C, D, cap, tau, tg, fp8, loss, lse, L, ws, nsm, s);
}

static ss_status backward_impl(const uint16_t* H, const uint16_t* W, const int32_t* cand,
                               const int32_t* slot, const float* lse, int64_t T, int64_t V,
                               int64_t C, int64_t D, float cap, float tau, const Targets& tg,
                               int fp8, float scale, int accumulate, uint16_t* dH, float* dW,
                               void* workspace, size_t workspace_bytes, ss_stream stream) {
  const ss_status st = check_sizes(T, V, C, D);
  if (st != SS_OK) return st;
  if (!W || !cand || !dW || !workspace || (T > 0 && (!H || !slot || !lse || !dH)))
    return SS_ERR_INVALID;
  if (!aligned(H, 16) || !aligned(W, 16) || !aligned(dH, 16) || !aligned(dW, 16) ||
      !aligned(workspace, 16) || !aligned(cand, 4) || !aligned(slot, 4) || !aligned(lse, 4))
    return SS_ERR_INVALID;
  if (accumulate != 0 && accumulate != 1) return SS_ERR_INVALID;
  const Layout L = make_layout(T, C, D);
  if (workspace_bytes < L.total) return SS_ERR_WORKSPACE;
  const int nsm = num_sms_current();
  if (nsm <= 0) return fail("cudaGetDevice/cudaDeviceGetAttribute", cudaGetLastError());
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  int* status = reinterpret_cast<int*>(ws + L.hdr);
  if (T == 0) return accumulate ? SS_OK : enqueue_zero_rows(cand, C, V, D, dW, status, nsm, s);
  const ss_status sg = enqueue_gather_operands(W, cand, H, T, C, V, D, fp8, L, ws, nsm, s);
  if (sg != SS_OK) return sg;
  return enqueue_backward(H, cand, slot, lse, T, V, C, D, cap, tau, tg, fp8, scale, accumulate, dH,
                          dW, L, ws, nsm, s);
}

static ss_status step_impl(const int32_t* targets, const uint16_t* H, const uint16_t* W,
                           int64_t T, int64_t V, int64_t C, int64_t D, uint64_t seed, float cap,
                           float tau, const Targets& tg, int fp8, float scale, int accumulate,
                           int32_t* cand, int32_t* slot, float* loss, float* lse, uint16_t* dH,
                           float* dW, void* workspace, size_t workspace_bytes, ss_stream stream) {
  const ss_status st = step_args_status(targets, H, W, T, V, C, D, accumulate, cand, slot, loss,
                                        lse, dH, dW, workspace, workspace_bytes);
  if (st != SS_OK) return st;
  if (T * tg.K >= (int64_t(1) << 31)) return SS_ERR_UNSUPPORTED;
  const Layout L = make_layout(T, C, D);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  // the FP8 head: max |H| and H's e4m3 codes depend on no candidate, so they
  // are made beside the candidate build (one cluster of 8 SMs); the amax and
  // barrier words are zeroed before it
  float* amax = reinterpret_cast<float*>(ws + L.hdr + kHdrAmax);
  const bool h_beside = fp8 != 0 && T > 0;
  if (h_beside) {
    if ((T + 63) / 64 * (D / 64) > INT32_MAX / 2) return SS_ERR_UNSUPPORTED;
    static_assert(kHdrBar == kHdrAmax + 8, "one memset clears amax[2] and bar[2]");
    const cudaError_t e = cudaMemsetAsync(amax, 0, 16, s);
    if (e != cudaSuccess) return fail("cudaMemsetAsync(amax)", e);
  }
  // the candidate set covers every target of every token (targets [K, T])
  const ss_status sb = ss_build_candidates(targets, T * tg.K, V, C, seed, cand, slot, nullptr,
                                           workspace, workspace_bytes, stream);
  if (sb != SS_OK) return sb;
  const int nsm = num_sms_current();
  if (nsm <= 0) return fail("cudaGetDevice/cudaDeviceGetAttribute", cudaGetLastError());
  int* status = reinterpret_cast<int*>(ws + L.hdr);
  if (T == 0) return accumulate ? SS_OK : enqueue_zero_rows(cand, C, V, D, dW, status, nsm, s);
  if (h_beside) {
    trace_pre(s, "prepare_h");
    const int grid = 4 * nsm;
    const cudaError_t e = launch_pdl(
        k_h_prep_beside, dim3(grid), dim3(256), 0, s, T * D / 8, amax,
        reinterpret_cast<uint32_t*>(ws + L.hdr + kHdrBar),
        static_cast<uint32_t>(grid + SS_BESIDE_EXTRA_ARRIVALS),
        static_cast<uint64_t>(SS_BESIDE_WAIT_NS), h_rows_job(H, T, D, L, ws, false),
        h_tiles_job(H, T, D, L, ws, false), fp8);
    trace_post(s);
    if (e != cudaSuccess) return fail("launch k_h_prep_beside", e);
  }
  // one gather of W[cand] serves the forward and the backward
  ss_status r = enqueue_gather_operands(W, cand, H, T, C, V, D, fp8, L, ws, nsm, s, h_beside);
  if (r != SS_OK) return r;
  // the bf16 head keeps the forward's probabilities: the plain head, and
  // the capped head up to kStoredCapMax, any targets per token
  if (fp8 == 0 && !(cap > kStoredCapMax))
    return enqueue_step_stored(H, cand, slot, T, V, C, D, head_cap(cap, tau), tg, scale,
                               accumulate, loss, lse, dH, dW, L, ws, nsm, s);
  r = enqueue_forward(H, slot, T, C, D, cap, tau, tg, fp8, loss, lse, L, ws, nsm, s);
  if (r != SS_OK) return r;
  return enqueue_backward(H, cand, slot, lse, T, V, C, D, cap, tau, tg, fp8, scale, accumulate, dH,
                          dW, L, ws, nsm, s);
}

// K targets per token with host weights w[0..K): 1 <= K <= kMaxTargets, each
// w[k] finite and >= 0, their sum > 0
static ss_status targets_args(int64_t K, const float* w, Targets* tg) {
  if (K < 1 || K > kMaxTargets || !w) return SS_ERR_INVALID;
  float sum = 0.f;
  *tg = Targets{static_cast<int>(K), {}};
  for (int64_t k = 0; k < K; ++k) {
    if (!(w[k] >= 0.f) || !std::isfinite(w[k])) return SS_ERR_INVALID;
    tg->w[k] = w[k];
    sum += w[k];
  }
  return sum > 0.f && std::isfinite(sum) ? SS_OK : SS_ERR_INVALID;
}

// the head options: NULL or cap == 0 is the plain head; fp8 = 1 or 2 (plain
// logits only) sets *fp8
static ss_status head_args(const ss_head* head, float* cap, float* tau, int* fp8 = nullptr) {
  *cap = 0.f;
  *tau = 1.f;
  if (fp8) *fp8 = 0;
  if (head && head->fp8 != 0) {
    if (head->fp8 != 1 && head->fp8 != 2) return SS_ERR_INVALID;
    if (!fp8) return SS_ERR_UNSUPPORTED;  // this entry point has no FP8 path
    *fp8 = head->fp8;
  }
  if (!head || head->cap == 0.f) return SS_OK;
  if (!(head->cap > 0.f) || !std::isfinite(head->cap) || !(head->tau > 0.f) ||
      !std::isfinite(head->tau))
    return SS_ERR_INVALID;
  *cap = head->cap;
  *tau = head->tau;
  return SS_OK;
}

ss_status ss_forward(const uint16_t* H, const uint16_t* W, const int32_t* cand,
                     const int32_t* slot, int64_t T, int64_t V, int64_t C, int64_t D,
                     float* loss, float* lse, void* workspace, size_t workspace_bytes,
                     ss_stream stream) {
  return forward_impl(H, W, cand, slot, T, V, C, D, 0.f, 1.f, kOneTarget, false, loss, lse,
                      workspace, workspace_bytes, stream);
}

ss_status ss_forward_head(const uint16_t* H, const uint16_t* W, const int32_t* cand,
                          const int32_t* slot, int64_t T, int64_t V, int64_t C, int64_t D,
                          const ss_head* head, float* loss, float* lse, void* workspace,
                          size_t workspace_bytes, ss_stream stream) {
  float cap, tau;
  int fp8;
  const ss_status h = head_args(head, &cap, &tau, &fp8);
  if (h != SS_OK) return h;
  if (fp8 && D % 128 != 0) return SS_ERR_UNSUPPORTED;
  return forward_impl(H, W, cand, slot, T, V, C, D, cap, tau, kOneTarget, fp8, loss, lse,
                      workspace, workspace_bytes, stream);
}

ss_status ss_backward(const uint16_t* H, const uint16_t* W, const int32_t* cand,
                      const int32_t* slot, const float* lse, int64_t T, int64_t V, int64_t C,
                      int64_t D, float scale, int accumulate, uint16_t* dH, float* dW,
                      void* workspace, size_t workspace_bytes, ss_stream stream) {
  return backward_impl(H, W, cand, slot, lse, T, V, C, D, 0.f, 1.f, kOneTarget, false, scale,
                       accumulate, dH, dW, workspace, workspace_bytes, stream);
}

ss_status ss_backward_head(const uint16_t* H, const uint16_t* W, const int32_t* cand,
                           const int32_t* slot, const float* lse, int64_t T, int64_t V,
                           int64_t C, int64_t D, const ss_head* head, float scale,
                           int accumulate, uint16_t* dH, float* dW, void* workspace,
                           size_t workspace_bytes, ss_stream stream) {
  float cap, tau;
  int fp8;
  const ss_status h = head_args(head, &cap, &tau, &fp8);
  if (h != SS_OK) return h;
  if (fp8 && D % 128 != 0) return SS_ERR_UNSUPPORTED;
  return backward_impl(H, W, cand, slot, lse, T, V, C, D, cap, tau, kOneTarget, fp8, scale,
                       accumulate, dH, dW, workspace, workspace_bytes, stream);
}

ss_status ss_step(const int32_t* targets, const uint16_t* H, const uint16_t* W, int64_t T,
                  int64_t V, int64_t C, int64_t D, uint64_t seed, float scale, int accumulate,
                  int32_t* cand, int32_t* slot, float* loss, float* lse, uint16_t* dH, float* dW,
                  void* workspace, size_t workspace_bytes, ss_stream stream) {
  return step_impl(targets, H, W, T, V, C, D, seed, 0.f, 1.f, kOneTarget, false, scale, accumulate,
                   cand, slot, loss, lse, dH, dW, workspace, workspace_bytes, stream);
}

ss_status ss_step_head(const int32_t* targets, const uint16_t* H, const uint16_t* W, int64_t T,
                       int64_t V, int64_t C, int64_t D, uint64_t seed, const ss_head* head,
                       float scale, int accumulate, int32_t* cand, int32_t* slot, float* loss,
                       float* lse, uint16_t* dH, float* dW, void* workspace,
                       size_t workspace_bytes, ss_stream stream) {
  float cap, tau;
  int fp8;
  const ss_status h = head_args(head, &cap, &tau, &fp8);
  if (h != SS_OK) return h;
  if (fp8 && D % 128 != 0) return SS_ERR_UNSUPPORTED;
  return step_impl(targets, H, W, T, V, C, D, seed, cap, tau, kOneTarget, fp8, scale, accumulate,
                   cand, slot, loss, lse, dH, dW, workspace, workspace_bytes, stream);
}

ss_status ss_forward_mtp(const uint16_t* H, const uint16_t* W, const int32_t* cand,
                         const int32_t* slot, int64_t K, const float* weights, int64_t T,
                         int64_t V, int64_t C, int64_t D, const ss_head* head, float* loss,
                         float* lse, void* workspace, size_t workspace_bytes, ss_stream stream) {
  float cap, tau;
  Targets tg;
  ss_status a = head_args(head, &cap, &tau);
  if (a == SS_OK) a = targets_args(K, weights, &tg);
  if (a != SS_OK) return a;
  return forward_impl(H, W, cand, slot, T, V, C, D, cap, tau, tg, false, loss, lse, workspace,
                      workspace_bytes, stream);
}

ss_status ss_backward_mtp(const uint16_t* H, const uint16_t* W, const int32_t* cand,
                          const int32_t* slot, int64_t K, const float* weights, const float* lse,
                          int64_t T, int64_t V, int64_t C, int64_t D, const ss_head* head,
                          float scale, int accumulate, uint16_t* dH, float* dW, void* workspace,
                          size_t workspace_bytes, ss_stream stream) {
  float cap, tau;
  Targets tg;
  ss_status a = head_args(head, &cap, &tau);
  if (a == SS_OK) a = targets_args(K, weights, &tg);
  if (a != SS_OK) return a;
  return backward_impl(H, W, cand, slot, lse, T, V, C, D, cap, tau, tg, false, scale, accumulate,
                       dH, dW, workspace, workspace_bytes, stream);
}

ss_status ss_step_mtp(const int32_t* targets, int64_t K, const float* weights, const uint16_t* H,
                      const uint16_t* W, int64_t T, int64_t V, int64_t C, int64_t D, uint64_t seed,
                      const ss_head* head, float scale, int accumulate, int32_t* cand,
                      int32_t* slot, float* loss, float* lse, uint16_t* dH, float* dW,
                      void* workspace, size_t workspace_bytes, ss_stream stream) {
  float cap, tau;
  Targets tg;
  ss_status a = head_args(head, &cap, &tau);
  if (a == SS_OK) a = targets_args(K, weights, &tg);
  if (a != SS_OK) return a;
  return step_impl(targets, H, W, T, V, C, D, seed, cap, tau, tg, false, scale, accumulate, cand,
                   slot, loss, lse, dH, dW, workspace, workspace_bytes, stream);
}

int64_t ss_schedule_candidates(int64_t step, int64_t total_steps, int64_t V) {
  if (V < 1 || V > SS_MAX_V || total_steps < 1 || step < 0 || step >= total_steps) return -1;
  const int64_t sampled = total_steps > SS_SCHEDULE_FULL_STEPS
                              ? total_steps - SS_SCHEDULE_FULL_STEPS
                              : 0;
  if (step >= sampled) return V;
  static const int64_t kPhaseC[3] = {10240, 14336, 24576};
  const int64_t c = kPhaseC[(3 * step) / sampled];
  return c < V ? c : V;
}

ss_status ss_quantize_e4m3(const uint16_t* x, int64_t n, uint8_t* q, uint16_t* xq,
                           void* workspace, size_t workspace_bytes, ss_stream stream) {
  if (n < 0 || n % 8 != 0) return SS_ERR_INVALID;
  if (n == 0) return SS_OK;
  if (!x || !q || !xq || !workspace || !aligned(x, 16) || !aligned(q, 8) || !aligned(xq, 16) ||
      !aligned(workspace, 16))
    return SS_ERR_INVALID;
  if (workspace_bytes < kHdrBytes) return SS_ERR_WORKSPACE;
  const int nsm = num_sms_current();
  if (nsm <= 0) return fail("cudaGetDevice/cudaDeviceGetAttribute", cudaGetLastError());
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  // A status word of its own, cleared with amax: the call neither depends on
  // nor disturbs the status of the steps that share the workspace.
  float* amax = reinterpret_cast<float*>(ws + kHdrQuant);
  int* status = reinterpret_cast<int*>(ws + kHdrQuant + 4);
  cudaError_t e = cudaMemsetAsync(amax, 0, 8, s);
  if (e == cudaSuccess)
    e = launch_pdl(k_amax_bf16, dim3(nsm * 2), dim3(256), 0, s, x, n / 8, amax, status);
  const QuantJob j{x, q, xq, amax, n / 8};
  const QuantJob none{x, q, xq, amax, 0};
  if (e == cudaSuccess)
    e = launch_pdl(k_quantize_e4m3, dim3(nsm * 4), dim3(256), 0, s, j, none, status,
                   static_cast<const uint32_t*>(nullptr));
  return e == cudaSuccess ? SS_OK : fail("ss_quantize_e4m3", e);
}

ss_status ss_clear_rows(const int32_t* rows, int64_t n, int64_t V, int64_t D, float* dW,
                        void* workspace, size_t workspace_bytes, ss_stream stream) {
  if (n < 0 || V < 1 || n > V || D <= 0) return SS_ERR_INVALID;
  if (V > SS_MAX_V || D < 64 || D % 64 != 0 || D > SS_MAX_D) return SS_ERR_UNSUPPORTED;
  if (n == 0) return SS_OK;
  if (!rows || !dW || !workspace || !aligned(rows, 4) || !aligned(dW, 16) ||
      !aligned(workspace, 16))
    return SS_ERR_INVALID;
  if (workspace_bytes < kHdrBytes) return SS_ERR_WORKSPACE;
  const int nsm = num_sms_current();
  if (nsm <= 0) return fail("cudaGetDevice/cudaDeviceGetAttribute", cudaGetLastError());
  return enqueue_zero_rows(rows, n, V, D, dW, static_cast<int*>(workspace), nsm,
                           static_cast<cudaStream_t>(stream));
}

ss_status ss_forward_noalloc(const uint16_t* H, const uint16_t* W, const int32_t* cand,
                             const int32_t* slot, int64_t T, int64_t V, int64_t C, int64_t D,
                             float* loss, float* lse, int32_t* status_host, ss_stream stream) {
  const ss_status st = check_sizes(T, V, C, D);
  if (st != SS_OK) return st;
  if (!W || !cand || (T > 0 && (!H || !slot || !loss || !lse))) return SS_ERR_INVALID;
  if (!aligned(H, 16) || !aligned(W, 16) || !aligned(cand, 4) || !aligned(slot, 4) ||
      !aligned(loss, 4) || !aligned(lse, 4))
    return SS_ERR_INVALID;
  // Everything up to the G region of the ordinary workspace: header, W_c,
  // forward partials, target logits.
  const Layout L = make_layout(T, C, D);
  const size_t need = L.g;
  if (need > SS_NOALLOC_SCRATCH_BYTES) {
    snprintf(g_err, sizeof g_err,
             "ss_forward_noalloc: T=%lld C=%lld D=%lld needs %zu bytes of scratch, the fixed "
             "array holds %u",
             static_cast<long long>(T), static_cast<long long>(C), static_cast<long long>(D),
             need, static_cast<unsigned>(SS_NOALLOC_SCRATCH_BYTES));
    return SS_ERR_UNSUPPORTED;
  }
  if (T == 0) {
    if (status_host) *status_host = SS_OK;
    return SS_OK;
  }
  const int nsm = num_sms_current();
  if (nsm <= 0) return fail("cudaGetDevice/cudaDeviceGetAttribute", cudaGetLastError());
  void* base = nullptr;
  cudaError_t e = noalloc_scratch_address(&base);
  if (e != cudaSuccess) return fail("cudaGetSymbolAddress(scratch)", e);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(base);
  int* status = reinterpret_cast<int*>(ws + L.hdr);
  uint16_t* Wc = reinterpret_cast<uint16_t*>(ws + L.wc);
  float2* part = reinterpret_cast<float2*>(ws + L.part);
  float* tgt = reinterpret_cast<float*>(ws + L.tgt);

  // The array keeps the previous call's contents: the status word must start
  // at zero; W_c, the partials and the target logits are overwritten before
  // they are read.
  e = cudaMemsetAsync(status, 0, 2 * sizeof(int), s);
  if (e != cudaSuccess) return fail("cudaMemsetAsync(scratch status)", e);
  trace_pre(s, "gather_rows");
  cudaError_t eg = launch_pdl(k_gather_rows<false>, dim3(rows_grid(C, nsm)), dim3(256), 0, s, W, cand,
                              static_cast<int>(C), static_cast<int>(V), static_cast<int>(D), Wc,
                              static_cast<float*>(nullptr), static_cast<const uint16_t*>(nullptr),
                              int64_t(0), static_cast<float*>(nullptr), status);
  trace_post(s);
  if (eg != cudaSuccess) return fail("launch k_gather_rows", eg);
  CUtensorMap tH, tWc;
  if (!make_map(&tH, H, D, T, D * 2, 64, 128) || !make_map(&tWc, Wc, D, C, D * 2, 64, kBnLogits))
    return fail("cuTensorMapEncodeTiled", cudaErrorInvalidValue);
  trace_pre(s, "gemm_forward_lse");
  e = launch_forward_logits(tH, tWc, static_cast<int>(T), static_cast<int>(C),
                            static_cast<int>(D), slot, part, tgt, 0.f, 1.f, kOneTarget, nullptr,
                            status, nsm, s);
  trace_post(s);
  if (e != cudaSuccess) return fail("launch gemm_forward_lse", e);
  trace_pre(s, "lse_merge");
  e = launch_pdl(k_lse_merge, dim3(static_cast<int>((T * kMergeLanes + 255) / 256)), dim3(256), 0, s,
                 part, tgt, slot, static_cast<int>(T), static_cast<int>(C),
                 static_cast<int>(L.n_ct * fwd_groups(0.f)), kOneTarget, loss, lse, status);
  trace_post(s);
  if (e != cudaSuccess) return fail("launch k_lse_merge", e);
  if (status_host) {
    int32_t h[2] = {0, 0};
    e = cudaMemcpyAsync(h, status, sizeof h, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return fail("read scratch status", e);
    *status_host = h[0];
    return static_cast<ss_status>(h[0]);
  }
  return SS_OK;
}

ss_status ss_read_status(const void* workspace, size_t workspace_bytes, ss_stream stream,
                         int32_t* device_status_host, int32_t* U_status_host) {
  if (!workspace || !aligned(workspace, 16)) return SS_ERR_INVALID;
  if (workspace_bytes < kHdrBytes) return SS_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t h[2] = {0, 0};
  cudaError_t e = cudaMemcpyAsync(h, workspace, sizeof h, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail("ss_read_status", e);
  if (device_status_host) *device_status_host = h[0];
  if (U_status_host) *U_status_host = h[1];
  return static_cast<ss_status>(h[0]);
}

ss_status ss_trace_begin(void** events, int capacity) {
  if (capacity < 0 || (capacity > 0 && !events)) return SS_ERR_INVALID;
  Trace& t = g_trace;
  t.on = true;
  t.events = reinterpret_cast<cudaEvent_t*>(events);
  t.capacity = capacity;
  t.count = 0;
  t.failed = false;
  t.names.clear();
  t.kernels.clear();
  return SS_OK;
}

int ss_trace_end(void) {
  Trace& t = g_trace;
  t.on = false;
  return t.failed ? -1 : t.count;
}

const char* ss_trace_kernel_name(int k) {
  const Trace& t = g_trace;
  if (k < 0 || k >= t.count || k >= static_cast<int>(t.names.size())) return nullptr;
  return t.names[k];
}

int ss_trace_kernel_launches(int k) {
  const Trace& t = g_trace;
  if (k < 0 || k >= t.count || k >= static_cast<int>(t.kernels.size())) return -1;
  return t.kernels[k];
}

}  // extern "C"

// Capture step_impl on a private stream into a graph and find the candidate
// kernel's node (the only one whose arguments change between replays: seed).
static ss_status graph_create(const int32_t* targets, const Targets& tg, const uint16_t* H,
                              const uint16_t* W, int64_t T, int64_t V, int64_t C, int64_t D,
                              float cap, float tau, int fp8, float scale, int accumulate,
                              int32_t* cand, int32_t* slot, float* loss, float* lse, uint16_t* dH,
                              float* dW, void* workspace, size_t workspace_bytes,
                              ss_step_graph** graph) {
  if (fp8 && D % 128 != 0) return SS_ERR_UNSUPPORTED;
  ss_status st = step_args_status(targets, H, W, T, V, C, D, accumulate, cand, slot, loss, lse,
                                  dH, dW, workspace, workspace_bytes);
  if (st != SS_OK) return st;
  if (T * tg.K >= (int64_t(1) << 31)) return SS_ERR_UNSUPPORTED;
  cudaStream_t cs = nullptr;
  cudaError_t e = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking);
  if (e != cudaSuccess) return fail("cudaStreamCreateWithFlags", e);
  e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeRelaxed);
  if (e != cudaSuccess) {
    cudaStreamDestroy(cs);
    return fail("cudaStreamBeginCapture", e);
  }
  const ss_status r = step_impl(targets, H, W, T, V, C, D, 0, cap, tau, tg, fp8, scale,
                                accumulate, cand, slot, loss, lse, dH, dW, workspace,
                                workspace_bytes, cs);
  cudaGraph_t g = nullptr;
  e = cudaStreamEndCapture(cs, &g);
  cudaStreamDestroy(cs);
  if (r != SS_OK || e != cudaSuccess) {
    if (g) cudaGraphDestroy(g);
    return r != SS_OK ? r : fail("cudaStreamEndCapture", e);
  }
  auto* sg = new ss_step_graph;
  sg->graph = g;
  size_t n = 0;
  e = cudaGraphGetNodes(g, nullptr, &n);
  std::vector<cudaGraphNode_t> nodes(n);
  if (e == cudaSuccess && n > 0) e = cudaGraphGetNodes(g, nodes.data(), &n);
  for (size_t i = 0; e == cudaSuccess && i < n && !sg->cand_node; ++i) {
    cudaGraphNodeType type;
    if (cudaGraphNodeGetType(nodes[i], &type) != cudaSuccess || type != cudaGraphNodeTypeKernel)
      continue;
    cudaKernelNodeParams p = {};
    if (cudaGraphKernelNodeGetParams(nodes[i], &p) == cudaSuccess &&
        p.func == build_candidates_kernel()) {
      sg->cand_node = nodes[i];
      sg->base = p;
    }
  }
  if (e == cudaSuccess && !sg->cand_node) e = cudaErrorInvalidValue;
  if (e == cudaSuccess) e = cudaGraphInstantiate(&sg->exec, g, 0);
  if (e != cudaSuccess) {
    ss_step_graph_destroy(sg);
    return fail("capture of ss_step into a graph", e);
  }
  // the candidate kernel runs over all K * T targets (targets [K, T])
  sg->targets = targets;
  sg->T = static_cast<int>(T * tg.K);
  sg->V = static_cast<int>(V);
  sg->C = static_cast<int>(C);
  sg->cand = cand;
  sg->slot = slot;
  sg->hdr = static_cast<int*>(workspace);
  void* a[8] = {&sg->targets, &sg->T, &sg->V, &sg->C, &sg->seed, &sg->cand, &sg->slot, &sg->hdr};
  for (int i = 0; i < 8; ++i) sg->args[i] = a[i];
  *graph = sg;
  return SS_OK;
}

extern "C" {

ss_status ss_step_graph_create(const int32_t* targets, const uint16_t* H, const uint16_t* W,
                               int64_t T, int64_t V, int64_t C, int64_t D, const ss_head* head,
                               float scale, int accumulate, int32_t* cand, int32_t* slot,
                               float* loss, float* lse, uint16_t* dH, float* dW, void* workspace,
                               size_t workspace_bytes, ss_step_graph** graph) {
  if (!graph) return SS_ERR_INVALID;
  *graph = nullptr;
  float cap, tau;
  int fp8;
  const ss_status st = head_args(head, &cap, &tau, &fp8);
  if (st != SS_OK) return st;
  return graph_create(targets, kOneTarget, H, W, T, V, C, D, cap, tau, fp8, scale, accumulate,
                      cand, slot, loss, lse, dH, dW, workspace, workspace_bytes, graph);
}

ss_status ss_step_graph_create_mtp(const int32_t* targets, int64_t K, const float* weights,
                                   const uint16_t* H, const uint16_t* W, int64_t T, int64_t V,
                                   int64_t C, int64_t D, const ss_head* head, float scale,
                                   int accumulate, int32_t* cand, int32_t* slot, float* loss,
                                   float* lse, uint16_t* dH, float* dW, void* workspace,
                                   size_t workspace_bytes, ss_step_graph** graph) {
  if (!graph) return SS_ERR_INVALID;
  *graph = nullptr;
  float cap, tau;
  Targets tg;
  ss_status st = head_args(head, &cap, &tau);
  if (st == SS_OK) st = targets_args(K, weights, &tg);
  if (st != SS_OK) return st;
  return graph_create(targets, tg, H, W, T, V, C, D, cap, tau, 0, scale, accumulate, cand, slot,
                      loss, lse, dH, dW, workspace, workspace_bytes, graph);
}

ss_status ss_step_graph_launch(ss_step_graph* graph, uint64_t seed, ss_stream stream) {
  if (!graph || !graph->exec) return SS_ERR_INVALID;
  graph->seed = seed;
  cudaKernelNodeParams p = graph->base;
  p.kernelParams = graph->args;
  p.extra = nullptr;
  cudaError_t e = cudaGraphExecKernelNodeSetParams(graph->exec, graph->cand_node, &p);
  if (e != cudaSuccess) return fail("cudaGraphExecKernelNodeSetParams", e);
  e = cudaGraphLaunch(graph->exec, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SS_OK : fail("cudaGraphLaunch", e);
}

void ss_step_graph_destroy(ss_step_graph* graph) {
  if (!graph) return;
  if (graph->exec) cudaGraphExecDestroy(graph->exec);
  if (graph->graph) cudaGraphDestroy(graph->graph);
  delete graph;
}

const char* ss_last_error(void) { return g_err; }

const char* ss_status_string(ss_status status) {
  switch (status) {
    case SS_OK: return "ok";
    case SS_ERR_INVALID: return "invalid argument";
    case SS_ERR_UNSUPPORTED: return "unsupported size";
    case SS_ERR_CAPACITY: return "more distinct targets than candidate slots (U > C)";
    case SS_ERR_TARGET_RANGE: return "target id outside [0, V)";
    case SS_ERR_WORKSPACE: return "workspace too small";
    case SS_ERR_CUDA: return "CUDA error";
    case SS_ERR_TIMEOUT: return "device wait timed out";
    case SS_ERR_INDEX: return "cand entry outside [0, V) or slot outside [0, C)";
  }
  return "unknown status";
}

}  // extern "C"
