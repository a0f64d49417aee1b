/*
 * ss_oracle.c -- plain, slow CPU oracle for sampled-softmax cross-entropy over
 * a shared candidate set.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the CPU
 * baseline / reference arms of the benchmark load this library. The CUDA
 * library never calls it, and the two share no code, headers or tables.
 *
 * What is computed, and where it comes from:
 *   - "KellerJordan/modded-nanogpt" README, technique list: the training loss
 *     is a sampled softmax over ONE candidate set shared by the whole batch.
 *   - "NanoGPT Training Record: Technical Optimizations & Speed", section "Key
 *     Optimizations and Ablation Table Results" (and "Technical Architecture
 *     and Implementation Details"): only the candidate rows of the vocabulary
 *     are scored, in both the forward and the backward pass; the candidate
 *     count follows a schedule that ends at the full vocabulary (C = V).
 *   - the record tweet quoted on the airebao page: a token that occurs in the
 *     batch is always scored, a token that does not is scored only sometimes.
 *     Reading: every batch target is a candidate; the rest of the set is
 *     filled with sampled non-target ids.
 * The pages give no formula. The textbook softmax cross-entropy restricted to
 * the candidate rows is written out below, step by step, in the pages' terms:
 *
 *   candidates  u = sorted unique targets (U of them); k = C - U negatives =
 *               the k non-target ids with the smallest keys, sorted by id;
 *               cand = u ++ negatives; slot[t] = position of target[t] in u.
 *   forward     s[t][j] = sum_d H[t][d] * W[cand[j]][d]           (d ascending)
 *               lse[t]  = m + log(sum_j exp(s[t][j] - m)), m = max_j s[t][j]
 *               loss[t] = lse[t] - s[t][slot[t]]
 *   backward    G[t][j] = scale * (exp(s[t][j] - lse[t]) - [j == slot[t]])
 *               dH[t]   = sum_j G[t][j] * W[cand[j]]               (j ascending)
 *               dW[cand[j]] = sum_t G[t][j] * H[t]                 (t ascending)
 *
 * Head variant ("KellerJordan/modded-nanogpt" README, technique list: the
 * logits are rescaled asymmetrically and soft-capped; the pages give no
 * formula). Reading: a logistic cap applied to every candidate logit before
 * the softmax,
 *               z[t][j] = A / (1 + exp(-s[t][j] / tau))        A > 0, tau > 0,
 *   bounded to (0, A), not symmetric about 0 (up to a shift, which the
 *   softmax ignores, it is the symmetric cap (A/2) tanh(s / (2 tau))). The
 *   forward and backward above then run on z: lse and loss from z, and by the
 *   chain rule G[t][j] = scale * (exp(z - lse) - [j == slot[t]]) * dz/ds with
 *   dz/ds = z (A - z) / (A tau). A = 0 selects the plain head (z = s).
 *
 * Several targets per token ("KellerJordan/modded-nanogpt" README,
 * technique list: multi-token prediction, a prefix-token prediction
 * auxiliary loss; no formula on the pages). Reading: token t has K targets
 * y[k][t] with weights w[k] >= 0, all scored against the same logits (one
 * GEMM), and the candidate set is built over all K*T targets:
 *               loss[t] = sum_k w[k] * (lse[t] - z[t][slot[k][t]])
 *               G[t][j] = scale * (W exp(z[t][j] - lse[t]) - sum_k w[k] [j == slot[k][t]]) dz/ds
 *   with W = sum_k w[k]. K = 1, w = 1 is the single-target loss above.
 *
 * Negative-sampling key (the pages name no sampler; reading: uniform without
 * replacement over the non-targets, driven by a counter-based generator so
 * that a CPU and a GPU implementation can agree bit for bit):
 *   key(v) = (high 32 bits of SplitMix64 output number v of a stream whose
 *             state starts at `seed`) * 2^32 + v
 *   where output number i (0-based) of SplitMix64 (Steele, Lea and Flood,
 *   "Fast splittable pseudorandom number generators", OOPSLA 2014; the
 *   splitmix64.c reference by S. Vigna) is mix(seed + (i + 1) * 0x9E3779B97F4A7C15).
 *
 * FP8 head ("KellerJordan/modded-nanogpt" README, technique list: FP8 for
 * the head; no format details on the pages). Reading: the head's operands are
 * rounded to the e4m3 grid (1 sign, 4 exponent bits with bias 7, 3 mantissa
 * bits, subnormals down to 2^-9, largest value 448; round to nearest, ties to
 * even) after scaling by one power of two per tensor, 2^e with e the largest
 * integer such that amax * 2^e <= 448 (amax = max |x| over the tensor: all of
 * H, all candidate rows of W), then scaled back. Everything downstream (the
 * logits, the softmax, the gradients, which use the same rounded operands)
 * is the definition above applied to the rounded H and W[cand]; G itself
 * stays in the working precision.
 *
 * FP8 through the backward pass ("NanoGPT Training Record: Technical
 * Optimizations & Speed": FP8 quantisation reaches through the backward pass;
 * no format on the pages). Reading, after the common FP8 training split of
 * e4m3 for values and e5m2 for gradients (Micikevicius et al., "FP8 Formats
 * for Deep Learning", 2022): on top of the FP8 head above, the gradient
 * matrix before the factor `scale` is scaled by 2^15 (so that its bound
 * |P - Y| <= 1 stays inside e5m2's largest finite value 57344) and rounded
 * to the e5m2 grid (1 sign, 5 exponent bits with bias 15, 2 mantissa bits,
 * subnormals down to 2^-16; round to nearest, ties to even):
 *               G8[t][j] = round_e5m2(2^15 (exp(s[t][j] - lse[t]) - [j == slot[t]]))
 *               dH[t]    = scale 2^-15 sum_j G8[t][j] * W[cand[j]]
 *               dW[cand[j]] = scale 2^-15 sum_t G8[t][j] * H[t]
 *   with H and W the e4m3-rounded operands. With the capped head the
 *   gradient matrix carries the factor dz/ds, at most A / (4 tau) (at
 *   z = A / 2), so its bound is B = A / (4 tau) instead of 1, and the power
 *   of two is 2^eG with eG the largest integer such that B 2^eG <= 57344
 *   (eG = 15 for the plain head):
 *               G8 = round_e5m2(2^eG (exp(z - lse) - [j == slot]) dz/ds).
 *
 * Precision: the definition is fp32. Its inputs are bf16 bit patterns widened
 * exactly to float. An fp64 instantiation of the same loops, on double inputs,
 * exists for the finite-difference and library cross-checks. Build with
 * -ffp-contract=off so that x86-64 and aarch64 round identically.
 *
 * Parallelism: OpenMP over independent output rows only (tokens for the
 * forward and dH, candidate rows for dW); every sum keeps the order above.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum {
  ORC_OK = 0,
  ORC_ERR_INVALID = 1,
  ORC_ERR_CAPACITY = 3,     /* more unique targets than candidate slots */
  ORC_ERR_TARGET_RANGE = 4, /* a target id outside [0, V) */
  ORC_ERR_NOMEM = 8
};

static float bf16_to_float(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* ---------------------------------------------------------------- SplitMix64 */

uint64_t orc_splitmix64_output(uint64_t seed, uint64_t i) {
  uint64_t z = seed + (i + 1u) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

uint64_t orc_negative_key(uint64_t seed, int64_t v) {
  uint64_t hi = orc_splitmix64_output(seed, (uint64_t)v) >> 32;
  return (hi << 32) | (uint64_t)(uint32_t)v;
}

/* ---------------------------------------------------------- candidate build */

static int cmp_i32(const void* a, const void* b) {
  int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
  return (x > y) - (x < y);
}

static int cmp_u64(const void* a, const void* b) {
  uint64_t x = *(const uint64_t*)a, y = *(const uint64_t*)b;
  return (x > y) - (x < y);
}

/* index of v in the sorted array u[0..n), or -1 */
static int64_t find_sorted(const int32_t* u, int64_t n, int32_t v) {
  int64_t lo = 0, hi = n;
  while (lo < hi) {
    int64_t mid = lo + (hi - lo) / 2;
    if (u[mid] < v) lo = mid + 1;
    else hi = mid;
  }
  return (lo < n && u[lo] == v) ? lo : -1;
}

/*
 * Build the shared candidate set of one batch.
 *   targets[T] in [0, V); cand[C] and slot[T] are written; *U_out = U.
 * Returns ORC_ERR_TARGET_RANGE if a target is outside [0, V) and
 * ORC_ERR_CAPACITY if U > C (then *U_out is still set and cand/slot are not).
 */
int orc_build_candidates(const int32_t* targets, int64_t T, int64_t V, int64_t C,
                         uint64_t seed, int32_t* cand, int32_t* slot, int64_t* U_out) {
  if (T < 0 || V <= 0 || C <= 0 || C > V) return ORC_ERR_INVALID;
  for (int64_t t = 0; t < T; ++t)
    if (targets[t] < 0 || targets[t] >= V) return ORC_ERR_TARGET_RANGE;

  /* u = sorted unique targets */
  int32_t* u = (int32_t*)malloc(sizeof(int32_t) * (size_t)(T > 0 ? T : 1));
  if (!u) return ORC_ERR_NOMEM;
  memcpy(u, targets, sizeof(int32_t) * (size_t)T);
  qsort(u, (size_t)T, sizeof(int32_t), cmp_i32);
  int64_t U = 0;
  for (int64_t i = 0; i < T; ++i)
    if (U == 0 || u[U - 1] != u[i]) u[U++] = u[i];
  *U_out = U;
  if (U > C) { free(u); return ORC_ERR_CAPACITY; }

  /* negatives: the k non-targets with the smallest keys, then sorted by id */
  int64_t k = C - U;
  int64_t n_non = V - U;
  uint64_t* keys = (uint64_t*)malloc(sizeof(uint64_t) * (size_t)(n_non > 0 ? n_non : 1));
  if (!keys) { free(u); return ORC_ERR_NOMEM; }
  int64_t n = 0;
  for (int64_t v = 0; v < V; ++v)
    if (find_sorted(u, U, (int32_t)v) < 0) keys[n++] = orc_negative_key(seed, v);
  qsort(keys, (size_t)n, sizeof(uint64_t), cmp_u64);
  int32_t* neg = (int32_t*)malloc(sizeof(int32_t) * (size_t)(k > 0 ? k : 1));
  if (!neg) { free(keys); free(u); return ORC_ERR_NOMEM; }
  for (int64_t i = 0; i < k; ++i) neg[i] = (int32_t)(keys[i] & 0xFFFFFFFFull);
  qsort(neg, (size_t)k, sizeof(int32_t), cmp_i32);

  for (int64_t i = 0; i < U; ++i) cand[i] = u[i];
  for (int64_t i = 0; i < k; ++i) cand[U + i] = neg[i];
  for (int64_t t = 0; t < T; ++t) slot[t] = (int32_t)find_sorted(u, U, targets[t]);

  free(neg);
  free(keys);
  free(u);
  return ORC_OK;
}

/* ------------------------------------------------------ forward / backward */
/*
 * The loops below are written once as a macro and instantiated twice:
 *   f32: inputs are bf16 bit patterns, arithmetic in float (the definition);
 *   f64: inputs are doubles, arithmetic in double (finite differences and
 *        library cross-checks, which need inputs that are not on the bf16 grid).
 * Row subsets: `rows` (token indices, nrows of them) or NULL for all T rows;
 * `cols` (candidate indices j, ncols of them) or NULL for all C candidates.
 * Outputs for a subset are packed in subset order.
 */
#define LOAD_BF16(x) bf16_to_float(x)
#define LOAD_REAL(x) (x)

#define ORC_DEFINE(REAL, SUF, IN_T, LOAD, EXP, LOG)                                          \
  /* logits of token t against every candidate: s[j], j = 0..C-1 */                         \
  static void logits_##SUF(const IN_T* H, const IN_T* W, const int32_t* cand, int64_t C,    \
                           int64_t D, int64_t t, REAL* s) {                                 \
    const IN_T* h = H + t * D;                                                               \
    for (int64_t j = 0; j < C; ++j) {                                                        \
      const IN_T* w = W + (int64_t)cand[j] * D;                                              \
      REAL acc = 0;                                                                          \
      for (int64_t d = 0; d < D; ++d) acc += (REAL)LOAD(h[d]) * (REAL)LOAD(w[d]);            \
      s[j] = acc;                                                                            \
    }                                                                                        \
  }                                                                                          \
                                                                                             \
  /* the head transform z(s) (cap A = 0: the plain head, z = s) and dz/ds */                 \
  static REAL head_z_##SUF(REAL s, REAL cap, REAL tau) {                                     \
    return cap > 0 ? cap / ((REAL)1 + EXP(-s / tau)) : s;                                    \
  }                                                                                          \
  static REAL head_dz_##SUF(REAL z, REAL cap, REAL tau) {                                    \
    return cap > 0 ? z * (cap - z) / (cap * tau) : (REAL)1;                                  \
  }                                                                                          \
                                                                                             \
  /* K targets per token: slot[k * T + t], weights w[k] */                                  \
  void orc_forward_mtp_##SUF(const IN_T* H, const IN_T* W, const int32_t* cand,              \
                             const int32_t* slot, int64_t K, const REAL* w, int64_t T,       \
                             int64_t C, int64_t D, REAL cap, REAL tau, const int64_t* rows,  \
                             int64_t nrows, REAL* loss, REAL* lse) {                         \
    int64_t n = rows ? nrows : T;                                                            \
    _Pragma("omp parallel")                                                                  \
    {                                                                                        \
      REAL* s = (REAL*)malloc(sizeof(REAL) * (size_t)C);                                     \
      _Pragma("omp for schedule(dynamic, 1)")                                                \
      for (int64_t i = 0; i < n; ++i) {                                                      \
        int64_t t = rows ? rows[i] : i;                                                      \
        logits_##SUF(H, W, cand, C, D, t, s);                                                \
        for (int64_t j = 0; j < C; ++j) s[j] = head_z_##SUF(s[j], cap, tau);                 \
        REAL m = s[0];                                                                       \
        for (int64_t j = 1; j < C; ++j)                                                      \
          if (s[j] > m) m = s[j];                                                            \
        REAL sum = 0;                                                                        \
        for (int64_t j = 0; j < C; ++j) sum += EXP(s[j] - m);                                \
        REAL l = m + LOG(sum);                                                               \
        lse[i] = l;                                                                          \
        REAL acc = 0;                                                                        \
        for (int64_t k = 0; k < K; ++k) acc += w[k] * (l - s[slot[k * T + t]]);              \
        loss[i] = acc;                                                                       \
      }                                                                                      \
      free(s);                                                                               \
    }                                                                                        \
  }                                                                                          \
                                                                                             \
  /* the weighted target indicator sum_k w[k] [j == slot[k][t]] */                           \
  static REAL target_weight_##SUF(const int32_t* slot, int64_t K, const REAL* w, int64_t T,  \
                                  int64_t t, int64_t j) {                                    \
    REAL y = 0;                                                                              \
    for (int64_t k = 0; k < K; ++k)                                                          \
      if (slot[k * T + t] == j) y += w[k];                                                   \
    return y;                                                                                \
  }                                                                                          \
                                                                                             \
  /* dH rows: needs lse of those tokens (lse_rows packed like rows) */                       \
  void orc_backward_dH_mtp_##SUF(const IN_T* H, const IN_T* W, const int32_t* cand,          \
                                 const int32_t* slot, int64_t K, const REAL* w,              \
                                 const REAL* lse_rows, int64_t T, int64_t C, int64_t D,      \
                                 REAL cap, REAL tau, REAL scale, const int64_t* rows,        \
                                 int64_t nrows, REAL* dH) {                                  \
    int64_t n = rows ? nrows : T;                                                            \
    REAL wsum = 0;                                                                           \
    for (int64_t k = 0; k < K; ++k) wsum += w[k];                                            \
    _Pragma("omp parallel")                                                                  \
    {                                                                                        \
      REAL* s = (REAL*)malloc(sizeof(REAL) * (size_t)C);                                     \
      _Pragma("omp for schedule(dynamic, 1)")                                                \
      for (int64_t i = 0; i < n; ++i) {                                                      \
        int64_t t = rows ? rows[i] : i;                                                      \
        logits_##SUF(H, W, cand, C, D, t, s);                                                \
        REAL* out = dH + i * D;                                                              \
        for (int64_t d = 0; d < D; ++d) out[d] = 0;                                          \
        for (int64_t j = 0; j < C; ++j) {                                                    \
          REAL y = target_weight_##SUF(slot, K, w, T, t, j);                                 \
          REAL z = head_z_##SUF(s[j], cap, tau);                                             \
          REAL g = scale * (wsum * EXP(z - lse_rows[i]) - y) * head_dz_##SUF(z, cap, tau);   \
          const IN_T* wr = W + (int64_t)cand[j] * D;                                         \
          for (int64_t d = 0; d < D; ++d) out[d] += g * (REAL)LOAD(wr[d]);                   \
        }                                                                                    \
      }                                                                                      \
      free(s);                                                                               \
    }                                                                                        \
  }                                                                                          \
                                                                                             \
  /* dW_c rows (candidate index j): needs lse of ALL T tokens */                             \
  void orc_backward_dW_mtp_##SUF(const IN_T* H, const IN_T* W, const int32_t* cand,          \
                                 const int32_t* slot, int64_t K, const REAL* w,              \
                                 const REAL* lse, int64_t T, int64_t C, int64_t D, REAL cap, \
                                 REAL tau, REAL scale, const int64_t* cols, int64_t ncols,   \
                                 REAL* dWc) {                                                \
    int64_t n = cols ? ncols : C;                                                            \
    REAL wsum = 0;                                                                           \
    for (int64_t k = 0; k < K; ++k) wsum += w[k];                                            \
    _Pragma("omp parallel for schedule(dynamic, 1)")                                         \
    for (int64_t i = 0; i < n; ++i) {                                                        \
      int64_t j = cols ? cols[i] : i;                                                        \
      const IN_T* wr = W + (int64_t)cand[j] * D;                                             \
      REAL* out = dWc + i * D;                                                               \
      for (int64_t d = 0; d < D; ++d) out[d] = 0;                                            \
      for (int64_t t = 0; t < T; ++t) {                                                      \
        const IN_T* h = H + t * D;                                                           \
        REAL st = 0;                                                                         \
        for (int64_t d = 0; d < D; ++d) st += (REAL)LOAD(h[d]) * (REAL)LOAD(wr[d]);          \
        REAL y = target_weight_##SUF(slot, K, w, T, t, j);                                   \
        REAL z = head_z_##SUF(st, cap, tau);                                                 \
        REAL g = scale * (wsum * EXP(z - lse[t]) - y) * head_dz_##SUF(z, cap, tau);          \
        for (int64_t d = 0; d < D; ++d) out[d] += g * (REAL)LOAD(h[d]);                      \
      }                                                                                      \
    }                                                                                        \
  }                                                                                          \
                                                                                             \
  /* one target per token */                                                                 \
  void orc_forward_head_##SUF(const IN_T* H, const IN_T* W, const int32_t* cand,             \
                              const int32_t* slot, int64_t T, int64_t C, int64_t D,          \
                              REAL cap, REAL tau, const int64_t* rows, int64_t nrows,        \
                              REAL* loss, REAL* lse) {                                       \
    const REAL one = 1;                                                                      \
    orc_forward_mtp_##SUF(H, W, cand, slot, 1, &one, T, C, D, cap, tau, rows, nrows, loss,   \
                          lse);                                                              \
  }                                                                                          \
  void orc_backward_dH_head_##SUF(const IN_T* H, const IN_T* W, const int32_t* cand,         \
                                  const int32_t* slot, const REAL* lse_rows, int64_t T,      \
                                  int64_t C, int64_t D, REAL cap, REAL tau, REAL scale,      \
                                  const int64_t* rows, int64_t nrows, REAL* dH) {            \
    const REAL one = 1;                                                                      \
    orc_backward_dH_mtp_##SUF(H, W, cand, slot, 1, &one, lse_rows, T, C, D, cap, tau, scale, \
                              rows, nrows, dH);                                              \
  }                                                                                          \
  void orc_backward_dW_head_##SUF(const IN_T* H, const IN_T* W, const int32_t* cand,         \
                                  const int32_t* slot, const REAL* lse, int64_t T, int64_t C, \
                                  int64_t D, REAL cap, REAL tau, REAL scale,                 \
                                  const int64_t* cols, int64_t ncols, REAL* dWc) {           \
    const REAL one = 1;                                                                      \
    orc_backward_dW_mtp_##SUF(H, W, cand, slot, 1, &one, lse, T, C, D, cap, tau, scale, cols, \
                              ncols, dWc);                                                   \
  }                                                                                          \
                                                                                             \
  /* the plain head */                                                                       \
  void orc_forward_##SUF(const IN_T* H, const IN_T* W, const int32_t* cand,                  \
                         const int32_t* slot, int64_t T, int64_t C, int64_t D,               \
                         const int64_t* rows, int64_t nrows, REAL* loss, REAL* lse) {        \
    orc_forward_head_##SUF(H, W, cand, slot, T, C, D, 0, 1, rows, nrows, loss, lse);         \
  }                                                                                          \
  void orc_backward_dH_##SUF(const IN_T* H, const IN_T* W, const int32_t* cand,              \
                             const int32_t* slot, const REAL* lse_rows, int64_t T,           \
                             int64_t C, int64_t D, REAL scale, const int64_t* rows,          \
                             int64_t nrows, REAL* dH) {                                      \
    orc_backward_dH_head_##SUF(H, W, cand, slot, lse_rows, T, C, D, 0, 1, scale, rows,       \
                               nrows, dH);                                                   \
  }                                                                                          \
  void orc_backward_dW_##SUF(const IN_T* H, const IN_T* W, const int32_t* cand,              \
                             const int32_t* slot, const REAL* lse, int64_t T, int64_t C,     \
                             int64_t D, REAL scale, const int64_t* cols, int64_t ncols,      \
                             REAL* dWc) {                                                    \
    orc_backward_dW_head_##SUF(H, W, cand, slot, lse, T, C, D, 0, 1, scale, cols, ncols,     \
                               dWc);                                                         \
  }

ORC_DEFINE(float, f32, uint16_t, LOAD_BF16, expf, logf)
ORC_DEFINE(double, f64, double, LOAD_REAL, exp, log)

/* ------------------------------------------------------------- e4m3 rounding */

/* x rounded to the e4m3 grid, ties to even; |x| >= 448 saturates to 448. */
float orc_round_e4m3(float x) {
  if (x != x) return x;
  const float a = fabsf(x);
  if (a == 0.0f) return x;
  if (a >= 448.0f) return copysignf(448.0f, x);
  int e2;
  frexpf(a, &e2);          /* a = m * 2^e2, m in [0.5, 1): a in [2^(e2-1), 2^e2) */
  int E = e2 - 1;          /* binade exponent */
  if (E < -6) E = -6;      /* below 2^-6: subnormals, spacing 2^-9 */
  const float q = ldexpf(1.0f, E - 3);  /* grid spacing in this binade */
  return copysignf(rintf(a / q) * q, x); /* a / q is exact; rintf rounds half to even */
}

/* the largest integer e with amax * 2^e <= 448 (0 for amax = 0) */
int orc_e4m3_scale_exponent(float amax) {
  if (!(amax > 0.0f)) return 0;
  int k;
  const float m = frexpf(amax, &k); /* amax = m 2^k, m in [0.5, 1); 448 = 0.875 * 2^9 */
  return m <= 0.875f ? 9 - k : 8 - k;
}

/* out[i] = round_e4m3(x[i] * 2^e) * 2^-e for the bf16 values x (n of them), as
 * bf16 bit patterns (the rounded values are exact in bf16) */
void orc_quantize_e4m3_bf16(const uint16_t* x, int64_t n, int e, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) {
    const float v = ldexpf(orc_round_e4m3(ldexpf(bf16_to_float(x[i]), e)), -e);
    uint32_t u;
    memcpy(&u, &v, 4);
    out[i] = (uint16_t)(u >> 16); /* exact: at most 4 significant bits */
  }
}

/* ------------------------------------------------------------- e5m2 rounding */

/* x rounded to the e5m2 grid, ties to even; |x| >= 57344 saturates to 57344. */
float orc_round_e5m2(float x) {
  if (x != x) return x;
  const float a = fabsf(x);
  if (a == 0.0f) return x;
  if (a >= 57344.0f) return copysignf(57344.0f, x);
  int e2;
  frexpf(a, &e2);          /* a in [2^(e2-1), 2^e2) */
  int E = e2 - 1;
  if (E < -14) E = -14;    /* below 2^-14: subnormals, spacing 2^-16 */
  const float q = ldexpf(1.0f, E - 2);  /* grid spacing in this binade */
  return copysignf(rintf(a / q) * q, x);
}

/* the largest integer e with B 2^e <= 57344, B the bound of |(P - Y) dz/ds|:
 * 1 for the plain head (A = 0, e = 15), A / (4 tau) for the capped head */
int orc_g8_exponent(float cap, float tau) {
  const double B = cap > 0 ? (double)cap / (4.0 * (double)tau) : 1.0;
  int e = 15;
  while (B * ldexp(1.0, e) > 57344.0) --e;
  while (B * ldexp(1.0, e + 1) <= 57344.0) ++e;
  return e;
}

/* G8 of one logit s (z = the head's logit): round_e5m2(2^e (exp(z - lse) - y) dz/ds) */
static float g8_of(float s, float lse, float y, float cap, float tau, int e) {
  const float z = head_z_f32(s, cap, tau);
  return orc_round_e5m2(ldexpf((expf(z - lse) - y) * head_dz_f32(z, cap, tau), e));
}

/* FP8 gradients, one target per token, plain head: dH rows (lse_rows of
 * exactly those rows), inputs already rounded to e4m3 (bf16 bit patterns). */
void orc_backward_dH_g8(const uint16_t* H, const uint16_t* W, const int32_t* cand,
                        const int32_t* slot, const float* lse_rows, int64_t T, int64_t C,
                        int64_t D, float cap, float tau, float scale, const int64_t* rows,
                        int64_t nrows, float* dH) {
  int64_t n = rows ? nrows : T;
  const int e = orc_g8_exponent(cap, tau);
  const float f = ldexpf(scale, -e);
#pragma omp parallel
  {
    float* s = (float*)malloc(sizeof(float) * (size_t)C);
#pragma omp for schedule(dynamic, 1)
    for (int64_t i = 0; i < n; ++i) {
      int64_t t = rows ? rows[i] : i;
      logits_f32(H, W, cand, C, D, t, s);
      float* out = dH + i * D;
      for (int64_t d = 0; d < D; ++d) out[d] = 0;
      for (int64_t j = 0; j < C; ++j) {
        const float g = f * g8_of(s[j], lse_rows[i], slot[t] == j ? 1.0f : 0.0f, cap, tau, e);
        const uint16_t* wr = W + (int64_t)cand[j] * D;
        for (int64_t d = 0; d < D; ++d) out[d] += g * bf16_to_float(wr[d]);
      }
    }
    free(s);
  }
}

/* ... and dW_c rows (candidate index j; lse of ALL T tokens) */
void orc_backward_dW_g8(const uint16_t* H, const uint16_t* W, const int32_t* cand,
                        const int32_t* slot, const float* lse, int64_t T, int64_t C, int64_t D,
                        float cap, float tau, float scale, const int64_t* cols, int64_t ncols,
                        float* dWc) {
  int64_t n = cols ? ncols : C;
  const int e = orc_g8_exponent(cap, tau);
  const float f = ldexpf(scale, -e);
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < n; ++i) {
    int64_t j = cols ? cols[i] : i;
    const uint16_t* wr = W + (int64_t)cand[j] * D;
    float* out = dWc + i * D;
    for (int64_t d = 0; d < D; ++d) out[d] = 0;
    for (int64_t t = 0; t < T; ++t) {
      const uint16_t* h = H + t * D;
      float st = 0;
      for (int64_t d = 0; d < D; ++d) st += bf16_to_float(h[d]) * bf16_to_float(wr[d]);
      const float g = f * g8_of(st, lse[t], slot[t] == j ? 1.0f : 0.0f, cap, tau, e);
      for (int64_t d = 0; d < D; ++d) out[d] += g * bf16_to_float(h[d]);
    }
  }
}

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
