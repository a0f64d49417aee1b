/*
 * ss.h -- C ABI of libss, sampled-softmax cross-entropy over a shared candidate
 * set, forward and backward, as hand-written CUDA for GB300 (sm_103a).
 *
 * The method. The lm_head of a language model scores every vocabulary row for
 * every token; sampled softmax scores only a candidate subset of the rows, in
 * the forward and in the backward pass, with one candidate set shared by the
 * whole batch:
 *   - "KellerJordan/modded-nanogpt" README, technique list (sampled softmax
 *     over a shared candidate set for most of training);
 *   - "NanoGPT Training Record: Technical Optimizations & Speed", section "Key
 *     Optimizations and Ablation Table Results" (fewer vocabulary elements
 *     scored in forward and backward; candidate counts 10,240, 14,336 and
 *     24,576, then all 50,304 rows for the final steps), and section
 *     "Technical Architecture and Implementation Details";
 *   - the record tweet quoted on the airebao page (a token present in the
 *     batch is always scored; absent tokens only some of the time).
 * Definitions used here (textbook softmax cross-entropy restricted to the
 * candidate rows; notation: T tokens, D model width, V vocabulary rows,
 * C candidates, U distinct targets):
 *   cand   = the sorted distinct targets, then C - U non-target ids chosen
 *            uniformly without replacement (seeded; see ss_build_candidates),
 *            sorted by id;        slot[t] = index of target[t] in cand.
 *   S      = H . W[cand]^T                         (T x C logits, fp32)
 *   lse[t] = log sum_j exp(S[t,j]);   loss[t] = lse[t] - S[t, slot[t]]
 *   G      = scale * (exp(S - lse) - onehot(slot))
 *   dH     = G . W[cand];             dW[cand[j]] = (G^T . H)[j]
 *
 * Conventions for every entry point:
 *   - Every pointer argument except U_host / device_status_host / U_status_host
 *     is a DEVICE pointer on the current CUDA device. The caller owns every
 *     buffer; the library allocates no device memory and keeps no state
 *     between calls other than what it writes into the caller's workspace.
 *   - bf16 tensors are passed as uint16_t bit patterns. Matrices are
 *     row-major and dense: H [T, D], W [V, D], dH [T, D], dW [V, D].
 *   - H, W, dH, dW and the workspace must be 16-byte aligned; targets, cand,
 *     slot, loss, lse 4-byte aligned. Misaligned pointers -> SS_ERR_INVALID.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL means
 *     the legacy default stream). Only ss_build_candidates with a non-NULL
 *     U_host, and ss_read_status, synchronise that stream.
 *   - Argument errors are returned before anything is enqueued. Errors found
 *     on the device (a target id outside [0, V), more distinct targets than
 *     C, a cand or slot entry out of range, a device wait that timed out) are
 *     recorded in a status word inside the workspace: the first error wins,
 *     later kernels of any call that shares the workspace see it and do no
 *     work, and ss_read_status returns it. ss_build_candidates clears it. A
 *     new workspace must start with its first 1024 bytes (the header) zero,
 *     unless its first call is ss_build_candidates or ss_step.
 *   - Limits: 1 <= C <= V <= SS_MAX_V; 0 <= T < 2^31; D % 64 == 0 and
 *     64 <= D <= SS_MAX_D. Out of range -> SS_ERR_UNSUPPORTED (or
 *     SS_ERR_INVALID for values that can never be valid).
 *   - No C++ exception crosses this boundary.
 */
#ifndef SS_H_
#define SS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SS_MAX_V 524288
#define SS_MAX_D 16384

typedef enum ss_status {
  SS_OK = 0,
  SS_ERR_INVALID = 1,      /* bad argument: null pointer, bad size, misalignment */
  SS_ERR_UNSUPPORTED = 2,  /* valid in principle, outside this library's limits */
  SS_ERR_CAPACITY = 3,     /* U > C: more distinct targets than candidate slots */
  SS_ERR_TARGET_RANGE = 4, /* a target id outside [0, V) */
  SS_ERR_WORKSPACE = 5,    /* workspace smaller than ss_workspace_size() */
  SS_ERR_CUDA = 6,         /* a CUDA runtime/driver call or launch failed */
  SS_ERR_TIMEOUT = 7,      /* a device-side wait gave up (kernel returned early) */
  SS_ERR_INDEX = 8         /* a cand entry outside [0, V) or slot outside [0, C) */
} ss_status;

typedef void* ss_stream; /* cudaStream_t */

/*
 * Bytes of device workspace that ss_build_candidates, ss_forward and
 * ss_backward need for problem size (T, V, C, D); 0 if the sizes are invalid.
 * One workspace serves all three calls of a batch. Contents: a status header,
 * the gathered candidate rows W[cand] (C x D bf16), per-tile softmax partials
 * of the forward pass, and the bf16 softmax-gradient matrix G (T x C) of the
 * backward pass.
 */
size_t ss_workspace_size(int64_t T, int64_t V, int64_t C, int64_t D);

/*
 * Build the shared candidate set of one batch
 * ("KellerJordan/modded-nanogpt" README, technique list; airebao page, the
 * quoted record tweet: every in-batch target is scored).
 *   targets [T] int32, device: token ids, each in [0, V).
 *   seed        : selects the negatives. Non-target id v gets the key
 *                 (high 32 bits of SplitMix64 output number v of the stream
 *                 seeded with `seed`) * 2^32 + v; the C - U non-targets with
 *                 the smallest keys are the negatives (a uniform sample
 *                 without replacement when the keys behave as random).
 *   cand [C] int32, device, out: sorted distinct targets in [0, U), then the
 *                 negatives in ascending id order in [U, C).
 *   slot [T] int32, device, out: cand[slot[t]] == targets[t].
 *   U_host      : NULL, or a host int32 that receives U after the stream is
 *                 synchronised; with it the call also returns the device
 *                 status (SS_ERR_TARGET_RANGE, SS_ERR_CAPACITY).
 * Clears the workspace status word first. On a device-side error cand and
 * slot are left unspecified and the status word holds the error.
 */
ss_status ss_build_candidates(const int32_t* targets, int64_t T, int64_t V, int64_t C,
                              uint64_t seed, int32_t* cand, int32_t* slot, int32_t* U_host,
                              void* workspace, size_t workspace_bytes, ss_stream stream);

/*
 * Forward pass over the candidate rows ("NanoGPT Training Record: Technical
 * Optimizations & Speed", "Key Optimizations and Ablation Table Results":
 * only candidates are scored). The T x C logits never reach device memory:
 * tensor-core tiles are reduced to per-row log-sum-exp partials on chip.
 *   H [T, D] bf16, W [V, D] bf16, cand [C], slot [T]: inputs (device).
 *   loss [T] fp32 out: lse[t] - S[t, slot[t]].
 *   lse  [T] fp32 out: log-sum-exp over the C candidates; ss_backward needs it.
 */
ss_status ss_forward(const uint16_t* H, const uint16_t* W, const int32_t* cand,
                     const int32_t* slot, int64_t T, int64_t V, int64_t C, int64_t D,
                     float* loss, float* lse, void* workspace, size_t workspace_bytes,
                     ss_stream stream);

/*
 * Backward pass over the candidate rows (same sections as ss_forward: the
 * backward pass also scores only candidates). Recomputes the logits tile by
 * tile from H, W[cand] and the saved lse, forms G = scale * (P - Y) in bf16,
 * then dH = G . W[cand] and dW[cand] = G^T . H with fp32 accumulation.
 *   lse [T] fp32: from ss_forward on the same inputs.
 *   scale      : d(objective)/d(loss[t]); 1 for the sum over tokens, 1/T for
 *                the mean.
 *   accumulate : 0 -> dW[cand[j]] = dW_c[j]; 1 -> dW[cand[j]] += dW_c[j]
 *                (gradient accumulation over steps). Rows of dW that are not
 *                candidates are never read or written; cand must hold
 *                distinct ids (as ss_build_candidates makes them), which is
 *                what makes this write-back race-free without atomics.
 *   dH [T, D] bf16 out (overwritten), dW [V, D] fp32 in/out.
 */
ss_status ss_backward(const uint16_t* H, const uint16_t* W, const int32_t* cand,
                      const int32_t* slot, const float* lse, int64_t T, int64_t V, int64_t C,
                      int64_t D, float scale, int accumulate, uint16_t* dH, float* dW,
                      void* workspace, size_t workspace_bytes, ss_stream stream);

/*
 * Head options ("KellerJordan/modded-nanogpt" README, technique list: the
 * head's logits are rescaled asymmetrically and soft-capped; the pages give
 * no formula). With cap > 0 every candidate logit s passes through
 *   z = cap / (1 + exp(-s / tau))          (bounded to (0, cap))
 * before the softmax: lse and loss are of z, and the backward multiplies
 * G by dz/ds = z (cap - z) / (cap tau). Up to a shift, which the softmax
 * ignores, z is the symmetric soft cap (cap/2) tanh(s / (2 tau)).
 *   cap : 0 (or a NULL ss_head pointer) -> the plain head; else finite > 0.
 *   tau : finite > 0 when cap > 0.
 * Other values -> SS_ERR_INVALID. The *_head entry points below take it; the
 * same head must be passed to the forward and the backward of one batch.
 *
 * fp8 = 1: the FP8 head ("KellerJordan/modded-nanogpt" README, technique
 * list: FP8 for the head). H and the candidate rows W_c are each scaled by
 * 2^e (e the largest integer with max|x| * 2^e <= 448), rounded to e4m3 (to
 * nearest, ties to even) and used in that form by both logit GEMMs
 * (tcgen05 kind::f8f6f4, twice the bf16 rate); the gradient GEMMs use the
 * same rounded operands in bf16, G stays bf16. Results are those of the
 * plain head on the rounded operands.
 * fp8 = 2: the same, and FP8 through the backward pass too ("NanoGPT
 * Training Record: Technical Optimizations & Speed": FP8 quantisation
 * reaches through the backward pass; the pages give no format). Reading,
 * after the usual FP8 training split (E4M3 for values, E5M2 for gradients;
 * Micikevicius et al., "FP8 Formats for Deep Learning", 2022): the gradient
 * matrix, before the factor `scale`, is scaled by 2^15 (its bound
 * |P - Y| <= 1 then stays within e5m2's largest finite value 57344) and
 * rounded to e5m2 (to nearest, ties to even), G8 = e5m2(2^15 (P - Y));
 * the two gradient GEMMs run on G8 and the e4m3 operands
 * (dH = scale 2^-15 G8 . W_c,q and dW_c = scale 2^-15 G8^T . H_q).
 * Both modes combine with the capped head (the pages' head is FP8 and
 * soft-capped): the logits z are taken from the rounded operands, and with
 * FP8 gradients G8 = e5m2(2^e (P - Y) dz/ds) with e the largest integer such
 * that B 2^e <= 57344, B = cap / (4 tau) the bound of dz/ds (e = 15 for the
 * plain head; also 15 for cap = 4 tau). Both modes require D % 128 == 0
 * (else SS_ERR_UNSUPPORTED); the several-targets entry points take no FP8
 * head (SS_ERR_UNSUPPORTED); other fp8 values -> SS_ERR_INVALID.
 */
typedef struct ss_head {
  float cap;
  float tau;
  int fp8;  /* 0: bf16 operands; 1: FP8 logit GEMMs; 2: FP8 logit and gradient GEMMs */
} ss_head;

ss_status ss_forward_head(const uint16_t* H, const uint16_t* W, const int32_t* cand,
                          const int32_t* slot, int64_t T, int64_t V, int64_t C, int64_t D,
                          const ss_head* head, float* loss, float* lse, void* workspace,
                          size_t workspace_bytes, ss_stream stream);
ss_status ss_backward_head(const uint16_t* H, const uint16_t* W, const int32_t* cand,
                           const int32_t* slot, const float* lse, int64_t T, int64_t V,
                           int64_t C, int64_t D, const ss_head* head, float scale,
                           int accumulate, uint16_t* dH, float* dW, void* workspace,
                           size_t workspace_bytes, ss_stream stream);

/*
 * One training step of the loss in a single call: ss_build_candidates (with
 * U_host = NULL), ss_forward and ss_backward on the same batch, with the same
 * arguments and results as those three calls. The candidate rows W[cand] are
 * gathered once and serve both passes (the separate ss_backward gathers them
 * again, since it cannot know whether W or cand changed after ss_forward).
 * With bf16 operands (the plain head, or the capped head with cap <= 64;
 * also in ss_step_mtp, any targets and weights) the logits are computed
 * once: the forward keeps exp(S - r) in bf16 for the backward (r a per-row
 * reference; with the cap, exp(z - cap) dz/ds) instead of the backward
 * recomputing them. The results then equal
 * the three calls' within the library's tolerances (loss and lse 1e-3
 * relative, dH and dW 2e-2 relative Frobenius) rather than bit for bit; a row
 * whose logits exceed the reference's range makes the step recompute the
 * logits for the whole batch, with the same results. Other heads: the three
 * calls' results exactly.
 * Pages: as for ss_forward and ss_backward.
 */
ss_status ss_step(const int32_t* targets, const uint16_t* H, const uint16_t* W, int64_t T,
                  int64_t V, int64_t C, int64_t D, uint64_t seed, float scale, int accumulate,
                  int32_t* cand, int32_t* slot, float* loss, float* lse, uint16_t* dH, float* dW,
                  void* workspace, size_t workspace_bytes, ss_stream stream);
/* ss_step with head options (see ss_head). */
ss_status ss_step_head(const int32_t* targets, const uint16_t* H, const uint16_t* W, int64_t T,
                       int64_t V, int64_t C, int64_t D, uint64_t seed, const ss_head* head,
                       float scale, int accumulate, int32_t* cand, int32_t* slot, float* loss,
                       float* lse, uint16_t* dH, float* dW, void* workspace,
                       size_t workspace_bytes, ss_stream stream);

/*
 * Several targets per token scored against the same logits
 * ("KellerJordan/modded-nanogpt" README, technique list: multi-token
 * prediction; a prefix-token prediction auxiliary loss; the pages give no
 * formula). Token t has K targets targets[k * T + t] (k-major, [K, T]) with
 * host weights w[k] >= 0 (finite, sum W > 0), 1 <= K <= SS_MAX_TARGETS:
 *   loss[t] = sum_k w[k] (lse[t] - z[t, slot[k * T + t]])
 *   G       = scale (W P - sum_k w[k] onehot(slot[k])) (* dz/ds when capped)
 * The candidate set is built over all K * T targets, so slot is [K, T] too.
 * Same conventions and results otherwise as ss_forward / ss_backward /
 * ss_step with the same head; K = 1, w = {1} gives their results exactly.
 * Bad K or weights -> SS_ERR_INVALID.
 */
/*
 * The FP8 head's rounding of one tensor (see ss_head): x [n] bf16 (device,
 * n % 8 == 0) is scaled by 2^e, e the largest integer with max|x| 2^e <= 448,
 * rounded to e4m3 (to nearest, ties to even) into q [n] (device, 8-byte
 * aligned, e4m3 codes), and scaled back into xq [n] bf16 (exact; xq may alias
 * x). Uses 8 bytes of the workspace header of its own (any ss_workspace_size;
 * the workspace's status word is neither read nor written). Stream-ordered.
 */
ss_status ss_quantize_e4m3(const uint16_t* x, int64_t n, uint8_t* q, uint16_t* xq,
                           void* workspace, size_t workspace_bytes, ss_stream stream);

#define SS_MAX_TARGETS 8
ss_status ss_forward_mtp(const uint16_t* H, const uint16_t* W, const int32_t* cand,
                         const int32_t* slot, int64_t K, const float* weights, int64_t T,
                         int64_t V, int64_t C, int64_t D, const ss_head* head, float* loss,
                         float* lse, void* workspace, size_t workspace_bytes, ss_stream stream);
ss_status ss_backward_mtp(const uint16_t* H, const uint16_t* W, const int32_t* cand,
                          const int32_t* slot, int64_t K, const float* weights, const float* lse,
                          int64_t T, int64_t V, int64_t C, int64_t D, const ss_head* head,
                          float scale, int accumulate, uint16_t* dH, float* dW, void* workspace,
                          size_t workspace_bytes, ss_stream stream);
ss_status ss_step_mtp(const int32_t* targets, int64_t K, const float* weights, const uint16_t* H,
                      const uint16_t* W, int64_t T, int64_t V, int64_t C, int64_t D, uint64_t seed,
                      const ss_head* head, float scale, int accumulate, int32_t* cand,
                      int32_t* slot, float* loss, float* lse, uint16_t* dH, float* dW,
                      void* workspace, size_t workspace_bytes, ss_stream stream);

/*
 * The pages' candidate schedule ("NanoGPT Training Record: Technical
 * Optimizations & Speed", "Key Optimizations and Ablation Table Results":
 * 10,240, then 14,336, then 24,576 candidates, then all rows for the final
 * 87 steps). The pages do not say where the first three phases end; here
 * the steps before the final SS_SCHEDULE_FULL_STEPS are split into three
 * equal consecutive phases (step s of those n steps is in phase 3s / n,
 * rounded down). Each count is capped at V.
 *   step        : 0-based training step, 0 <= step < total_steps.
 * Returns C for that step, or -1 for invalid arguments (V < 1 or V > SS_MAX_V,
 * total_steps < 1, step outside [0, total_steps)).
 */
#define SS_SCHEDULE_FULL_STEPS 87
int64_t ss_schedule_candidates(int64_t step, int64_t total_steps, int64_t V);

/*
 * Zero the rows rows[0 .. n) of dW [V, D] fp32 (device pointers; rows holds
 * distinct ids in [0, V)), e.g. the rows an accumulation window wrote, before
 * the next window accumulates into them ("KellerJordan/modded-nanogpt"
 * README, technique list: lm_head gradients accumulated over 2 steps).
 * Entries outside [0, V) set SS_ERR_INDEX in the workspace status word and
 * are skipped. Stream-ordered; the workspace needs only its header
 * (ss_workspace_size of any shape is enough).
 */
ss_status ss_clear_rows(const int32_t* rows, int64_t n, int64_t V, int64_t D, float* dW,
                        void* workspace, size_t workspace_bytes, ss_stream stream);

/*
 * ss_step captured once into a CUDA graph and replayed ("NanoGPT Training
 * Record: Technical Optimizations & Speed", "Key Optimizations and Ablation
 * Table Results": training-step graph capture). ss_step_graph_create records
 * ss_step_head (head may be NULL: the plain head) with the given arguments (all of them fixed for the graph's life:
 * the same buffers, shapes, scale and accumulate flag; the buffers' contents
 * may change between launches) without running it. ss_step_graph_launch
 * runs it on `stream` with `seed` for the candidate build; results are those
 * of ss_step with the same arguments. The buffers must stay allocated until
 * ss_step_graph_destroy. One graph must not run concurrently with itself or
 * with another call on the same workspace. create returns the errors of
 * ss_step's argument checks, or SS_ERR_CUDA.
 */
typedef struct ss_step_graph ss_step_graph;
ss_status ss_step_graph_create(const int32_t* targets, const uint16_t* H, const uint16_t* W,
                               int64_t T, int64_t V, int64_t C, int64_t D, const ss_head* head,
                               float scale, int accumulate, int32_t* cand, int32_t* slot,
                               float* loss, float* lse, uint16_t* dH, float* dW, void* workspace,
                               size_t workspace_bytes, ss_step_graph** graph);
/* The same for ss_step_mtp: K weighted targets per token (targets [K, T],
 * slot [K, T]); its errors are those of ss_step_mtp's argument checks, or
 * SS_ERR_CUDA. The graph is launched and destroyed as above. */
ss_status ss_step_graph_create_mtp(const int32_t* targets, int64_t K, const float* weights,
                                   const uint16_t* H, const uint16_t* W, int64_t T, int64_t V,
                                   int64_t C, int64_t D, const ss_head* head, float scale,
                                   int accumulate, int32_t* cand, int32_t* slot, float* loss,
                                   float* lse, uint16_t* dH, float* dW, void* workspace,
                                   size_t workspace_bytes, ss_step_graph** graph);
ss_status ss_step_graph_launch(ss_step_graph* graph, uint64_t seed, ss_stream stream);
void ss_step_graph_destroy(ss_step_graph* graph);

/*
 * Allocation-free forward pass. Not part of the method the pages describe
 * (they have no counterpart): an operational variant of ss_forward for callers
 * that cannot allocate device memory at all -- for example code running as a
 * plugin inside a host program that has planned and owns every byte of device
 * memory and hands the plugin only its input and output buffers, or code on a
 * path where a cudaMalloc (which can synchronise the whole device) is not
 * acceptable. Such a caller has no workspace to pass.
 *
 * Same arguments and results as ss_forward, minus the workspace: the scratch
 * (gathered candidate rows, softmax partials, status word) lives in a
 * fixed-size array inside the library's own device data, of
 * SS_NOALLOC_SCRATCH_BYTES. Every GPU that loads the library holds that array
 * until the process exits. Sizes whose scratch, 1 KB + C*D*2 +
 * ceil(C/256)*T*16 + T*40 bytes (each term rounded up to 1 KB), exceeds it are
 * rejected with SS_ERR_UNSUPPORTED (ss_last_error says by how much).
 *   status_host : NULL, or a host int32 that receives the device status
 *                 word of this call after the stream is synchronised; the
 *                 call then also returns it (e.g. SS_ERR_INDEX). With NULL
 *                 the call does not synchronise, and a device-side error
 *                 (a candidate id or slot out of range) cannot be observed
 *                 afterwards: the status word lives in the library's private
 *                 array, which ss_read_status cannot reach. loss and lse are
 *                 then left as they were. Pass a status_host whenever cand
 *                 and slot are not known to be valid.
 * The first call on a device looks up the array's device address (with that
 * device current; again after the device's context is replaced, e.g. by
 * cudaDeviceReset); make that first call before any stream capture. The call allocates nothing: no cudaMalloc, no cudaFree, no
 * allocating library routine. All calls share the one array, which keeps the
 * previous call's contents; each call clears its status word first and
 * overwrites everything else it reads. Calls whose work overlaps on the GPU
 * (other streams, other host threads) race on the array: serialise them.
 */
#define SS_NOALLOC_SCRATCH_BYTES (32u << 20)
ss_status ss_forward_noalloc(const uint16_t* H, const uint16_t* W, const int32_t* cand,
                             const int32_t* slot, int64_t T, int64_t V, int64_t C, int64_t D,
                             float* loss, float* lse, int32_t* status_host, ss_stream stream);

/*
 * Synchronise `stream` and read the workspace status word (one of ss_status)
 * into *device_status_host and the last U written by ss_build_candidates into
 * *U_status_host (either may be NULL). Returns SS_ERR_CUDA if the
 * synchronisation fails, else the device status.
 */
ss_status ss_read_status(const void* workspace, size_t workspace_bytes, ss_stream stream,
                         int32_t* device_status_host, int32_t* U_status_host);

/* Static English text for a status code. */
const char* ss_status_string(ss_status status);

/* Text of the last failure recorded by libss on the calling host thread (the
 * failing CUDA call with its error string and code, or a size limit that was
 * exceeded), or "" if none yet. Valid until the next libss call on this
 * thread. */
const char* ss_last_error(void);

/*
 * Diagnostics: per-stage timing with CUDA events, for benchmarks.
 * Between ss_trace_begin and ss_trace_end, on the calling host thread, every
 * stage of the path that libss launches (one kernel, or a few kernels that
 * make one stage: the forward's first-tile and other-tile launches, the dH
 * and dW launches beyond L2) is bracketed by cudaEventRecord(events[2k]) and
 * cudaEventRecord(events[2k + 1]) on the launch stream, for k = 0, 1, ...
 * while k < capacity; later stages are counted but not recorded.
 *   events   : host array of 2 * capacity cudaEvent_t created by the caller.
 * ss_trace_end returns the number of stages since ss_trace_begin, or -1 if
 * an event record failed (e.g. an invalid event handle; the launches
 * themselves are unaffected); ss_trace_kernel_name(k) is the static name of
 * stage k (k < capacity and k < that count), or NULL;
 * ss_trace_kernel_launches(k) is the number of kernels stage k launched (0
 * for a stage with nothing to do), or -1. Tracing adds only the event
 * records.
 */
ss_status ss_trace_begin(void** events, int capacity);
int ss_trace_end(void);
const char* ss_trace_kernel_name(int k);
int ss_trace_kernel_launches(int k);

#ifdef __cplusplus
}
#endif

#endif /* SS_H_ */
