/*
 * sparse_mqa.h -- C ABI of the GB300 (sm_103a) top-k sparse multi-query
 * attention library: forward and backward with a per-head attention sink.
 *
 * The operation is the one behind `sparse_mqa_fwd_interface` and
 * `sparse_mqa_bwd_interface` on the DeepSeek-V4 kernel pages of NeMo
 * AutoModel (tilelang_sparse_mla_fwd, tilelang_sparse_mla_bwd):
 *
 *   every query token (b, s) has H heads that attend only to the `topk` rows
 *   of ONE shared kv tensor (used as both keys and values) listed in
 *   topk_idxs[b, s, :]; a slot whose index lies outside [0, S_kv) is masked;
 *   head h adds exp(attn_sink[h]) to its softmax denominator; the forward
 *   returns O and the base-2 log of that denominator (sink included), which
 *   the backward consumes together with dO to produce dQ and dKV.
 *
 * Conventions for every entry point
 *   - Tensors are row-major and contiguous, in DEVICE memory of the current
 *     CUDA device, with the shapes given below.  bf16 tensors are passed as
 *     `const void*` and hold IEEE bfloat16 values.
 *   - q, kv, o, dO, dq, dkv and the workspace must be 16-byte aligned; fp32
 *     and int32 tensors 4-byte aligned.
 *   - The caller allocates and owns every buffer; the library never allocates
 *     and never frees.  Inputs are only read.
 *   - Calls are asynchronous on `stream` (0 = the legacy default stream).
 *     Argument checks happen on the host before anything is launched; a
 *     rejected call launches nothing and leaves every output untouched.
 *   - A kernel that waits longer than its bounded limit (4 s per wait, or
 *     SMQA_WAIT_LIMIT_NS nanoseconds from the environment, or the value set by
 *     smqa_set_wait_limit_ns) records
 *     SMQA_ERR_DEVICE_TIMEOUT in a per-device status word and exits cleanly;
 *     read it with smqa_device_status().  The word is sticky: while it is set,
 *     the forward and backward-main kernels skip their work (their outputs
 *     are left undefined) until smqa_device_status(1) clears it.
 *   - Supported shapes: 1 <= H <= 128, D in {64, 512}, topk >= 1, B, S,
 *     S_kv >= 1, B*S_kv*D < 2^31, B*S*H < 2^31.  Anything else returns
 *     SMQA_ERR_UNSUPPORTED.
 */
#ifndef SPARSE_MQA_H_
#define SPARSE_MQA_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SMQA_ABI_VERSION 6

typedef enum {
    SMQA_OK = 0,
    SMQA_ERR_INVALID_ARG = 1,     /* null / misaligned pointer, non-positive size */
    SMQA_ERR_UNSUPPORTED = 2,     /* shape outside the supported set, small workspace */
    SMQA_ERR_CUDA = 3,            /* a CUDA runtime or driver call failed */
    SMQA_ERR_DEVICE_TIMEOUT = 4   /* a kernel's bounded wait ran out (device status) */
} smqa_status;

typedef struct {
    int32_t B;      /* batch                                  */
    int32_t S;      /* query tokens per batch element         */
    int32_t S_kv;   /* kv rows per batch element              */
    int32_t H;      /* query heads sharing the one kv tensor  */
    int32_t D;      /* head dim of q, of kv and of O          */
    int32_t topk;   /* index slots per query token            */
} smqa_shape;

/* smqa_fwd: form the exp2 argument as (score * sm_scale) * log2(e), two fp32
 * roundings, instead of score * (sm_scale * log2(e)).  The pages' forward
 * interface has this switch (`reference_rounding`: the scaled-logit fp32
 * arithmetic of the original inference kernel, LSE still in log2); both
 * orders agree to within one fp32 rounding of the logit. */
#define SMQA_FLAG_REFERENCE_ROUNDING 2u

/* smqa_bwd: write dkv as fp32 (the raw accumulator) instead of bf16.  The
 * pages' backward interface has the same switch (`return_dkv_accum_dtype`). */
#define SMQA_FLAG_RETURN_DKV_FP32 1u

/* smqa_bwd: accumulate dkv deterministically.  Every contribution is added
 * as a signed 64-bit fixed-point integer (the fp32 value times 2^k, rounded
 * to nearest) with 64-bit integer atomics, whose sum does not depend on the
 * order of the additions; the result is converted back to bf16 (or fp32 with
 * SMQA_FLAG_RETURN_DKV_FP32).  The binary point k is chosen per call on the
 * GPU (no host synchronisation) from maxima of the inputs (|q|, |dO|, the
 * row norms of dO and kv, |Delta|) and the largest number of slots naming
 * one kv row, so that no contribution or sum can exceed 2^61: the resolution
 * follows the magnitude of the gradients (a dO scaled by 2^-30 gives the
 * same relative accuracy as one of order 1), and the result is bit-identical
 * from run to run for the same inputs.  The workspace holds the 8-byte
 * accumulator, 256 bytes of statistics and a 4-byte count per kv row.  Not a
 * flag of the pages. */
#define SMQA_FLAG_DETERMINISTIC_DKV 4u

/*
 * Bytes of device workspace smqa_fwd needs for `shape`: 0 when D = 64; for
 * D = 512 the exchange pool (4 KB of slot flags and the token counter + 96
 * slots of 198 KB).  For D = 512 pairs of CTAs that own one half of D each
 * work through the tokens, taking them one at a time from the counter;
 * every 64-slot block a pair trades its partial scores through its slot of
 * this pool (it stays in L2).  The contents need no initialisation:
 * smqa_fwd clears the slot flags and the counter on its stream.  Returns 0
 * for an unsupported shape.
 */
size_t smqa_fwd_workspace_bytes(smqa_shape shape);

/*
 * Forward (tilelang_sparse_mla_fwd: `sparse_mqa_fwd_interface`, the kernel
 * factory `sparse_mqa_fwd`).
 *   q         [B,S,H,D]    bf16  queries
 *   kv        [B,S_kv,D]   bf16  shared keys/values
 *   attn_sink [H]          fp32  per-head denominator bias (enters as exp)
 *   topk_idxs [B,S,topk]   int32 kv row per slot; outside [0,S_kv) = masked
 *   sm_scale               score multiplier; <= 0 (or NaN) selects D^-1/2
 *   o         [B,S,H,D]    bf16  output (written)
 *   lse       [B,S,H]      fp32  log2(sum_valid exp(sm_scale*q.k) + exp(sink))
 *   workspace, workspace_bytes  a 256-byte-aligned device buffer of at least
 *                          smqa_fwd_workspace_bytes(shape) bytes (may be NULL
 *                          with size 0 when that is 0); a smaller one is
 *                          rejected with SMQA_ERR_UNSUPPORTED.  Calls whose
 *                          kernels may overlap must not share it.
 *   flags                  0 or SMQA_FLAG_REFERENCE_ROUNDING
 * A token whose slots are all masked gets O = 0 and lse = sink/ln 2.
 * For D = 512 a score is the fp32 sum of two half-D partial scores, each
 * already multiplied by sm_scale*log2(e) (by sm_scale with
 * SMQA_FLAG_REFERENCE_ROUNDING, the sum then by log2(e)) and rounded to
 * block floating point: per head and 64-slot block, one power-of-two scale
 * and int16 mantissas, so each partial carries an absolute error of at most
 * 2^-15 (1 + 2^-14) of the largest partial magnitude of its head and block.
 */
smqa_status smqa_fwd(const void* q, const void* kv, const float* attn_sink,
                     const int32_t* topk_idxs, smqa_shape shape, float sm_scale,
                     void* o, float* lse, void* workspace, size_t workspace_bytes,
                     unsigned flags, cudaStream_t stream);

/*
 * Bytes of device workspace smqa_bwd needs for `shape` and `flags`: the fp32
 * dKV accumulator [B,S_kv,D] (absent with SMQA_FLAG_RETURN_DKV_FP32, where
 * dkv itself accumulates; with SMQA_FLAG_DETERMINISTIC_DKV always present,
 * 8 bytes per element, followed by 256 bytes of per-call statistics and a
 * uint32 count per kv row), Delta [B,S,H] fp32, and for D = 512 the exchange
 * pool of smqa_bwd_exchange_bytes(shape), each 256-byte aligned.
 * Returns 0 for an unsupported shape.
 */
size_t smqa_bwd_workspace_bytes(smqa_shape shape, unsigned flags);

/*
 * Bytes of the exchange pool the main backward kernel uses for `shape`
 * (0 when D = 64; 4 KB of slot flags and the token counter + 96 slots of
 * 132 KB when D = 512).  For D = 512 pairs of CTAs that own one half of D
 * each work through the tokens, taking them one at a time from the counter;
 * every 64-slot block a pair trades its partial scores and dP, in block
 * floating point (16-bit mantissas with one power-of-two exponent per head
 * and block, so the precision is relative to the block's largest value at any
 * magnitude), through its slot of this pool (it stays in L2).  The pool's
 * contents need no initialisation: smqa_bwd_main clears the slot flags and
 * the counter on its stream.  Returns 0 for an unsupported shape.
 */
size_t smqa_bwd_exchange_bytes(smqa_shape shape);

/*
 * Backward (tilelang_sparse_mla_bwd: `sparse_mqa_bwd_interface`, which runs
 * its `preprocess`, `bwd` and `postprocess` kernels in that order).
 *   q, kv, attn_sink, topk_idxs, sm_scale   as in smqa_fwd
 *   o         [B,S,H,D]  bf16  the forward's output
 *   dout      [B,S,H,D]  bf16  gradient of the loss w.r.t. o
 *   lse       [B,S,H]    fp32  the forward's log2 LSE
 *   dq        [B,S,H,D]  bf16  written
 *   dkv       [B,S_kv,D] bf16 written, or fp32 with SMQA_FLAG_RETURN_DKV_FP32;
 *                              rows no slot names are 0
 *   dsink     [H]        fp32  gradient w.r.t. attn_sink, written; may be NULL
 *                              (not among the pages' outputs: the sink adds
 *                              exp(attn_sink[h]) to every row's denominator,
 *                              so dsink[h] = -sum over tokens of
 *                              exp(attn_sink[h] - LSE_e) * rowsum(o * dout))
 *   workspace, workspace_bytes  >= smqa_bwd_workspace_bytes(shape, flags)
 * dkv sums contributions with fp32 atomics, so its low bits may differ from
 * run to run (bit-identical with SMQA_FLAG_DETERMINISTIC_DKV); dq and dsink
 * are deterministic.  flags: any of SMQA_FLAG_RETURN_DKV_FP32,
 * SMQA_FLAG_DETERMINISTIC_DKV.
 */
smqa_status smqa_bwd(const void* q, const void* kv, const float* attn_sink, const void* o,
                     const void* dout, const int32_t* topk_idxs, const float* lse,
                     smqa_shape shape, float sm_scale, void* dq, void* dkv, float* dsink,
                     void* workspace, size_t workspace_bytes, unsigned flags,
                     cudaStream_t stream);

/*
 * Forward and backward for callers that cannot allocate device memory.  (The
 * sparse MQA pages have no counterpart: these entry points exist for this
 * library's users, not for parity with the pages.)
 *
 * smqa_fwd and smqa_bwd need a device workspace of smqa_fwd_workspace_bytes()
 * and smqa_bwd_workspace_bytes() bytes.  Some callers cannot provide one:
 * code running under a memory planner that has already handed every byte of
 * device memory to its own pool, plugins that get only the tensors they are
 * given, or hot paths that must not take the device-wide synchronisation
 * cudaMalloc/cudaFree may imply.  These entry
 * points compute exactly what smqa_fwd and smqa_bwd compute, with the same
 * arguments minus the workspace, and allocate nothing: their scratch is a
 * static device buffer of SMQA_STATIC_SCRATCH_BYTES inside the library, which
 * every GPU that loads the library holds until the process exits.  The
 * forward's scratch always fits.
 *   - Shapes whose smqa_bwd_workspace_bytes(shape, flags) exceeds
 *     SMQA_STATIC_SCRATCH_BYTES are rejected with SMQA_ERR_UNSUPPORTED before
 *     anything runs (smqa_last_error() gives both sizes).  With
 *     SMQA_FLAG_RETURN_DKV_FP32 only Delta (B*S*H floats) and, for D = 512,
 *     the exchange pool need the buffer.
 *   - The first call on a device looks up the buffer's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.
 *   - All calls (forward and backward) share the one buffer per device, and
 *     it keeps the previous call's contents (each call re-zeroes what must
 *     start at zero).  Calls whose kernels may overlap on the GPU -- different streams without
 *     ordering between them, or several host threads -- race on it and give
 *     wrong results; order them on one stream.
 */
#define SMQA_STATIC_SCRATCH_BYTES (64u << 20)
smqa_status smqa_fwd_static_scratch(const void* q, const void* kv, const float* attn_sink,
                                    const int32_t* topk_idxs, smqa_shape shape, float sm_scale,
                                    void* o, float* lse, unsigned flags, cudaStream_t stream);
smqa_status smqa_bwd_static_scratch(const void* q, const void* kv, const float* attn_sink,
                                    const void* o, const void* dout, const int32_t* topk_idxs,
                                    const float* lse, smqa_shape shape, float sm_scale, void* dq,
                                    void* dkv, float* dsink, unsigned flags, cudaStream_t stream);

/*
 * Forward, and forward + backward, on HOST buffers.  (The sparse MQA pages
 * have no counterpart: the pages' interfaces take device tensors.)
 *
 * Every tensor argument below is HOST memory with the shape and dtype of
 * smqa_fwd / smqa_bwd (page-locked memory lets the copies run asynchronously
 * and overlap the kernels; pageable memory works but each copy then blocks
 * the calling thread).  The call copies the inputs into `workspace` (DEVICE
 * memory of the current device, 256-byte aligned, at least the size the
 * matching *_workspace_bytes function returns), runs the kernels of smqa_fwd
 * and smqa_bwd and copies the results back.  It works in token chunks (at
 * most about 24 per call, at least 256 tokens each except a last group of
 * whole batch elements; see smqa_host_chunk_plan) so that the copies of one
 * chunk overlap the kernels of others: a
 * host->device stream, the caller's `stream` for the forward, a backward
 * stream and a device->host stream, ordered by events.  Every token's
 * arithmetic is that of smqa_fwd / smqa_bwd, so o, lse, dq and dsink are
 * bit-identical to theirs (dkv too with SMQA_FLAG_DETERMINISTIC_DKV).
 *
 * Ordering: the work starts after what is already queued on `stream`, and
 * `stream` continues only after all of it (the host outputs are complete once
 * `stream` is synchronized).  The three helper streams and their events are
 * created by the first call on a device and shared by all calls on it (calls
 * from several threads are serialised while they enqueue).  Inputs must stay
 * unchanged and outputs untouched until `stream` has reached the call's end.
 * A workspace must not be shared by calls that may overlap.
 *
 * Errors: arguments are checked before anything is queued (null or device
 * pointers for host tensors, a workspace that is not device memory of the
 * current device, a small workspace, bad flags, unsupported shapes); a
 * failing CUDA call part-way returns SMQA_ERR_CUDA with the work queued so
 * far left in place and `stream` still ordered after it.
 *
 * smqa_fwd_host      : q, kv, attn_sink, topk_idxs -> o, lse.
 *                      flags: 0 or SMQA_FLAG_REFERENCE_ROUNDING.
 * smqa_fwd_bwd_host  : the forward, then the backward with the given dout
 *                      (the gradient of the loss w.r.t. o, known to the
 *                      caller in advance: a fixed upstream gradient, a
 *                      gradient check, a benchmark) -> o, lse, dq, dkv and,
 *                      if dsink is non-NULL, dsink.  flags: any of
 *                      SMQA_FLAG_REFERENCE_ROUNDING, SMQA_FLAG_RETURN_DKV_FP32,
 *                      SMQA_FLAG_DETERMINISTIC_DKV.
 * The *_workspace_bytes functions return 0 for an unsupported shape.  The
 * workspace holds a device copy of every input and output plus the scratch
 * of smqa_fwd and smqa_bwd (q, o: 2*B*S*H*D bytes each; forward + backward
 * adds dout and dq of the same size and the dkv accumulator).
 */
size_t smqa_fwd_host_workspace_bytes(smqa_shape shape);

/* The token chunks of smqa_fwd_host / smqa_fwd_bwd_host for `shape`, in the
 * order they are processed: writes min(count, max_chunks) quadruples
 * (b0, nb, s0, ns) -- batch elements [b0, b0 + nb) x positions [s0, s0 + ns),
 * nb > 1 only with s0 = 0 and ns = S -- into `out` (4 int32 per chunk; may be
 * NULL) and returns the number of chunks, or 0 for an unsupported shape.
 * Pieces of S are whole multiples of the tokens one backward launch holds on
 * the GPU at once, so the plan reads the current device's SM count (152, a
 * GB300's, when no device is visible); it launches and allocates nothing. */
int smqa_host_chunk_plan(smqa_shape shape, int32_t* out, int max_chunks);
size_t smqa_fwd_bwd_host_workspace_bytes(smqa_shape shape, unsigned flags);
smqa_status smqa_fwd_host(const void* q, const void* kv, const float* attn_sink,
                          const int32_t* topk_idxs, smqa_shape shape, float sm_scale, void* o,
                          float* lse, void* workspace, size_t workspace_bytes, unsigned flags,
                          cudaStream_t stream);
smqa_status smqa_fwd_bwd_host(const void* q, const void* kv, const float* attn_sink,
                              const int32_t* topk_idxs, const void* dout, smqa_shape shape,
                              float sm_scale, void* o, float* lse, void* dq, void* dkv,
                              float* dsink, void* workspace, size_t workspace_bytes,
                              unsigned flags, cudaStream_t stream);

/*
 * The backward stages one at a time (same arguments as smqa_bwd; used
 * to time and profile them separately).
 *   preprocess  : delta[B,S,H] = rowsum(o * dout) in fp32, and dkv_accum
 *                 [B,S_kv,D] fp32 set to zero
 *   main        : dq, and dkv_accum += every slot's dKV contribution
 *   postprocess : dkv_bf16 = round-to-nearest-even(dkv_accum)
 *   sink_grad   : dsink[H] from attn_sink, the forward's lse and the
 *                 preprocess's delta (the optional output of smqa_bwd)
 * smqa_bwd_main also takes the exchange pool: a 256-byte-aligned device
 * buffer of at least smqa_bwd_exchange_bytes(shape) bytes (may be NULL with
 * size 0 when that is 0); a smaller pool is rejected with
 * SMQA_ERR_UNSUPPORTED.  Calls whose kernels may overlap must not share it.
 */
smqa_status smqa_bwd_preprocess(const void* o, const void* dout, smqa_shape shape,
                                float* delta, float* dkv_accum, cudaStream_t stream);
smqa_status smqa_bwd_main(const void* q, const void* kv, const float* attn_sink,
                          const void* dout, const int32_t* topk_idxs, const float* lse,
                          const float* delta, smqa_shape shape, float sm_scale, void* dq,
                          float* dkv_accum, void* exchange, size_t exchange_bytes,
                          cudaStream_t stream);
smqa_status smqa_bwd_postprocess(const float* dkv_accum, smqa_shape shape, void* dkv_bf16,
                                 cudaStream_t stream);
smqa_status smqa_bwd_sink_grad(const float* attn_sink, const float* lse, const float* delta,
                               smqa_shape shape, float* dsink, cudaStream_t stream);

/*
 * Lightning-indexer backward (tilelang_indexer_bwd: `indexer_bwd_interface`,
 * "backward interface for a single batch element").  The page gives the
 * tensors, not the formula; the library computes the gradient with respect
 * to index_q of the lightning indexer's scores
 *     score[t,j] = sum_h weights[t,h] * ReLU(<index_q[t,h,:], index_k[idx[t,j],:]>)
 * given grad_scores, that is
 *     dq[t,h,:] = weights[t,h] * sum_j grad_scores[t,j] * [<q[t,h,:], k_j> > 0] * k_j
 * over the slots whose index lies in [0, S_kv) (others are masked; a slot
 * listed twice counts twice; the ReLU's slope is taken as 0 at 0).
 *   index_q      bf16 [S, H, D]       weights      fp32 [S, H]
 *   index_k      bf16 [S_kv, D]       topk_indices int32 [S, topk]
 *   grad_scores  fp32 [S, topk]       dq           bf16 [S, H, D] (output)
 * shape.B must be 1; 1 <= H <= 128, D in {64, 128}.  The logits are formed
 * in fp32 by the tensor core, so where <q, k_j> lies within fp32 rounding of
 * 0 the gate may differ from an exact evaluation.  grad_scores enter the
 * tensor core as bf16.  Device pointers; asynchronous on `stream`; nothing
 * is allocated.  Not a function of the attention pages.
 */
smqa_status smqa_indexer_bwd(const void* index_q, const float* weights, const void* index_k,
                             const int32_t* topk_indices, const float* grad_scores,
                             smqa_shape shape, void* dq, cudaStream_t stream);

/*
 * The same for a batch in the page's `batched_indexer_bwd` layouts (which
 * the page describes as looping over the batch; here every batch element
 * runs in the same launch):
 *   index_q      bf16 [S, B, H, D]    weights      fp32 [S, B, H]
 *   index_k      bf16 [S_kv, B, D]    topk_indices int32 [B, S, topk]
 *   grad_scores  fp32 [B, S, topk]    dq           bf16 [S, B, H, D] (output)
 * Indices address rows of the same batch element.
 */
smqa_status smqa_batched_indexer_bwd(const void* index_q, const float* weights,
                                     const void* index_k, const int32_t* topk_indices,
                                     const float* grad_scores, smqa_shape shape, void* dq,
                                     cudaStream_t stream);

/*
 * Reads the device status word that kernels set when a bounded wait runs out
 * (SMQA_OK if none did).  Synchronizes the current device first.  A nonzero
 * `clear` resets the word afterwards.
 */
smqa_status smqa_device_status(int clear);

/*
 * Sets the limit, in nanoseconds, of every bounded wait in the kernels
 * launched after this call (all devices, all threads); 0 restores the
 * default (SMQA_WAIT_LIMIT_NS from the environment, else 4 s).  Returns the
 * limit in force before the call.  A wait that runs out makes its kernel
 * record SMQA_ERR_DEVICE_TIMEOUT and exit without finishing its work (the
 * outputs of that call are undefined); the GPU context stays usable.  This
 * is how a watchdog can be tightened, and how the failure path is tested
 * without hanging a GPU.  Not a function of the pages.
 */
uint64_t smqa_set_wait_limit_ns(uint64_t ns);

/*
 * Test hook for the failure path.  In every forward, backward-main and
 * indexer-backward launch after this call, CTA `cta` (a block index of the
 * launch; -1 turns the hook
 * off) stops after issuing its first tensor-core instruction and waits for a
 * condition that never comes true.  The wait is bounded like every other, so
 * after the wait limit the CTA records SMQA_ERR_DEVICE_TIMEOUT, drains its
 * copies and MMAs, frees TMEM and exits, and the other CTAs stop at their
 * next check of the status word: the same path a real stall would take, with
 * no fault, trap or endless loop.  Outputs of those launches are undefined.
 * Not for production use.  Not a function of the pages.
 */
void smqa_debug_stall(int cta);

/* Human-readable name of a status code (static storage, never NULL). */
const char* smqa_status_string(smqa_status status);

/* Text describing the last failure seen by this thread's calls (a rejected
 * argument or a failing CUDA call); static thread-local storage. */
const char* smqa_last_error(void);

/* SMQA_ABI_VERSION of the built library. */
int smqa_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SPARSE_MQA_H_ */
