/*
 * gdn.h: C ABI of the GB300 (sm_103a) Gated DeltaNet recurrence library.
 *
 * The operation ("Optimizing on-device inference for Apple Silicon",
 * section "Qwen creates three workload shapes"): a Gated DeltaNet layer keeps
 * one fixed-size recurrent state per value head; a learned gate decides how
 * much of it survives each token and a delta update writes the token in.
 * Per value head h the state S is a dv x dk fp32 matrix (the section "Keep
 * recurrent state on chip" fixes state and gate as fp32 and q/k as bf16) and
 * each token t does
 *
 *     alpha_t = exp(log_alpha_t)
 *     S_t     = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *     o_t     = S_t q_t
 *
 * with value head h reading query/key head h / (hv / hk).  Long prompts may be
 * fed in pieces: passing one call's final_state as the next call's init_state
 * gives the same result as one call over the whole prompt (section "Bound
 * scratch memory by chunking the prompt").
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller, except the
 *     ones whose name ends in _host.  The library allocates nothing on these
 *     calls.  Between calls it keeps only:
 *       - one error word per device, shared by all streams of that device
 *         (see gdn_device_error);
 *       - the fixed scratch array of gdn_prefill_noalloc, one per device,
 *         which holds the last gdn_prefill_noalloc call's intermediates;
 *       - host-side caches per device (kernel attributes, symbol addresses).
 *   - Every device pointer, and the stream, must belong to the CURRENT device
 *     (cudaSetDevice): the kernels are launched there.  Before launching, the
 *     prefill calls check q, out, final_state and the workspace (decode:
 *     state and out) with cudaPointerGetAttributes and return
 *     GDN_ERR_INVALID_ARG for host memory or another device's memory.  The
 *     check is skipped while the stream is capturing a CUDA graph.
 *   - Every tensor is dense, row-major, with the shape given below, and its
 *     base address is 16-byte aligned.
 *   - By default q and k are used exactly as given: the caller has already
 *     L2-normalised them and scaled q (e.g. by 1/sqrt(dk)).  The qk_norm and
 *     q_scale arguments are the one exception: they ask the kernels to do
 *     that preparation themselves.
 *   - log_alpha must be <= 0 (it may be -INFINITY) and beta in [0, 1].  The
 *     GPU paths clamp log_alpha to >= -20 (alpha >= 2.1e-9) so that decay
 *     ratios inside a chunk stay finite; the effect is below fp32 resolution
 *     of any state that is not already negligible.
 *   - `stream` is a cudaStream_t passed as void* (NULL: the legacy default
 *     stream).  Calls are asynchronous on that stream.
 *   - Argument errors are detected on the host before anything is launched
 *     and returned synchronously; nothing is written in that case.  A launch
 *     failure returns GDN_ERR_CUDA.  Faults inside a kernel surface on a later
 *     synchronisation, as with any CUDA work.
 *   - Supported head sizes: dk == dv, and dk in {32, 64, 128} for GDN_ALGO_SCAN
 *     and gdn_decode_step; dk == dv == 128 for GDN_ALGO_CHUNKED (other sizes
 *     return GDN_ERR_UNSUPPORTED).
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define GDN_API __attribute__((visibility("default")))
#else
#define GDN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1,  /* null pointer, bad size, bad cu_seqlens, ... */
    GDN_ERR_UNSUPPORTED = 2,  /* well-formed but not implemented (head size, dtype, algo) */
    GDN_ERR_ALIGNMENT = 3,    /* a pointer is not 16-byte aligned */
    GDN_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
    GDN_ERR_TIMEOUT = 5,      /* a bounded device-side wait gave up (see gdn_device_error) */
    GDN_ERR_INTERNAL = 6,     /* a device-side consistency check failed */
    GDN_ERR_WORKSPACE = 7     /* workspace missing or smaller than gdn_prefill_workspace_size */
} gdn_status;

typedef enum {
    GDN_ALGO_CHUNKED = 0,  /* blocked evaluation, 64-token chunks, tcgen05 tensor cores */
    GDN_ALGO_SCAN = 1,     /* direct token-by-token scan, state held in registers; when no sequence
                              has more than 32 tokens and the batch needs more than one wave of
                              16-row CTAs, each state row is instead streamed once through all of
                              its sequence's tokens (the decode step's mapping) */
    GDN_ALGO_AUTO = 2      /* the faster of the two for this problem, chosen on the host (gdn_prefill_algo) */
} gdn_algo;

typedef enum {
    GDN_DTYPE_BF16 = 0,
    GDN_DTYPE_F32 = 1
} gdn_dtype;

/*
 * gdn_prefill: run the recurrence over n_seqs packed sequences.
 *
 *   n_seqs           number of sequences (>= 1)
 *   total_tokens     T = cu_seqlens[n_seqs] (>= 0)
 *   hk, hv, dk, dv   query/key heads, value heads (hv % hk == 0), head sizes
 *   q, k             bf16 [T, hk, dk]
 *   v                bf16 [T, hv, dv]
 *   log_alpha, beta  fp32 [T, hv]
 *   init_state       fp32 [n_seqs, hv, dv, dk] (row = value index), or NULL for zeros
 *   cu_seqlens       int32 [n_seqs + 1] on the device: sequence n is tokens
 *                    [cu_seqlens[n], cu_seqlens[n+1])
 *   cu_seqlens_host  the same n_seqs + 1 values in host memory; used to plan the
 *                    launch without a device synchronisation (the workspace, the
 *                    grids, and which sequences one state-pass CTA carries one
 *                    after another).  It must start at 0, be non-decreasing and
 *                    end at total_tokens.  The kernels also clamp the device
 *                    copy to [0, total_tokens]; where the device copy gives a
 *                    state-pass CTA other chunks than the host copy planned, that
 *                    CTA records GDN_ERR_INTERNAL and runs nothing.
 *   out              [T, hv, dv], dtype out_dtype (GDN_DTYPE_BF16 or _F32)
 *   final_state      fp32 [n_seqs, hv, dv, dk] or NULL.  It may be the same
 *                    buffer as init_state (updated in place); any other overlap
 *                    with an input is an error.
 *   qk_norm, q_scale query/key preparation inside the kernels ("Optimizing
 *                    on-device inference for Apple Silicon", section "Reduce
 *                    intermediate and state traffic": the decode path fuses
 *                    query and key preparation).  With qk_norm = 1 every q and
 *                    k head vector x is used as x / sqrt(|x|^2 + 1e-6); in all
 *                    cases q is then multiplied by q_scale (a finite float;
 *                    1/sqrt(dk) for raw projections).  qk_norm = 0, q_scale = 1
 *                    uses q and k exactly as given.
 *   norm_weight,     fused output normalisation, as for gdn_decode_step: with
 *   norm_eps         norm_weight (fp32 [dv] device array) each head's output
 *                    vector o of every token becomes
 *                    o / sqrt(mean(o^2) + norm_eps) * norm_weight; NULL
 *                    leaves the outputs as computed.
 *   gate_scale,      gates computed inside the kernels.  Both NULL: log_alpha
 *   gate_bias        and beta are the gates.  Both given (fp32 [hv] device
 *                    arrays; gate_scale[h] finite and >= 0): log_alpha and
 *                    beta hold each token's raw projections a and y, and the
 *                    kernels use, per token and value head h,
 *                        log_alpha = -gate_scale[h] * softplus(a + gate_bias[h])
 *                        beta      = 1 / (1 + exp(-y))
 *                    in fp32 (the section "Keep recurrent state on chip" keeps
 *                    the state and its gate in fp32; the form is the
 *                    configured workloads' gate recipe with per-head
 *                    parameters, our reading).  One without the other:
 *                    GDN_ERR_INVALID_ARG.
 *   algo             GDN_ALGO_CHUNKED, GDN_ALGO_SCAN or GDN_ALGO_AUTO
 *   workspace        device scratch of at least gdn_prefill_workspace_size()
 *                    bytes (may be NULL when that size is 0), 256-byte aligned.
 *                    Its contents on entry do not matter.
 *   stream           cudaStream_t as void*
 */
GDN_API gdn_status gdn_prefill(int n_seqs, int total_tokens, int hk, int hv, int dk, int dv,
                       const void *q, const void *k, const void *v,
                       const float *log_alpha, const float *beta,
                       const float *init_state,
                       const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                       void *out, int out_dtype, float *final_state,
                       int qk_norm, float q_scale, const float *norm_weight, float norm_eps,
                       const float *gate_scale, const float *gate_bias,
                       int algo, void *workspace, size_t workspace_bytes, void *stream);

/*
 * gdn_prefill_chunked_phase: one of the two phases of the chunked prefill, for
 * callers that schedule or time them separately.  gdn_prefill with
 * GDN_ALGO_CHUNKED is exactly GDN_PHASE_PREP followed by GDN_PHASE_PASS on the
 * same stream with the same arguments and the same workspace, whose contents
 * must not change in between.
 *   GDN_PHASE_PREP  per-chunk preparation, parallel over (chunk, value head):
 *                   reads q, k, log_alpha, beta, cu_seqlens; writes the workspace.
 *   GDN_PHASE_PASS  state passing across chunks and the outputs: reads every
 *                   input and the workspace; writes out and final_state.
 * Arguments, validation and errors as for gdn_prefill (algo is implied).
 */
typedef enum {
    GDN_PHASE_PREP = 1,
    GDN_PHASE_PASS = 2
} gdn_phase;

GDN_API gdn_status gdn_prefill_chunked_phase(int phase, int n_seqs, int total_tokens, int hk, int hv, int dk, int dv,
                                             const void *q, const void *k, const void *v,
                                             const float *log_alpha, const float *beta,
                                             const float *init_state,
                                             const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                                             void *out, int out_dtype, float *final_state,
                                             int qk_norm, float q_scale, const float *norm_weight, float norm_eps,
                                             const float *gate_scale, const float *gate_bias,
                                             void *workspace, size_t workspace_bytes, void *stream);

/*
 * Bytes of device workspace gdn_prefill needs for this problem (0 when the
 * algorithm is, or GDN_ALGO_AUTO resolves to, GDN_ALGO_SCAN).  Returns 0 and
 * sets *status (if non-NULL) to an error code when the arguments are invalid.
 */
GDN_API size_t gdn_prefill_workspace_size(int n_seqs, int total_tokens, int hk, int hv, int dk, int dv,
                                  const int32_t *cu_seqlens_host, int algo, gdn_status *status);

/*
 * gdn_prefill_algo: the algorithm GDN_ALGO_AUTO resolves to for this problem
 * (GDN_ALGO_CHUNKED or GDN_ALGO_SCAN), or -1 when the arguments are invalid.
 * "Optimizing on-device inference for Apple Silicon", section "Qwen creates
 * three workload shapes": whether the direct scan or the blocked form is
 * faster depends on the model dimensions, the workload and the hardware.  The
 * rule is a host-side function of the sequence lengths and head count, fitted
 * to a sweep of both paths on GB300 (N sequences of T tokens, d = 128, 32
 * value heads):
 *   - the scan when the longest sequence has at most 16 tokens, or at most 32
 *     tokens with n_seqs * hv <= 64 (the chunked path pays a fixed cost of
 *     about 12 us for one short sequence and 34 us for eight);
 *   - the scan whenever dk != 128 (the chunked path implements d = 128 only);
 *   - the chunked path otherwise.
 * It needs no CUDA call.  gdn_prefill and gdn_prefill_workspace_size apply the
 * same rule, so a workspace sized for GDN_ALGO_AUTO fits what gdn_prefill runs.
 */
GDN_API int gdn_prefill_algo(int n_seqs, int total_tokens, int hk, int hv, int dk, int dv,
                             const int32_t *cu_seqlens_host);

/*
 * gdn_prefill_pass_plan: how the chunked path's state pass groups the
 * sequences into buckets, for inspection.  A bucket is a run of consecutive
 * sequences that one state-pass CTA per (value head, 32-row slice) carries one
 * after another; the chunks of one sequence are sequential ("Optimizing
 * on-device inference for Apple Silicon", section "Qwen creates three workload
 * shapes": the blocked form still passes the state from chunk to chunk).  The
 * plan is the one gdn_prefill makes on a device with `multiprocessors` SMs
 * (152 on GB300): either one wave of buckets of several sequences each, or one
 * bucket per sequence, whichever a chunk-count cost estimate favours.
 *
 *   cu_seqlens_host    int32 [n_seqs + 1] host array, as for gdn_prefill
 *   bucket_first_seq   host array of `capacity` ints; on success entries
 *                      [0, nb] hold the buckets' first sequences followed by
 *                      n_seqs (bucket b carries sequences [bucket_first_seq[b],
 *                      bucket_first_seq[b + 1])).  n_seqs + 1 entries always
 *                      suffice.
 *
 * Returns nb >= 1, or -1 when an argument is invalid or capacity < nb + 1.  It
 * needs no CUDA call.
 */
GDN_API int gdn_prefill_pass_plan(int n_seqs, int total_tokens, int hv, const int32_t *cu_seqlens_host,
                                  int multiprocessors, int *bucket_first_seq, int capacity);

/*
 * gdn_decode_step: one token for each of n independent states (batch-1 decode
 * of n layers, or n requests), updating the states in place.
 *
 *   state            fp32 [n, hv, dv, dk], read and overwritten
 *   q, k             bf16 [n, hk, dk]
 *   v                bf16 [n, hv, dv]
 *   log_alpha, beta  fp32 [n, hv]
 *   out              [n, hv, dv], dtype out_dtype; must not overlap state
 *   qk_norm, q_scale as for gdn_prefill
 *   norm_weight      fp32 [dv] device array, or NULL.  When given, the output
 *                    normalisation is fused into the step: each head's output
 *                    vector o becomes o / sqrt(mean(o^2) + norm_eps) * norm_weight
 *                    ("Optimizing on-device inference for Apple Silicon",
 *                    section "Reduce intermediate and state traffic": the
 *                    decode path fuses the recurrent update with its
 *                    normalisation; the form of the norm is our reading).
 *   norm_eps         finite, >= 0; used only with norm_weight
 *   gate_scale,      as for gdn_prefill: the gates computed from raw inputs
 *   gate_bias        in log_alpha and beta ([n, hv]), or both NULL
 */
GDN_API gdn_status gdn_decode_step(int n, int hk, int hv, int dk, int dv, float *state,
                           const void *q, const void *k, const void *v,
                           const float *log_alpha, const float *beta,
                           void *out, int out_dtype, int qk_norm, float q_scale,
                           const float *norm_weight, float norm_eps,
                           const float *gate_scale, const float *gate_bias, void *stream);

/*
 * Synchronise `stream` and return (and clear) the device-side error word the
 * kernels set when a bounded wait gives up (GDN_ERR_TIMEOUT) or an internal
 * check fails (GDN_ERR_INTERNAL).  GDN_OK when nothing was recorded.  The word
 * belongs to the current device, not to the stream: it collects what every
 * call on that device recorded, whatever its stream, and reading it clears it
 * for all of them.
 */
GDN_API gdn_status gdn_device_error(void *stream);

/*
 * gdn_selftest_bounded_wait: a check of the failure path that every kernel of
 * the library shares; it computes nothing (the pages have no counterpart).
 * Every device-side wait of the kernels gives up after 1 s, records
 * GDN_ERR_TIMEOUT in the device error word and lets the kernel return, so a
 * stalled kernel ends with an error status instead of hanging the GPU.  This
 * call launches one CTA on `stream` that waits, through the same code, for a
 * barrier phase that nothing completes, giving up after `limit_us`
 * microseconds (1 to 1000000).  Afterwards gdn_device_error(stream) returns
 * GDN_ERR_TIMEOUT (and clears the word), and the CUDA context stays usable.
 * Returns GDN_ERR_INVALID_ARG for a limit outside that range (nothing is
 * launched), GDN_ERR_CUDA if the launch fails, else GDN_OK.
 */
GDN_API gdn_status gdn_selftest_bounded_wait(int limit_us, void *stream);

/*
 * gdn_prefill_noalloc: the chunked prefill (GDN_ALGO_CHUNKED) for callers that
 * cannot allocate device memory, so cannot supply the workspace gdn_prefill
 * needs: code that must not call cudaMalloc while it runs (an allocation can
 * synchronise the device and stall other work), plugins whose host framework
 * owns every device allocation, and small runtimes without a device allocator.
 * The paper has no counterpart; it is a packaging of gdn_prefill.
 *
 * Arguments, layouts and errors as for gdn_prefill, without algo and
 * workspace.  The scratch is one library-owned device array of
 * GDN_NOALLOC_SCRATCH_BYTES (97 MiB), held on every GPU that loads the library
 * until the process exits:
 *   - problems that need more scratch than that (gdn_prefill_workspace_size
 *     with GDN_ALGO_CHUNKED above GDN_NOALLOC_SCRATCH_BYTES; e.g. more than
 *     4096 tokens at 32 value heads) return GDN_ERR_WORKSPACE, nothing runs;
 *   - the first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, once per device, with that device current); make
 *     that first call before any CUDA stream capture;
 *   - every call shares the array, which keeps the last call's contents;
 *     calls whose GPU work overlaps in time (other streams, other host
 *     threads) race on it and must be serialised by the caller;
 *   - it calls no cudaMalloc, cudaFree or other allocating routine.
 */
#define GDN_NOALLOC_SCRATCH_BYTES (97ull * 1024ull * 1024ull)

GDN_API gdn_status gdn_prefill_noalloc(int n_seqs, int total_tokens, int hk, int hv, int dk, int dv,
                                       const void *q, const void *k, const void *v,
                                       const float *log_alpha, const float *beta,
                                       const float *init_state,
                                       const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                                       void *out, int out_dtype, float *final_state,
                                       int qk_norm, float q_scale, const float *norm_weight, float norm_eps,
                                       const float *gate_scale, const float *gate_bias, void *stream);

/*
 * gdn_prefill_host: gdn_prefill on inputs and outputs in HOST memory, for
 * callers whose prompts arrive in host memory and whose results go back there.
 * Enqueued on `stream`, in this order:
 *   1. copies of q_host, k_host, v_host, log_alpha_host, beta_host,
 *      init_state_host (when not NULL) and cu_seqlens_host into `staging`;
 *   2. gdn_prefill on those device copies, with its workspace also taken from
 *      `staging`;
 *   3. copies of the outputs back into out_host and, when not NULL,
 *      final_state_host.
 * Shapes, dtypes, options and errors are those of gdn_prefill; the host arrays
 * are dense with gdn_prefill's layouts and need no particular alignment.
 * norm_weight, gate_scale and gate_bias, when given, are DEVICE arrays (model
 * parameters that stay resident).  init_state_host NULL means zero initial states; final_state_host
 * NULL skips the final states.
 *
 *   staging        device memory of at least gdn_prefill_host_staging_size()
 *                  bytes for the same problem, 256-byte aligned, owned by the
 *                  caller and used by the call until its step 3 has finished
 *                  on the stream.  Its contents on entry do not matter.
 *
 * The host arrays must stay valid, and the inputs unchanged, until the stream
 * has executed the copies that read or write them.  With page-locked (pinned)
 * host memory the call returns without waiting and the copies run
 * asynchronously, so calls alternated between two streams, each with its own
 * staging, overlap one call's copies with the other's kernels.  With pageable
 * host memory the CUDA runtime may complete the copies synchronously.  All
 * arguments are validated before anything is enqueued.
 */
GDN_API size_t gdn_prefill_host_staging_size(int n_seqs, int total_tokens, int hk, int hv, int dk, int dv,
                                             const int32_t *cu_seqlens_host, int out_dtype, int with_init_state,
                                             int with_final_state, int algo, gdn_status *status);

GDN_API gdn_status gdn_prefill_host(int n_seqs, int total_tokens, int hk, int hv, int dk, int dv,
                                    const void *q_host, const void *k_host, const void *v_host,
                                    const float *log_alpha_host, const float *beta_host,
                                    const float *init_state_host, const int32_t *cu_seqlens_host,
                                    void *out_host, int out_dtype, float *final_state_host,
                                    int qk_norm, float q_scale, const float *norm_weight, float norm_eps,
                                    const float *gate_scale, const float *gate_bias,
                                    int algo, void *staging, size_t staging_bytes, void *stream);

/* Static, human-readable name of a status code. */
GDN_API const char *gdn_status_string(gdn_status status);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
GDN_API int gdn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
