// Internal declarations shared by the translation units of libgdn.
// Nothing here is part of the public ABI (include/gdn.h is).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <atomic>

#include "../../include/gdn.h"

namespace gdn {

// Lowest log-decay the GPU paths use; see the gdn.h note on log_alpha.
constexpr float kLogAlphaFloor = -20.0f;
// Chunk length of the blocked evaluation, and the head size its kernels implement.
constexpr int kChunk = 64;
constexpr int kChunkedHeadDim = 128;

__device__ __forceinline__ float clamp_log_alpha(float la) { return fmaxf(la, kLogAlphaFloor); }

// Query/key preparation: with qk_norm a head vector x is used as x / sqrt(|x|^2 + kQkNormEps).
constexpr float kQkNormEps = 1e-6f;
__device__ __forceinline__ float qk_inv_norm(float sum_sq, int qk_norm) {
    return qk_norm ? rsqrtf(sum_sq + kQkNormEps) : 1.f;
}

// Gates computed from raw per-token inputs (gdn.h: gate_scale, gate_bias).  With gate parameters c, b ([hv]
// device arrays) the log_alpha and beta arrays hold the raw projections a and y of each token and value head h:
//     log_alpha = -c_h softplus(a + b_h),   beta = sigmoid(y),
// with softplus(x) = max(x, 0) + log(1 + e^{-|x|}) (no overflow, small-x tail kept).  Without them (c null)
// the arrays hold the gates themselves.  Every kernel that reads a gate goes through these two functions, so
// the preparation and state-passing kernels of the chunked path see identical values.
__device__ __forceinline__ float gate_log_alpha(float a, const float *__restrict__ c, const float *__restrict__ b,
                                                int h) {
    if (c == nullptr) return a;
    const float x = a + __ldg(b + h);
    return -__ldg(c + h) * (fmaxf(x, 0.f) + log1pf(expf(-fabsf(x))));
}
__device__ __forceinline__ float gate_beta(float y, const float *__restrict__ c) {
    return c == nullptr ? y : 1.f / (1.f + expf(-y));
}

__device__ __forceinline__ float bf16_lo(uint32_t packed) { return __uint_as_float(packed << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t packed) { return __uint_as_float(packed & 0xffff0000u); }

// Per-device host caches (kernel attributes set, symbol addresses looked up) hold at most this many devices;
// their entries are atomics, so host threads that fill the same entry at once only repeat the work.
constexpr int kMaxDevices = 256;

// Error word bits set by kernels (read back by gdn_device_error; kErrBounds is reported as GDN_ERR_INTERNAL).
enum : unsigned int { kErrTimeout = 1u, kErrInternal = 2u, kErrBounds = 4u };

__device__ __forceinline__ void raise_error(unsigned int *err, unsigned int bit) {
    if (err) atomicOr(err, bit);
}

// Bounds-checking build (compiled with -DGDN_DEBUG_BOUNDS, as libgdn_debug.so): before every global access
// whose address a kernel computes, and before every tensor-copy request, GDN_INB(last, extent, err) checks
// the highest element index the access touches against the extent of its buffer (in elements, or rows for a
// tensor copy).  An access out of range is skipped and kErrBounds is recorded in the device error word; a
// skipped tensor load leaves its barrier incomplete, so the kernel's bounded wait then ends it with
// GDN_ERR_TIMEOUT as well.  Nothing traps.  In the normal build GDN_INB is the constant true and costs nothing.
#ifdef GDN_DEBUG_BOUNDS
__device__ __forceinline__ bool in_bounds_check(long long last, long long extent, unsigned int *err) {
    if (last >= 0 && last < extent) return true;
    raise_error(err, kErrBounds);
    return false;
}
#define GDN_INB(last, extent, err) (::gdn::in_bounds_check((long long)(last), (long long)(extent), (err)))
#else
#define GDN_INB(last, extent, err) true
#endif

// Per-call plan passed to the launchers (validated on the host already).
struct PrefillProblem {
    int n_seqs, total_tokens, hk, hv, d;
    const __nv_bfloat16 *q, *k, *v;
    const float *log_alpha, *beta, *init_state;
    const int32_t *cu_seqlens;        // device
    const int32_t *cu_seqlens_host;   // host
    void *out;
    int out_f32;
    float *final_state;
    int qk_norm;        // L2-normalise q and k head vectors (x / sqrt(|x|^2 + kQkNormEps))
    float q_scale;      // then multiply q by this
    const float *norm_w;   // fused output normalisation weight [d], or null
    float norm_eps;
    const float *gate_c, *gate_b;   // gate parameters [hv] (log_alpha/beta hold raw inputs), or both null
    void *workspace;
    size_t workspace_bytes;
    unsigned int *err;
    cudaStream_t stream;
};

struct DecodeProblem {
    int n, hk, hv, d;
    float *state;
    const __nv_bfloat16 *q, *k, *v;
    const float *log_alpha, *beta;
    void *out;
    int out_f32;
    int qk_norm;
    float q_scale;
    const float *norm_w;   // fused output normalisation weight [d], or null
    float norm_eps;
    const float *gate_c, *gate_b;   // gate parameters [hv] (log_alpha/beta hold raw inputs), or both null
    unsigned int *err;
    cudaStream_t stream;
};

cudaError_t launch_decode(const DecodeProblem &p);
cudaError_t launch_scan_prefill(const PrefillProblem &p);
// The direct scan for batches whose longest sequence has at most kShortScanTokens tokens: state rows
// streamed once through all of a sequence's tokens (the decode step's mapping).
constexpr int kShortScanTokens = 32;
cudaError_t launch_short_prefill(const PrefillProblem &p);
// phases: bit 0 = per-chunk preparation, bit 1 = state passing + outputs
cudaError_t launch_chunked_prefill(const PrefillProblem &p, int phases);
size_t chunked_workspace_bytes(int n_seqs, const int32_t *cu_host, int hv, int d);
// The state pass's buckets for `sms` multiprocessors: first_seq[0..nb] (bucket b carries sequences
// [first_seq[b], first_seq[b + 1])); returns nb, or -1 when capacity < nb + 1.  Host only.
int plan_state_pass(int n_seqs, const int32_t *cu_host, int hv, int sms, int *first_seq, int capacity);

}  // namespace gdn
