// extern "C" entry points of libgdn: argument validation on the host, then a
// launch of the matching kernel on the caller's stream.  Validation never
// touches the CUDA runtime, so argument errors are reported without side
// effects (and work on machines without a GPU).
#include <math.h>
#include <string.h>

#include "gdn_internal.cuh"
#include "sm100.cuh"

namespace {

__device__ unsigned int g_device_error = 0;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool supported_dim(int d) { return d == 32 || d == 64 || d == 128; }

// [a, a + na) and [b, b + nb) byte ranges overlap?
bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

gdn_status check_heads(int hk, int hv, int dk, int dv) {
    if (hk <= 0 || hv <= 0 || dk <= 0 || dv <= 0) return GDN_ERR_INVALID_ARG;
    if (hv % hk != 0) return GDN_ERR_INVALID_ARG;
    if (dk != dv || !supported_dim(dk)) return GDN_ERR_UNSUPPORTED;
    return GDN_OK;
}

// The gate parameters come as a pair (both null: log_alpha and beta are the gates themselves).
gdn_status check_gate_params(const float *gate_scale, const float *gate_bias) {
    if ((gate_scale == nullptr) != (gate_bias == nullptr)) return GDN_ERR_INVALID_ARG;
    if (gate_scale && (!aligned16(gate_scale) || !aligned16(gate_bias))) return GDN_ERR_ALIGNMENT;
    return GDN_OK;
}

gdn_status check_cu(int n_seqs, int total_tokens, const int32_t *cu_host) {
    if (n_seqs <= 0 || total_tokens < 0 || !cu_host) return GDN_ERR_INVALID_ARG;
    if (cu_host[0] != 0 || cu_host[n_seqs] != total_tokens) return GDN_ERR_INVALID_ARG;
    for (int i = 0; i < n_seqs; ++i)
        if (cu_host[i + 1] < cu_host[i]) return GDN_ERR_INVALID_ARG;
    return GDN_OK;
}

// The algorithm GDN_ALGO_AUTO resolves to (arguments already validated); see gdn_prefill_algo in gdn.h.
int resolve_auto(int n_seqs, int hv, int dk, const int32_t *cu_host) {
    if (dk != gdn::kChunkedHeadDim) return GDN_ALGO_SCAN;
    int max_len = 0;
    for (int i = 0; i < n_seqs; ++i) max_len = cu_host[i + 1] - cu_host[i] > max_len ? cu_host[i + 1] - cu_host[i] : max_len;
    if (max_len <= 16) return GDN_ALGO_SCAN;
    if (max_len <= 32 && (long)n_seqs * hv <= 64) return GDN_ALGO_SCAN;
    return GDN_ALGO_CHUNKED;
}

// Multiprocessors of the current device (cached per device; 1 if the query fails).
int sm_count() {
    static std::atomic<int> cached[gdn::kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 1;
    const bool in_table = dev < gdn::kMaxDevices;
    if (in_table) {
        const int n = cached[dev].load(std::memory_order_relaxed);
        if (n > 0) return n;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
    if (in_table) cached[dev].store(n, std::memory_order_relaxed);
    return n;
}

// Device address of the error word of the current device.  Every device that loads the library has its own
// word; the address is looked up once per device (with that device current) and kept in a table of atomics.
unsigned int *device_error_ptr() {
    static std::atomic<unsigned int *> table[gdn::kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return nullptr;
    const bool in_table = dev < gdn::kMaxDevices;
    if (in_table) {
        unsigned int *p = table[dev].load(std::memory_order_relaxed);
        if (p) return p;
    }
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    if (in_table) table[dev].store(static_cast<unsigned int *>(p), std::memory_order_relaxed);
    return static_cast<unsigned int *>(p);
}

// Device pointers given to an entry point must belong to the current device: the kernels are launched there,
// on a stream of that device.  A pointer to host memory, to no allocation or to another GPU's memory is
// refused with GDN_ERR_INVALID_ARG before anything is launched.  While `stream` is being captured into a CUDA
// graph the query is skipped (it is not a stream operation, but a check that the capture mode refused would
// end the capture): calls recorded into a graph are the caller's to get right.
gdn_status check_on_current_device(const void *p, cudaStream_t stream) {
    if (!p) return GDN_OK;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
        cudaGetLastError();
        return GDN_ERR_CUDA;
    }
    if (cs != cudaStreamCaptureStatusNone) return GDN_OK;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return GDN_ERR_CUDA;
    }
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return GDN_ERR_INVALID_ARG;
    }
    if ((a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged) || a.device != dev)
        return GDN_ERR_INVALID_ARG;
    return GDN_OK;
}

// One CTA waits for the first phase of a shared-memory mbarrier that nothing arrives on: the same bounded
// wait and error word as every kernel of the library, with the caller's limit in place of the kernels' 1 s.
__global__ void selftest_wait_kernel(uint64_t limit_ns, unsigned int *err) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        gdn::sm100::mbar_init(&bar, 1);
        gdn::sm100::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !gdn::sm100::mbar_wait_for(&bar, 0, limit_ns)) gdn::raise_error(err, gdn::kErrTimeout);
}

}  // namespace

extern "C" {

int gdn_version(void) { return 200; }

const char *gdn_status_string(gdn_status s) {
    switch (s) {
        case GDN_OK: return "GDN_OK";
        case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG: invalid argument";
        case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED: unsupported shape, dtype or algorithm";
        case GDN_ERR_ALIGNMENT: return "GDN_ERR_ALIGNMENT: pointer not 16-byte aligned";
        case GDN_ERR_CUDA: return "GDN_ERR_CUDA: CUDA call or kernel launch failed";
        case GDN_ERR_TIMEOUT: return "GDN_ERR_TIMEOUT: a bounded device-side wait gave up";
        case GDN_ERR_INTERNAL: return "GDN_ERR_INTERNAL: device-side consistency check failed";
        case GDN_ERR_WORKSPACE: return "GDN_ERR_WORKSPACE: workspace missing or too small";
    }
    return "unknown gdn_status";
}

int gdn_prefill_algo(int n_seqs, int total_tokens, int hk, int hv, int dk, int dv, const int32_t *cu_seqlens_host) {
    if (check_heads(hk, hv, dk, dv) != GDN_OK || check_cu(n_seqs, total_tokens, cu_seqlens_host) != GDN_OK) return -1;
    return resolve_auto(n_seqs, hv, dk, cu_seqlens_host);
}

int gdn_prefill_pass_plan(int n_seqs, int total_tokens, int hv, const int32_t *cu_seqlens_host, int multiprocessors,
                          int *bucket_first_seq, int capacity) {
    if (hv < 1 || multiprocessors < 1 || !bucket_first_seq || check_cu(n_seqs, total_tokens, cu_seqlens_host) != GDN_OK)
        return -1;
    return gdn::plan_state_pass(n_seqs, cu_seqlens_host, hv, multiprocessors, bucket_first_seq, capacity);
}

size_t gdn_prefill_workspace_size(int n_seqs, int total_tokens, int hk, int hv, int dk, int dv,
                                  const int32_t *cu_seqlens_host, int algo, gdn_status *status) {
    gdn_status st = check_heads(hk, hv, dk, dv);
    if (st == GDN_OK) st = check_cu(n_seqs, total_tokens, cu_seqlens_host);
    if (st == GDN_OK && algo == GDN_ALGO_AUTO) algo = resolve_auto(n_seqs, hv, dk, cu_seqlens_host);
    if (st == GDN_OK && algo != GDN_ALGO_CHUNKED && algo != GDN_ALGO_SCAN) st = GDN_ERR_UNSUPPORTED;
    if (st == GDN_OK && algo == GDN_ALGO_CHUNKED && dk != gdn::kChunkedHeadDim) st = GDN_ERR_UNSUPPORTED;
    if (status) *status = st;
    if (st != GDN_OK || algo == GDN_ALGO_SCAN) return 0;
    return gdn::chunked_workspace_bytes(n_seqs, cu_seqlens_host, hv, dk);
}

}  // extern "C"

static gdn_status prefill_impl(int n_seqs, int total_tokens, int hk, int hv, int dk, int dv,
                       const void *q, const void *k, const void *v,
                       const float *log_alpha, const float *beta,
                       const float *init_state,
                       const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                       void *out, int out_dtype, float *final_state, int qk_norm, float q_scale,
                       const float *norm_weight, float norm_eps, const float *gate_scale, const float *gate_bias,
                       int algo, void *workspace, size_t workspace_bytes, void *stream, int phases) {
    gdn_status st = check_heads(hk, hv, dk, dv);
    if (st != GDN_OK) return st;
    if ((st = check_gate_params(gate_scale, gate_bias)) != GDN_OK) return st;
    if ((qk_norm != 0 && qk_norm != 1) || !isfinite(q_scale)) return GDN_ERR_INVALID_ARG;
    if (norm_weight && (!isfinite(norm_eps) || norm_eps < 0.f)) return GDN_ERR_INVALID_ARG;
    if (norm_weight && !aligned16(norm_weight)) return GDN_ERR_ALIGNMENT;
    if ((st = check_cu(n_seqs, total_tokens, cu_seqlens_host)) != GDN_OK) return st;
    if (out_dtype != GDN_DTYPE_BF16 && out_dtype != GDN_DTYPE_F32) return GDN_ERR_UNSUPPORTED;
    if (algo == GDN_ALGO_AUTO) algo = resolve_auto(n_seqs, hv, dk, cu_seqlens_host);
    if (algo != GDN_ALGO_CHUNKED && algo != GDN_ALGO_SCAN) return GDN_ERR_UNSUPPORTED;
    if (algo == GDN_ALGO_CHUNKED && dk != gdn::kChunkedHeadDim) return GDN_ERR_UNSUPPORTED;
    if (!cu_seqlens) return GDN_ERR_INVALID_ARG;
    if (total_tokens > 0 && (!q || !k || !v || !log_alpha || !beta || !out)) return GDN_ERR_INVALID_ARG;
    const void *ptrs[] = {q, k, v, log_alpha, beta, init_state, cu_seqlens, out, final_state, workspace};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return GDN_ERR_ALIGNMENT;

    const size_t T = (size_t)total_tokens;
    const size_t state_bytes = (size_t)n_seqs * hv * dv * dk * sizeof(float);
    const size_t out_bytes = T * hv * dv * (out_dtype == GDN_DTYPE_F32 ? 4 : 2);
    const struct { const void *p; size_t n; } inputs[] = {
        {q, T * hk * dk * 2}, {k, T * hk * dk * 2}, {v, T * hv * dv * 2},
        {log_alpha, T * hv * 4}, {beta, T * hv * 4}, {cu_seqlens, (size_t)(n_seqs + 1) * 4},
        {init_state, state_bytes}, {gate_scale, (size_t)hv * 4}, {gate_bias, (size_t)hv * 4}};
    for (const auto &in : inputs) {
        if (overlaps(out, out_bytes, in.p, in.n)) return GDN_ERR_INVALID_ARG;
        if (in.p != init_state && overlaps(final_state, state_bytes, in.p, in.n)) return GDN_ERR_INVALID_ARG;
    }
    if (final_state && init_state && final_state != init_state &&
        overlaps(final_state, state_bytes, init_state, state_bytes))
        return GDN_ERR_INVALID_ARG;
    if (overlaps(out, out_bytes, final_state, state_bytes)) return GDN_ERR_INVALID_ARG;

    size_t need = 0;
    if (algo == GDN_ALGO_CHUNKED) {
        need = gdn::chunked_workspace_bytes(n_seqs, cu_seqlens_host, hv, dk);
        if (need > 0 && (!workspace || workspace_bytes < need)) return GDN_ERR_WORKSPACE;
        if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u)) return GDN_ERR_ALIGNMENT;
        const struct { const void *p; size_t n; } all[] = {
            {q, T * hk * dk * 2}, {k, T * hk * dk * 2}, {v, T * hv * dv * 2}, {log_alpha, T * hv * 4},
            {beta, T * hv * 4}, {cu_seqlens, (size_t)(n_seqs + 1) * 4}, {init_state, state_bytes},
            {out, out_bytes}, {final_state, state_bytes}};
        for (const auto &a : all)
            if (overlaps(workspace, need, a.p, a.n)) return GDN_ERR_INVALID_ARG;
    }
    if (total_tokens == 0 && !final_state) return GDN_OK;
    {
        const cudaStream_t cs = static_cast<cudaStream_t>(stream);
        const void *anchors[] = {q, out, final_state, workspace};
        for (const void *a : anchors)
            if ((st = check_on_current_device(a, cs)) != GDN_OK) return st;
    }

    gdn::PrefillProblem p{};
    p.n_seqs = n_seqs; p.total_tokens = total_tokens; p.hk = hk; p.hv = hv; p.d = dk;
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.k = static_cast<const __nv_bfloat16 *>(k);
    p.v = static_cast<const __nv_bfloat16 *>(v);
    p.log_alpha = log_alpha; p.beta = beta; p.init_state = init_state;
    p.cu_seqlens = cu_seqlens; p.cu_seqlens_host = cu_seqlens_host;
    p.out = out; p.out_f32 = out_dtype == GDN_DTYPE_F32; p.final_state = final_state;
    p.qk_norm = qk_norm; p.q_scale = q_scale;
    p.norm_w = norm_weight; p.norm_eps = norm_eps;
    p.gate_c = gate_scale; p.gate_b = gate_bias;
    p.workspace = workspace; p.workspace_bytes = workspace_bytes;
    p.err = device_error_ptr();
    p.stream = static_cast<cudaStream_t>(stream);
    if (!p.err) return GDN_ERR_CUDA;
    cudaError_t e;
    if (algo == GDN_ALGO_SCAN) {
        // Two mappings of the direct scan.  The register scan (16 rows per CTA, three CTAs per SM) has the
        // shorter per-token chain; the row-streaming mapping needs half the CTAs and wins for short
        // sequences once the register scan would need more than one wave of CTAs.
        int max_len = 0;
        for (int i = 0; i < n_seqs; ++i)
            max_len = cu_seqlens_host[i + 1] - cu_seqlens_host[i] > max_len ? cu_seqlens_host[i + 1] - cu_seqlens_host[i]
                                                                               : max_len;
        const long scan_ctas = (long)n_seqs * hv * (dk / 16);
        e = max_len <= gdn::kShortScanTokens && scan_ctas > 3L * sm_count() ? gdn::launch_short_prefill(p)
                                                                             : gdn::launch_scan_prefill(p);
    } else {
        e = gdn::launch_chunked_prefill(p, phases);
    }
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

extern "C" {

gdn_status gdn_prefill(int n_seqs, int total_tokens, int hk, int hv, int dk, int dv,
                       const void *q, const void *k, const void *v,
                       const float *log_alpha, const float *beta,
                       const float *init_state,
                       const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                       void *out, int out_dtype, float *final_state, int qk_norm, float q_scale,
                       const float *norm_weight, float norm_eps, const float *gate_scale, const float *gate_bias,
                       int algo, void *workspace, size_t workspace_bytes, void *stream) {
    return prefill_impl(n_seqs, total_tokens, hk, hv, dk, dv, q, k, v, log_alpha, beta, init_state, cu_seqlens,
                        cu_seqlens_host, out, out_dtype, final_state, qk_norm, q_scale, norm_weight, norm_eps,
                        gate_scale, gate_bias, algo, workspace, workspace_bytes, stream, 3);
}

gdn_status gdn_prefill_chunked_phase(int phase, int n_seqs, int total_tokens, int hk, int hv, int dk, int dv,
                                     const void *q, const void *k, const void *v,
                                     const float *log_alpha, const float *beta,
                                     const float *init_state,
                                     const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                                     void *out, int out_dtype, float *final_state, int qk_norm, float q_scale,
                                     const float *norm_weight, float norm_eps, const float *gate_scale,
                                     const float *gate_bias, void *workspace, size_t workspace_bytes, void *stream) {
    if (phase != GDN_PHASE_PREP && phase != GDN_PHASE_PASS) return GDN_ERR_INVALID_ARG;
    return prefill_impl(n_seqs, total_tokens, hk, hv, dk, dv, q, k, v, log_alpha, beta, init_state, cu_seqlens,
                        cu_seqlens_host, out, out_dtype, final_state, qk_norm, q_scale, norm_weight, norm_eps,
                        gate_scale, gate_bias, GDN_ALGO_CHUNKED, workspace, workspace_bytes, stream,
                        phase == GDN_PHASE_PREP ? 1 : 2);
}

}  // extern "C"

namespace {

// Device staging area of gdn_prefill_host: every piece starts on a 256-byte boundary, the workspace last.
struct HostStaging {
    size_t q, k, v, la, b, init, cu, out, fin, ws, total;
    size_t q_n, v_n, g_n, state_n, cu_n, out_n, ws_n;
};

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

HostStaging host_staging(int n_seqs, int total_tokens, int hk, int hv, int dk, int dv, const int32_t *cu_host,
                         int out_dtype, bool with_init, bool with_final, int algo) {
    HostStaging s{};
    const size_t T = (size_t)total_tokens;
    s.q_n = T * hk * dk * 2;
    s.v_n = T * hv * dv * 2;
    s.g_n = T * hv * 4;
    s.state_n = (size_t)n_seqs * hv * dv * dk * 4;
    s.cu_n = (size_t)(n_seqs + 1) * 4;
    s.out_n = T * hv * dv * (out_dtype == GDN_DTYPE_F32 ? 4 : 2);
    s.ws_n = algo == GDN_ALGO_CHUNKED ? gdn::chunked_workspace_bytes(n_seqs, cu_host, hv, dk) : 0;
    size_t at = 0;
    s.q = at; at += round256(s.q_n);
    s.k = at; at += round256(s.q_n);
    s.v = at; at += round256(s.v_n);
    s.la = at; at += round256(s.g_n);
    s.b = at; at += round256(s.g_n);
    s.init = at; at += with_init ? round256(s.state_n) : 0;
    s.cu = at; at += round256(s.cu_n);
    s.out = at; at += round256(s.out_n);
    s.fin = at; at += with_final ? round256(s.state_n) : 0;
    s.ws = at; at += round256(s.ws_n);
    s.total = at;
    return s;
}

// Shape, option and algorithm checks shared by the two host-buffer calls; resolves GDN_ALGO_AUTO.
gdn_status check_host_problem(int n_seqs, int total_tokens, int hk, int hv, int dk, int dv, const int32_t *cu_host,
                              int out_dtype, int &algo) {
    gdn_status st = check_heads(hk, hv, dk, dv);
    if (st == GDN_OK) st = check_cu(n_seqs, total_tokens, cu_host);
    if (st != GDN_OK) return st;
    if (out_dtype != GDN_DTYPE_BF16 && out_dtype != GDN_DTYPE_F32) return GDN_ERR_UNSUPPORTED;
    if (algo == GDN_ALGO_AUTO) algo = resolve_auto(n_seqs, hv, dk, cu_host);
    if (algo != GDN_ALGO_CHUNKED && algo != GDN_ALGO_SCAN) return GDN_ERR_UNSUPPORTED;
    if (algo == GDN_ALGO_CHUNKED && dk != gdn::kChunkedHeadDim) return GDN_ERR_UNSUPPORTED;
    return GDN_OK;
}

}  // namespace

extern "C" {

size_t gdn_prefill_host_staging_size(int n_seqs, int total_tokens, int hk, int hv, int dk, int dv,
                                     const int32_t *cu_seqlens_host, int out_dtype, int with_init_state,
                                     int with_final_state, int algo, gdn_status *status) {
    gdn_status st = check_host_problem(n_seqs, total_tokens, hk, hv, dk, dv, cu_seqlens_host, out_dtype, algo);
    if (status) *status = st;
    if (st != GDN_OK) return 0;
    return host_staging(n_seqs, total_tokens, hk, hv, dk, dv, cu_seqlens_host, out_dtype, with_init_state != 0,
                        with_final_state != 0, algo)
        .total;
}

gdn_status gdn_prefill_host(int n_seqs, int total_tokens, int hk, int hv, int dk, int dv,
                            const void *q_host, const void *k_host, const void *v_host,
                            const float *log_alpha_host, const float *beta_host, const float *init_state_host,
                            const int32_t *cu_seqlens_host, void *out_host, int out_dtype, float *final_state_host,
                            int qk_norm, float q_scale, const float *norm_weight, float norm_eps,
                            const float *gate_scale, const float *gate_bias,
                            int algo, void *staging, size_t staging_bytes, void *stream) {
    gdn_status st = check_host_problem(n_seqs, total_tokens, hk, hv, dk, dv, cu_seqlens_host, out_dtype, algo);
    if (st != GDN_OK) return st;
    if ((st = check_gate_params(gate_scale, gate_bias)) != GDN_OK) return st;
    if ((qk_norm != 0 && qk_norm != 1) || !isfinite(q_scale)) return GDN_ERR_INVALID_ARG;
    if (norm_weight && (!isfinite(norm_eps) || norm_eps < 0.f)) return GDN_ERR_INVALID_ARG;
    if (norm_weight && !aligned16(norm_weight)) return GDN_ERR_ALIGNMENT;
    if (total_tokens > 0 && (!q_host || !k_host || !v_host || !log_alpha_host || !beta_host || !out_host))
        return GDN_ERR_INVALID_ARG;
    const HostStaging s = host_staging(n_seqs, total_tokens, hk, hv, dk, dv, cu_seqlens_host, out_dtype,
                                       init_state_host != nullptr, final_state_host != nullptr, algo);
    if (!staging || staging_bytes < s.total) return GDN_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(staging) & 255u) return GDN_ERR_ALIGNMENT;
    if (total_tokens == 0 && !final_state_host) return GDN_OK;
    if ((st = check_on_current_device(staging, static_cast<cudaStream_t>(stream))) != GDN_OK) return st;

    uint8_t *base = static_cast<uint8_t *>(staging);
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const struct { size_t off; const void *src; size_t n; } in[] = {
        {s.q, q_host, s.q_n}, {s.k, k_host, s.q_n}, {s.v, v_host, s.v_n}, {s.la, log_alpha_host, s.g_n},
        {s.b, beta_host, s.g_n}, {s.init, init_state_host, s.state_n}, {s.cu, cu_seqlens_host, s.cu_n}};
    for (const auto &c : in)
        if (c.src && c.n && cudaMemcpyAsync(base + c.off, c.src, c.n, cudaMemcpyHostToDevice, cs) != cudaSuccess)
            return GDN_ERR_CUDA;
    st = prefill_impl(n_seqs, total_tokens, hk, hv, dk, dv, base + s.q, base + s.k, base + s.v,
                      reinterpret_cast<const float *>(base + s.la), reinterpret_cast<const float *>(base + s.b),
                      init_state_host ? reinterpret_cast<const float *>(base + s.init) : nullptr,
                      reinterpret_cast<const int32_t *>(base + s.cu), cu_seqlens_host, base + s.out, out_dtype,
                      final_state_host ? reinterpret_cast<float *>(base + s.fin) : nullptr, qk_norm, q_scale,
                      norm_weight, norm_eps, gate_scale, gate_bias, algo, s.ws_n ? base + s.ws : nullptr, s.ws_n,
                      stream, 3);
    if (st != GDN_OK) return st;
    if (s.out_n && cudaMemcpyAsync(out_host, base + s.out, s.out_n, cudaMemcpyDeviceToHost, cs) != cudaSuccess)
        return GDN_ERR_CUDA;
    if (final_state_host &&
        cudaMemcpyAsync(final_state_host, base + s.fin, s.state_n, cudaMemcpyDeviceToHost, cs) != cudaSuccess)
        return GDN_ERR_CUDA;
    return GDN_OK;
}

gdn_status gdn_decode_step(int n, int hk, int hv, int dk, int dv, float *state,
                           const void *q, const void *k, const void *v,
                           const float *log_alpha, const float *beta,
                           void *out, int out_dtype, int qk_norm, float q_scale,
                           const float *norm_weight, float norm_eps, const float *gate_scale,
                           const float *gate_bias, void *stream) {
    gdn_status st = check_heads(hk, hv, dk, dv);
    if (st != GDN_OK) return st;
    if ((st = check_gate_params(gate_scale, gate_bias)) != GDN_OK) return st;
    if (n < 0) return GDN_ERR_INVALID_ARG;
    if ((qk_norm != 0 && qk_norm != 1) || !isfinite(q_scale)) return GDN_ERR_INVALID_ARG;
    if (norm_weight && (!isfinite(norm_eps) || norm_eps < 0.f)) return GDN_ERR_INVALID_ARG;
    if (norm_weight && !aligned16(norm_weight)) return GDN_ERR_ALIGNMENT;
    if (out_dtype != GDN_DTYPE_BF16 && out_dtype != GDN_DTYPE_F32) return GDN_ERR_UNSUPPORTED;
    if (n == 0) return GDN_OK;
    if (!state || !q || !k || !v || !log_alpha || !beta || !out) return GDN_ERR_INVALID_ARG;
    const void *ptrs[] = {state, q, k, v, log_alpha, beta, out};
    for (const void *p : ptrs)
        if (!aligned16(p)) return GDN_ERR_ALIGNMENT;
    const size_t state_bytes = (size_t)n * hv * dv * dk * 4;
    const size_t out_bytes = (size_t)n * hv * dv * (out_dtype == GDN_DTYPE_F32 ? 4 : 2);
    const struct { const void *p; size_t n; } inputs[] = {
        {q, (size_t)n * hk * dk * 2}, {k, (size_t)n * hk * dk * 2}, {v, (size_t)n * hv * dv * 2},
        {log_alpha, (size_t)n * hv * 4}, {beta, (size_t)n * hv * 4}, {out, out_bytes},
        {gate_scale, (size_t)hv * 4}, {gate_bias, (size_t)hv * 4}};
    for (const auto &in : inputs)
        if (overlaps(state, state_bytes, in.p, in.n)) return GDN_ERR_INVALID_ARG;
    if (overlaps(out, out_bytes, q, (size_t)n * hk * dk * 2) || overlaps(out, out_bytes, k, (size_t)n * hk * dk * 2) ||
        overlaps(out, out_bytes, v, (size_t)n * hv * dv * 2))
        return GDN_ERR_INVALID_ARG;
    if ((st = check_on_current_device(state, static_cast<cudaStream_t>(stream))) != GDN_OK ||
        (st = check_on_current_device(out, static_cast<cudaStream_t>(stream))) != GDN_OK)
        return st;

    gdn::DecodeProblem p{};
    p.n = n; p.hk = hk; p.hv = hv; p.d = dk; p.state = state;
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.k = static_cast<const __nv_bfloat16 *>(k);
    p.v = static_cast<const __nv_bfloat16 *>(v);
    p.log_alpha = log_alpha; p.beta = beta; p.out = out; p.out_f32 = out_dtype == GDN_DTYPE_F32;
    p.qk_norm = qk_norm; p.q_scale = q_scale;
    p.norm_w = norm_weight; p.norm_eps = norm_eps;
    p.gate_c = gate_scale; p.gate_b = gate_bias;
    p.err = device_error_ptr();
    if (!p.err) return GDN_ERR_CUDA;
    p.stream = static_cast<cudaStream_t>(stream);
    return gdn::launch_decode(p) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

gdn_status gdn_selftest_bounded_wait(int limit_us, void *stream) {
    if (limit_us < 1 || limit_us > 1000000) return GDN_ERR_INVALID_ARG;
    unsigned int *err = device_error_ptr();
    if (!err) return GDN_ERR_CUDA;
    selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>((uint64_t)limit_us * 1000ull, err);
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

gdn_status gdn_device_error(void *stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return GDN_ERR_CUDA;
    unsigned int *ptr = device_error_ptr();
    if (!ptr) return GDN_ERR_CUDA;
    unsigned int word = 0;
    if (cudaMemcpy(&word, ptr, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return GDN_ERR_CUDA;
    if (word) {
        const unsigned int zero = 0;
        if (cudaMemcpy(ptr, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return GDN_ERR_CUDA;
    }
    if (word & (gdn::kErrInternal | gdn::kErrBounds)) return GDN_ERR_INTERNAL;   // the cause, before its timeouts
    if (word & gdn::kErrTimeout) return GDN_ERR_TIMEOUT;
    return GDN_OK;
}

}  // extern "C"
