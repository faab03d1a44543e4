// gdn_prefill_noalloc: the chunked prefill with library-owned scratch, for
// callers that cannot allocate device memory.
//
// The chunked prefill needs per-chunk scratch between its two kernels.  The
// normal entry point takes that scratch from the caller.  Some callers cannot
// provide it:
//   - code that runs where allocation is forbidden or unsafe, e.g. inside a
//     serving loop that must not call cudaMalloc (which can synchronise the
//     device and stall other streams);
//   - plugins hosted by a framework that owns every device allocation and does
//     not hand out scratch buffers;
//   - small runtimes built without a device allocator.
// For them the scratch lives in one file-scope __device__ array of fixed size.
// Every GPU that loads this library holds the array until the process exits.
//
// Use rules (also stated in include/gdn.h):
//   - The first call on a device looks up the array's device address with
//     cudaGetSymbolAddress (once per device, with that device current).  Make
//     that first call before any CUDA stream capture.  First calls made at the
//     same time from several host threads are safe: each stores the same
//     address.
//   - All calls share the one array and it keeps the last call's contents;
//     nothing in it has to start at zero (each call writes all the scratch it
//     later reads).  Calls whose GPU work overlaps in time (different streams,
//     or different host threads without ordering) race on the array.
//   - Problems that need more than kNoAllocScratchBytes are rejected with
//     GDN_ERR_WORKSPACE before anything runs.
//   - No cudaMalloc, cudaFree or allocating library routine is called.
#include "gdn_internal.cuh"

namespace {

// 97 MiB = 2048 (chunk, value head) pairs of 48.5 KiB: one 4096-token prompt at
// 32 value heads, or 8192 tokens at 16.
constexpr size_t kNoAllocScratchBytes = size_t(97) << 20;
static_assert(kNoAllocScratchBytes == (size_t)GDN_NOALLOC_SCRATCH_BYTES, "header and library disagree");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch on the current device.  In host code the name
// g_noalloc_scratch is only a host-side stand-in, never a device address.  The
// table entries are atomics: host threads that make their first call on the
// same device at the same time each look the address up and store the same
// value, which is harmless.
void *scratch_device_address() {
    static std::atomic<void *> addr[gdn::kMaxDevices];
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= gdn::kMaxDevices) return nullptr;
    void *cached = addr[dev].load(std::memory_order_relaxed);
    if (cached) return cached;
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return nullptr;
    addr[dev].store(p, std::memory_order_relaxed);
    return p;
}

}  // namespace

extern "C" gdn_status gdn_prefill_noalloc(int n_seqs, int total_tokens, int hk, int hv, int dk, int dv,
                                          const void *q, const void *k, const void *v,
                                          const float *log_alpha, const float *beta,
                                          const float *init_state,
                                          const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                                          void *out, int out_dtype, float *final_state, int qk_norm,
                                          float q_scale, const float *norm_weight, float norm_eps,
                                          const float *gate_scale, const float *gate_bias, void *stream) {
    gdn_status st = GDN_OK;
    const size_t need = gdn_prefill_workspace_size(n_seqs, total_tokens, hk, hv, dk, dv, cu_seqlens_host,
                                                   GDN_ALGO_CHUNKED, &st);
    if (st != GDN_OK) return st;
    if (need > kNoAllocScratchBytes) return GDN_ERR_WORKSPACE;
    void *scratch = scratch_device_address();
    if (scratch == nullptr) return GDN_ERR_CUDA;
    return gdn_prefill(n_seqs, total_tokens, hk, hv, dk, dv, q, k, v, log_alpha, beta, init_state, cu_seqlens,
                       cu_seqlens_host, out, out_dtype, final_state, qk_norm, q_scale, norm_weight, norm_eps,
                       gate_scale, gate_bias, GDN_ALGO_CHUNKED, scratch, kNoAllocScratchBytes, stream);
}
