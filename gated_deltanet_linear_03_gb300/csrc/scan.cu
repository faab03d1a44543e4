// Direct-scan prefill: the recurrence evaluated token by token with the state
// held in registers for the whole sequence.
//
// "Optimizing on-device inference for Apple Silicon", section "Keep recurrent
// state on chip": the state matrix is loaded into registers once, carried
// through the whole scan with partial sums exchanged by SIMD (warp) shuffles
// rather than through shared memory, and written back only at the end.  The
// same page (section "Qwen creates three workload shapes") says that whether
// this direct scan or the blocked form is faster depends on the model
// dimensions, the workload and the hardware, so the library ships both.
//
// Mapping on sm_103a: one CTA of 128 threads owns 16 consecutive value rows of
// one (sequence, value head) state; thread (r, c) holds D/8 columns of row r in
// registers, in groups of four: columns 4(c + 8m) .. 4(c + 8m) + 3 for
// m = 0 .. D/32 - 1, so that the 8 threads of a row read consecutive 8-byte
// words of a staged k or q row (no bank conflicts); a row's dot products are
// finished with three shuffle levels.  Small slices give more CTAs (two or more per SM), whose
// warps hide each other's latency on the token-serial chain.  Inputs for the
// next 64 tokens are staged into shared memory with cp.async while the current
// 64 are scanned (k.q of each token is formed once while staging); outputs are
// staged and written back as coalesced rows.
#include "gdn_internal.cuh"
#include "sm100.cuh"

namespace gdn {
namespace {

using sm100::cluster_sync;
using sm100::ld_dsmem_f32;

constexpr int kThreads = 128;
constexpr int kRows = 16;   // value rows per CTA
constexpr int kTPR = kThreads / kRows;   // threads per row
constexpr int kTB = 64;     // tokens per staged block

// PREP adds the per-token query/key preparation factors (kept out of the plain layout: it is sized to fit
// three CTAs per SM).
template <int D, bool PREP>
struct ScanSmem {
    __nv_bfloat16 k[2][kTB][D];
    __nv_bfloat16 q[2][kTB][D];
    __nv_bfloat16 v[2][kTB][kRows];
    float la[2][kTB];
    float b[2][kTB];
    float kq[kTB];              // prepared k.q of each token of the block
    float fk[PREP ? kTB : 1];   // query/key preparation factors (1/|k| or 1, q_scale/|q| or q_scale)
    float fq[PREP ? kTB : 1];
    float o[kTB][kRows];
};

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async4(void *smem, const void *gmem) {
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_prev() { asm volatile("cp.async.wait_group 1;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }

template <int D, bool PREP>
__device__ __forceinline__ void stage_block(ScanSmem<D, PREP> &sm, int buf, long t0, int nt, int hk, int hv,
                                            int hq, int h, int row0, const __nv_bfloat16 *__restrict__ q,
                                            const __nv_bfloat16 *__restrict__ k,
                                            const __nv_bfloat16 *__restrict__ v,
                                            const float *__restrict__ log_alpha,
                                            const float *__restrict__ beta, long total, unsigned int *err) {
    constexpr int QK_CHUNKS = D / 8;      // 16-byte pieces per q/k row
    constexpr int V_CHUNKS = kRows / 8;   // 16-byte pieces of the v slice
    (void)total;
    (void)err;
    for (int i = threadIdx.x; i < nt * QK_CHUNKS; i += kThreads) {
        const int t = i / QK_CHUNKS, c = i % QK_CHUNKS;
        const size_t g = ((size_t)(t0 + t) * hk + hq) * D + c * 8;
        if (!GDN_INB(g + 7, total * hk * D, err)) continue;
        cp_async16(&sm.k[buf][t][c * 8], k + g);
        cp_async16(&sm.q[buf][t][c * 8], q + g);
    }
    for (int i = threadIdx.x; i < nt * V_CHUNKS; i += kThreads) {
        const int t = i / V_CHUNKS, c = i % V_CHUNKS;
        const size_t g = ((size_t)(t0 + t) * hv + h) * D + row0 + c * 8;
        if (!GDN_INB(g + 7, total * hv * D, err)) continue;
        cp_async16(&sm.v[buf][t][c * 8], v + g);
    }
    for (int t = threadIdx.x; t < nt; t += kThreads) {
        const size_t g = (size_t)(t0 + t) * hv + h;
        if (!GDN_INB(g, total * hv, err)) continue;
        cp_async4(&sm.la[buf][t], log_alpha + g);
        cp_async4(&sm.b[buf][t], beta + g);
    }
}

// PREP: query/key preparation enabled (qk_norm, or q_scale != 1); without it the token loop is the plain one.
// NORM: fused output normalisation (launched as a cluster of the head's slices); the plain instantiation
// carries no cluster code (its presence alone slowed the plain scan by 17%).
// GATE: the gates are formed from raw inputs (gdn.h: gate_scale, gate_bias); a separate instantiation for the
// same reason (the gate code alone changed the plain scan's register allocation and cost it 11%).
template <int D, bool PREP, bool NORM, bool GATE>
__global__ void __launch_bounds__(kThreads)
scan_prefill_kernel(int total_tokens, int hk, int hv, const __nv_bfloat16 *__restrict__ q,
                    const __nv_bfloat16 *__restrict__ k, const __nv_bfloat16 *__restrict__ v,
                    const float *__restrict__ log_alpha, const float *__restrict__ beta,
                    const float *__restrict__ init_state, const int32_t *__restrict__ cu_seqlens,
                    void *__restrict__ out, int out_f32, float *__restrict__ final_state, int qk_norm,
                    float q_scale, const float *__restrict__ norm_w, float norm_eps,
                    const float *__restrict__ gate_c, const float *__restrict__ gate_b, int n_seqs,
                    unsigned int *err) {
    constexpr int COLS = D / kTPR;        // state columns per thread
    constexpr int SLICES = D / kRows;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    ScanSmem<D, PREP> &sm = *reinterpret_cast<ScanSmem<D, PREP> *>(smem_raw);

    const int slice = blockIdx.x % SLICES;
    const int h = (blockIdx.x / SLICES) % hv;
    const int n = blockIdx.x / (SLICES * hv);
    const int hq = h / (hv / hk);
    const int row0 = slice * kRows;
    const int r = threadIdx.x / kTPR, c = threadIdx.x % kTPR;

    const long tbeg = min(max((long)cu_seqlens[n], 0L), (long)total_tokens);
    const long tend = min(max((long)cu_seqlens[n + 1], tbeg), (long)total_tokens);

    // S[4m + e] is column 4(c + kTPR m) + e of row r
    float S[COLS];
    const size_t srow = (((size_t)n * hv + h) * D + row0 + r) * D + 4 * c;
    const bool state_ok = GDN_INB(srow + kTPR * (COLS - 4) + 3, (long)n_seqs * hv * D * D, err);
    (void)n_seqs;
    if (init_state && state_ok) {
#pragma unroll
        for (int j = 0; j < COLS; j += 4) {
            const float4 x = *reinterpret_cast<const float4 *>(init_state + srow + kTPR * j);
            S[j] = x.x; S[j + 1] = x.y; S[j + 2] = x.z; S[j + 3] = x.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < COLS; ++j) S[j] = 0.f;
    }

    const long ntok = tend - tbeg;
    const int nblk = (int)((ntok + kTB - 1) / kTB);
    if (nblk > 0) {
        stage_block<D, PREP>(sm, 0, tbeg, (int)min((long)kTB, ntok), hk, hv, hq, h, row0, q, k, v, log_alpha, beta,
                             total_tokens, err);
        cp_async_commit();
    }
    for (int blk = 0; blk < nblk; ++blk) {
        const int buf = blk & 1;
        const long t0 = tbeg + (long)blk * kTB;
        const int nt = (int)min((long)kTB, tend - t0);
        if (blk + 1 < nblk) {
            const long t1 = t0 + kTB;
            stage_block<D, PREP>(sm, buf ^ 1, t1, (int)min((long)kTB, tend - t1), hk, hv, hq, h, row0, q, k, v,
                           log_alpha, beta, total_tokens, err);
        }
        cp_async_commit();
        cp_async_wait_prev();
        __syncthreads();
        if (GATE) {   // gates from raw inputs: mapped once per token of the block, in place (read after the
                      // barrier that ends the k.q pass below)
            for (int t = threadIdx.x; t < nt; t += kThreads) {
                sm.la[buf][t] = gate_log_alpha(sm.la[buf][t], gate_c, gate_b, h);
                sm.b[buf][t] = gate_beta(sm.b[buf][t], gate_c);
            }
        }
        // k.q (and |k|^2, |q|^2) of every token of the block, once: 16 lanes per token, 8 tokens per round.
        // Every warp runs the same number of rounds (the shuffles need all 32 lanes); tokens past nt compute
        // nothing.
        for (int t0k = 0; t0k < nt; t0k += kThreads / 16) {
            const int t = t0k + (threadIdx.x >> 4), l = threadIdx.x & 15;
            float acc = 0.f, kk = 0.f, qq = 0.f;
            if (t < nt) {
#pragma unroll
                for (int j = 0; j < D / 16; ++j) {
                    const float kx = __bfloat162float(sm.k[buf][t][l + 16 * j]);
                    const float qx = __bfloat162float(sm.q[buf][t][l + 16 * j]);
                    acc = fmaf(kx, qx, acc);
                    kk = fmaf(kx, kx, kk);
                    qq = fmaf(qx, qx, qq);
                }
            }
#pragma unroll
            for (int off = 8; off >= 1; off >>= 1) {
                acc += __shfl_xor_sync(0xffffffffu, acc, off);
                kk += __shfl_xor_sync(0xffffffffu, kk, off);
                qq += __shfl_xor_sync(0xffffffffu, qq, off);
            }
            if (l == 0 && t < nt) {
                if (PREP) {
                    const float fk = qk_inv_norm(kk, qk_norm), fq = q_scale * qk_inv_norm(qq, qk_norm);
                    sm.fk[t] = fk;
                    sm.fq[t] = fq;
                    sm.kq[t] = acc * fk * fq;
                } else {
                    sm.kq[t] = acc;
                }
            }
        }
        __syncthreads();

        for (int t = 0; t < nt; ++t) {
            float kk[COLS], qq[COLS];
            // this thread's COLS bf16 of k and q, 4 at a time (8-byte loads, word c + kTPR j of the row)
            const uint2 *kp = reinterpret_cast<const uint2 *>(&sm.k[buf][t][0]) + c;
            const uint2 *qp = reinterpret_cast<const uint2 *>(&sm.q[buf][t][0]) + c;
#pragma unroll
            for (int j = 0; j < COLS / 4; ++j) {
                const uint2 a = kp[kTPR * j], b = qp[kTPR * j];
                kk[4 * j + 0] = bf16_lo(a.x); kk[4 * j + 1] = bf16_hi(a.x);
                kk[4 * j + 2] = bf16_lo(a.y); kk[4 * j + 3] = bf16_hi(a.y);
                qq[4 * j + 0] = bf16_lo(b.x); qq[4 * j + 1] = bf16_hi(b.x);
                qq[4 * j + 2] = bf16_lo(b.y); qq[4 * j + 3] = bf16_hi(b.y);
            }
            float sk[4] = {0.f, 0.f, 0.f, 0.f}, sq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int j = 0; j < COLS; ++j) {
                sk[j & 3] = fmaf(S[j], kk[j], sk[j & 3]);
                sq[j & 3] = fmaf(S[j], qq[j], sq[j & 3]);
            }
            float a0 = (sk[0] + sk[1]) + (sk[2] + sk[3]);
            float a1 = (sq[0] + sq[1]) + (sq[2] + sq[3]);
#pragma unroll
            for (int off = 1; off < kTPR; off <<= 1) {
                a0 += __shfl_xor_sync(0xffffffffu, a0, off);
                a1 += __shfl_xor_sync(0xffffffffu, a1, off);
            }
            // prepared k and q are fk k and fq q: scale the reduced dots and the update coefficient
            const float a2 = sm.kq[t], fk = PREP ? sm.fk[t] : 1.f, fq = PREP ? sm.fq[t] : 1.f;
            const float alpha = expf(clamp_log_alpha(sm.la[buf][t]));
            const float bt = sm.b[buf][t];
            const float u = bt * (__bfloat162float(sm.v[buf][t][r]) - alpha * (fk * a0));
            const float uk = u * fk;
#pragma unroll
            for (int j = 0; j < COLS; ++j) S[j] = fmaf(alpha, S[j], uk * kk[j]);
            if (c == 0) sm.o[t][r] = fmaf(alpha, fq * a1, u * a2);
        }
        __syncthreads();
        if (NORM) {
            // Output normalisation over the head's d rows, which the SLICES CTAs of this cluster share: each CTA
            // sums the squares of its 16 rows per token (in kq's space, free until the next block), the totals
            // meet through distributed shared memory (into this block's la, also free), and the outputs are
            // scaled in place.
            float *ps = sm.kq, *tot = sm.la[buf];
            for (int t = threadIdx.x; t < nt; t += kThreads) {
                float x = 0.f;
#pragma unroll
                for (int j = 0; j < kRows; ++j) x = fmaf(sm.o[t][j], sm.o[t][j], x);
                ps[t] = x;
            }
            cluster_sync();
            for (int t = threadIdx.x; t < nt; t += kThreads) {
                float x = 0.f;
#pragma unroll
                for (int rk = 0; rk < SLICES; ++rk) x += ld_dsmem_f32(&ps[t], rk);
                tot[t] = rsqrtf(x * (1.f / D) + norm_eps);
            }
            cluster_sync();   // every peer has read ps before the next block rewrites it; tot is complete
            for (int i = threadIdx.x; i < nt * kRows; i += kThreads) {
                const int t = i / kRows, j = i % kRows;
                sm.o[t][j] *= tot[t] * norm_w[row0 + j];
            }
            __syncthreads();
        }
        // write this block's outputs: row-contiguous 32-value pieces
        for (int i = threadIdx.x; i < nt * kRows; i += kThreads) {
            const int t = i / kRows, j = i % kRows;
            const size_t oi = ((size_t)(t0 + t) * hv + h) * D + row0 + j;
            if (!GDN_INB(oi, (long)total_tokens * hv * D, err)) continue;
            if (out_f32) reinterpret_cast<float *>(out)[oi] = sm.o[t][j];
            else reinterpret_cast<__nv_bfloat16 *>(out)[oi] = __float2bfloat16_rn(sm.o[t][j]);
        }
        __syncthreads();
    }
    cp_async_wait_all();

    if (final_state && state_ok) {
#pragma unroll
        for (int j = 0; j < COLS; j += 4)
            *reinterpret_cast<float4 *>(final_state + srow + kTPR * j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
    }
}

template <int D, bool PREP, bool NORM, bool GATE>
cudaError_t launch_scan_dpg(const PrefillProblem &p) {
    const size_t smem = sizeof(ScanSmem<D, PREP>);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static std::atomic<bool> attr_set[kMaxDevices];
    const bool cached = dev >= 0 && dev < kMaxDevices;
    if (!cached || !attr_set[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(scan_prefill_kernel<D, PREP, NORM, GATE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
        if (cached) attr_set[dev].store(true, std::memory_order_release);
    }
    // with the output normalisation the D / kRows slices of a head form one cluster
    const unsigned grid = (unsigned)(p.n_seqs * p.hv * (D / kRows));
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = D / kRows;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = p.stream;
    cfg.attrs = attr;
    cfg.numAttrs = NORM ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, scan_prefill_kernel<D, PREP, NORM, GATE>, p.total_tokens, p.hk, p.hv, p.q, p.k, p.v, p.log_alpha,
                           p.beta, p.init_state, p.cu_seqlens, p.out, p.out_f32, p.final_state, p.qk_norm, p.q_scale,
                           p.norm_w, p.norm_eps, p.gate_c, p.gate_b, p.n_seqs, p.err);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int D, bool PREP, bool NORM>
cudaError_t launch_scan_dp(const PrefillProblem &p) {
    return p.gate_c ? launch_scan_dpg<D, PREP, NORM, true>(p) : launch_scan_dpg<D, PREP, NORM, false>(p);
}

template <int D, bool NORM>
cudaError_t launch_scan_dn(const PrefillProblem &p) {
    return (p.qk_norm || p.q_scale != 1.f) ? launch_scan_dp<D, true, NORM>(p) : launch_scan_dp<D, false, NORM>(p);
}

template <int D>
cudaError_t launch_scan_d(const PrefillProblem &p) {
    return p.norm_w ? launch_scan_dn<D, true>(p) : launch_scan_dn<D, false>(p);
}

}  // namespace

cudaError_t launch_scan_prefill(const PrefillProblem &p) {
    if (p.n_seqs == 0) return cudaSuccess;
    switch (p.d) {
        case 32: return launch_scan_d<32>(p);
        case 64: return launch_scan_d<64>(p);
        case 128: return launch_scan_d<128>(p);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gdn
