// Chunked (blocked) prefill on tcgen05 tensor cores.
//
// "Optimizing on-device inference for Apple Silicon", section "Qwen creates
// three workload shapes": instead of scanning token by token, prefill may
// regroup the updates into blocks that expose matrix operations and
// token-level parallelism.  The pages give no algorithm; this file evaluates
// the blocked form of the recurrence below, which is exact up to rounding.
//
// Within a chunk of L <= 64 tokens (local index i, running log-decay
// g_i = sum_{j<=i} log alpha_j, incoming state S0 of shape dv x dk):
//   A    = strict_lower(beta_i e^{g_i - g_j} k_i.k_j)          (C x C)
//   T    = (I + A)^-1                                          (unit lower)
//   Aqk  = lower_incl(e^{g_i - g_j} q_i.k_j)
//   X    = diag(beta) V - diag(beta e^g) K S0^T                (C x dv)
//   U    = T X                                                 (delta vectors)
//   O    = diag(e^g) Q S0^T + Aqk U   = diag(e^g) Q S0^T + R X, R = Aqk T
//   S_L  = e^{g_L} S0 + U^T diag(e^{g_L - g}) K
//        = e^{g_L} S0 + (P X)^T,                    P = K^T diag(e^{g_L-g}) T
// A, T, R and P depend only on k, q and the gates, so they are computed for
// every chunk in parallel by `chunk_prep_kernel`; only the X -> state step is
// sequential over chunks, in `state_pass_kernel`.
//
// Tensor-core use (tcgen05.mma, bf16 operands, fp32 accumulation in TMEM,
// operands staged by TMA in 128B-swizzled shared memory):
//   prep:  [K;Q] K^T (exact: q/k are bf16), P = K^T (Gamma T) with Gamma T split
//          into bf16 hi + lo parts, R = Aqk T (single bf16 pass: output path only)
//   pass:  [Q;K] [S_hi;S_lo]^T, P_hi [X_hi;X_lo]^T + P_lo X_hi^T, R X_hi^T
// Everything that feeds the carried state is either an exact bf16 input or a
// value split into two bf16 terms (about 16 significant bits), so the state
// error stays far below the fp32-state tolerance; the output-only terms use
// one bf16 pass.  The triangular solve runs in fp32 on the CUDA cores.
#include <cudaTypedefs.h>

#include "gdn_internal.cuh"
#include "sm100.cuh"

namespace gdn {
namespace {

using namespace sm100;

constexpr int D = 128;          // head size of the chunked path
constexpr int C = kChunk;       // 64 tokens per chunk
constexpr int DS = 32;          // value rows per state-passing CTA
constexpr int kThreads = 128;
constexpr uint32_t kSW = kLayoutSwizzle128B;

constexpr size_t kPTile = (size_t)D * C * 2;     // P_hi or P_lo of one (chunk, head): 16 KiB
constexpr size_t kRTile = (size_t)C * C * 2;     // R of one (chunk, head): 8 KiB

// ---------------------------------------------------------------- chunk lookup
struct ChunkLoc {
    int seq, t0, len;
};

__device__ __forceinline__ void seq_range(const int32_t *cu, int n, int total, int &a, int &b) {
    a = min(max(cu[n], 0), total);
    b = min(max(cu[n + 1], a), total);
}

// Global chunk gc -> (sequence, first token, length).  Chunks are numbered
// sequence by sequence; a chunk never straddles two sequences.
__device__ bool locate_chunk(const int32_t *cu, int n_seqs, int total, int gc, ChunkLoc &loc) {
    int acc = 0;
    for (int n = 0; n < n_seqs; ++n) {
        int a, b;
        seq_range(cu, n, total, a, b);
        const int nc = (b - a + C - 1) / C;
        if (gc < acc + nc) {
            loc.seq = n;
            loc.t0 = a + (gc - acc) * C;
            loc.len = min(C, b - loc.t0);
            return true;
        }
        acc += nc;
    }
    return false;
}

__device__ int first_chunk_of(const int32_t *cu, int n, int total) {
    int acc = 0;
    for (int m = 0; m < n; ++m) {
        int a, b;
        seq_range(cu, m, total, a, b);
        acc += (b - a + C - 1) / C;
    }
    return acc;
}

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(a));
    const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(b));
    return lo | (hi << 16);
}

__device__ __forceinline__ void split_bf16(float x, __nv_bfloat16 &hi, __nv_bfloat16 &lo) {
    hi = __float2bfloat16_rn(x);
    lo = __float2bfloat16_rn(x - __bfloat162float(hi));
}

// Inclusive cumulative log-decay of the chunk for this warp: lane l covers
// tokens 2l and 2l+1; tokens at or beyond `len` contribute 0 (their g equals
// g_{len-1}).  Returns the two g values of the lane.
__device__ __forceinline__ float2 chunk_cumsum(const float *__restrict__ log_alpha, int t0, int len, int hv, int h,
                                               int lane) {
    const int i0 = 2 * lane, i1 = 2 * lane + 1;
    const float la0 = i0 < len ? fminf(clamp_log_alpha(log_alpha[(size_t)(t0 + i0) * hv + h]), 0.f) : 0.f;
    const float la1 = i1 < len ? fminf(clamp_log_alpha(log_alpha[(size_t)(t0 + i1) * hv + h]), 0.f) : 0.f;
    const float pair = la0 + la1;
    float incl = pair;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    const float excl = incl - pair;
    return make_float2(excl + la0, excl + la0 + la1);
}

// g_i of token i from the per-lane pairs produced by chunk_cumsum.
__device__ __forceinline__ float g_of(float2 g2, int i) {
    const float a = __shfl_sync(0xffffffffu, g2.x, i >> 1);
    const float b = __shfl_sync(0xffffffffu, g2.y, i >> 1);
    return (i & 1) ? b : a;
}

// ============================================================================
// Kernel 1: per-chunk preparation (parallel over chunks x value heads)
// ============================================================================
// Shared memory (offsets from a 1 KiB-aligned base):
constexpr uint32_t PREP_KQ = 0;        // kb0: K rows | Q rows, kb1: K rows | Q rows (32 KiB);
                                       // the Q halves later hold T^T hi / lo
constexpr uint32_t PREP_A = 32768;     // fp32 A [64][68]; later (Gamma T)^T hi / lo
constexpr int A_LD = 68;
constexpr uint32_t PREP_AQK = PREP_A + 64 * A_LD * 4;   // 50176: Aqk hi, Aqk lo tiles [64 x 64] bf16
constexpr uint32_t PREP_G = PREP_AQK + 16384;           // g [64], beta [64]
constexpr uint32_t PREP_SMEM = PREP_G + 512 + 1024;     // + alignment slack
constexpr uint32_t PREP_TMEM_COLS = 128;

__global__ void __launch_bounds__(kThreads)
chunk_prep_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                  const float *__restrict__ log_alpha, const float *__restrict__ beta,
                  const int32_t *__restrict__ cu, int n_seqs, int total, int hk, int hv,
                  __nv_bfloat16 *__restrict__ ws_phi, __nv_bfloat16 *__restrict__ ws_plo,
                  __nv_bfloat16 *__restrict__ ws_rhi, __nv_bfloat16 *__restrict__ ws_rlo, unsigned int *err) {
    extern __shared__ uint8_t prep_raw[];
    uint8_t *sm = align1024(prep_raw);
    __shared__ uint64_t bar_tma, bar_mma;
    __shared__ uint32_t tmem_slot;

    const int gc = blockIdx.x;
    const int h = blockIdx.y;
    const int hq = h / (hv / hk);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    ChunkLoc loc;
    if (!locate_chunk(cu, n_seqs, total, gc, loc)) return;  // uniform for the CTA
    const int t0 = loc.t0, L = loc.len;
    const uint32_t base = smem_u32(sm);
    const uint32_t tlane = (uint32_t)(32 * warp) << 16;

    if (warp == 0) {
        tmem_alloc(&tmem_slot, PREP_TMEM_COLS);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&bar_tma, 1);
        mbar_init(&bar_mma, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(&bar_tma, 32768);
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
            tma_load_2d(sm + PREP_KQ + kb * 16384, &kmap, &bar_tma, hq * D + kb * 64, t0);
            tma_load_2d(sm + PREP_KQ + kb * 16384 + 8192, &qmap, &bar_tma, hq * D + kb * 64, t0);
        }
    }
    float *g_s = reinterpret_cast<float *>(sm + PREP_G);  // [64]
    float *b_s = g_s + 64;                                // [64]
    if (warp == 0) {
        const float2 g2 = chunk_cumsum(log_alpha, t0, L, hv, h, lane);
        g_s[2 * lane] = g2.x;
        g_s[2 * lane + 1] = g2.y;
        const int i0 = 2 * lane, i1 = 2 * lane + 1;
        b_s[i0] = i0 < L ? beta[(size_t)(t0 + i0) * hv + h] : 0.f;
        b_s[i1] = i1 < L ? beta[(size_t)(t0 + i1) * hv + h] : 0.f;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    bool ok = mbar_wait(&bar_tma, 0);
    ok = __syncthreads_and(ok);
    if (ok && tid == 0) {
        // D0[128 x 64] = [K ; Q] K^T  (rows 0-63: K K^T, rows 64-127: Q K^T), exact products
        const uint32_t idesc = idesc_bf16_f32(128, 64, false, false);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = base + PREP_KQ + (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_bf16(tmem, smem_desc(off, 16, 1024, kSW), smem_desc(off, 16, 1024, kSW), idesc, kk > 0);
        }
        mma_commit(&bar_mma);
    }
    if (ok) ok = mbar_wait(&bar_mma, 0);
    ok = __syncthreads_and(ok);
    tc_fence_after();

    if (ok) {
        // A (fp32, strictly lower) from the K K^T rows; Aqk (split into bf16 hi/lo tiles) from Q K^T rows
        const int i = tid & 63;
        float vals[64];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            float v16[16];
            tmem_ld16(tmem + tlane + c * 16, v16);
#pragma unroll
            for (int j = 0; j < 16; ++j) vals[c * 16 + j] = v16[j];
        }
        const float gi = g_s[i];
        const bool row_ok = i < L;
        if (tid < 64) {
            const float bi = b_s[i];
            float *arow = reinterpret_cast<float *>(sm + PREP_A) + i * A_LD;
#pragma unroll
            for (int j = 0; j < 64; j += 4) {
                float4 a;
                a.x = (row_ok && j + 0 < i) ? bi * expf(gi - g_s[j + 0]) * vals[j + 0] : 0.f;
                a.y = (row_ok && j + 1 < i) ? bi * expf(gi - g_s[j + 1]) * vals[j + 1] : 0.f;
                a.z = (row_ok && j + 2 < i) ? bi * expf(gi - g_s[j + 2]) * vals[j + 2] : 0.f;
                a.w = (row_ok && j + 3 < i) ? bi * expf(gi - g_s[j + 3]) * vals[j + 3] : 0.f;
                *reinterpret_cast<float4 *>(arow + j) = a;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 64; j += 8) {
                uint32_t hh[4], ll[4];
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    const float x0 = (row_ok && j + e <= i) ? expf(gi - g_s[j + e]) * vals[j + e] : 0.f;
                    const float x1 = (row_ok && j + e + 1 <= i) ? expf(gi - g_s[j + e + 1]) * vals[j + e + 1] : 0.f;
                    __nv_bfloat16 a0, b0, a1, b1;
                    split_bf16(x0, a0, b0);
                    split_bf16(x1, a1, b1);
                    hh[e / 2] = (uint32_t)__bfloat16_as_ushort(a0) | ((uint32_t)__bfloat16_as_ushort(a1) << 16);
                    ll[e / 2] = (uint32_t)__bfloat16_as_ushort(b0) | ((uint32_t)__bfloat16_as_ushort(b1) << 16);
                }
                const uint32_t off = sw128_offset(i, j);
                *reinterpret_cast<uint4 *>(sm + PREP_AQK + off) = make_uint4(hh[0], hh[1], hh[2], hh[3]);
                *reinterpret_cast<uint4 *>(sm + PREP_AQK + 8192 + off) = make_uint4(ll[0], ll[1], ll[2], ll[3]);
            }
        }
    }
    __syncthreads();

    // T = (I + A)^-1, one column per thread (threads 0..63): T_ij = [i == j] - sum_{k<i} A_ik T_kj
    const int j = tid;
    float tc[64];
#pragma unroll
    for (int i = 0; i < 64; ++i) tc[i] = 0.f;
    if (ok && tid < 64) {
        const float *Ah = reinterpret_cast<const float *>(sm + PREP_A);
#pragma unroll
        for (int i = 0; i < 64; ++i) {
            // four partial sums keep the dependent FMA chains short
            float a0 = (i == j) ? 1.f : 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
            for (int k4 = 0; k4 < i; k4 += 4) {   // A_ik = 0 for k >= i and tc[k] = 0 before it is set
                const float4 a = *reinterpret_cast<const float4 *>(Ah + i * A_LD + k4);
                a0 = fmaf(-a.x, tc[k4 + 0], a0);
                a1 = fmaf(-a.y, tc[k4 + 1], a1);
                a2 = fmaf(-a.z, tc[k4 + 2], a2);
                a3 = fmaf(-a.w, tc[k4 + 3], a3);
            }
            tc[i] = (a0 + a1) + (a2 + a3);
        }
    }
    __syncthreads();  // A is no longer read: its space takes the (Gamma T)^T tiles

    // operand tiles, row j = column j of T: T^T hi/lo (for R) and (Gamma T)^T hi/lo (for P)
    if (ok && tid < 64) {
        const float gl = g_s[L - 1];
        uint8_t *tth = sm + PREP_KQ + 8192, *ttl = sm + PREP_KQ + 24576;   // over the Q rows
        uint8_t *gth = sm + PREP_A, *gtl = sm + PREP_A + 8192;
#pragma unroll
        for (int c8 = 0; c8 < 64; c8 += 8) {
            uint32_t th[4], tl[4], hh[4], ll[4];
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
                const int i0 = c8 + e, i1 = c8 + e + 1;
                __nv_bfloat16 a0, b0, a1, b1;
                split_bf16(tc[i0], a0, b0);
                split_bf16(tc[i1], a1, b1);
                th[e / 2] = (uint32_t)__bfloat16_as_ushort(a0) | ((uint32_t)__bfloat16_as_ushort(a1) << 16);
                tl[e / 2] = (uint32_t)__bfloat16_as_ushort(b0) | ((uint32_t)__bfloat16_as_ushort(b1) << 16);
                const float x0 = i0 < L ? expf(gl - g_s[i0]) * tc[i0] : 0.f;
                const float x1 = i1 < L ? expf(gl - g_s[i1]) * tc[i1] : 0.f;
                split_bf16(x0, a0, b0);
                split_bf16(x1, a1, b1);
                hh[e / 2] = (uint32_t)__bfloat16_as_ushort(a0) | ((uint32_t)__bfloat16_as_ushort(a1) << 16);
                ll[e / 2] = (uint32_t)__bfloat16_as_ushort(b0) | ((uint32_t)__bfloat16_as_ushort(b1) << 16);
            }
            const uint32_t off = sw128_offset(j, c8);
            *reinterpret_cast<uint4 *>(tth + off) = make_uint4(th[0], th[1], th[2], th[3]);
            *reinterpret_cast<uint4 *>(ttl + off) = make_uint4(tl[0], tl[1], tl[2], tl[3]);
            *reinterpret_cast<uint4 *>(gth + off) = make_uint4(hh[0], hh[1], hh[2], hh[3]);
            *reinterpret_cast<uint4 *>(gtl + off) = make_uint4(ll[0], ll[1], ll[2], ll[3]);
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (ok && tid == 0) {
        // P = K^T (Gamma T): A = K tile read MN-major (M = dk = 128), B = (Gamma T)^T hi then lo
        const uint32_t idp = idesc_bf16_f32(128, 64, true, false);
        const uint32_t gth = base + PREP_A, gtl = base + PREP_A + 8192;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            mma_bf16(tmem + 64, smem_desc(base + PREP_KQ + kk * 2048, 16384, 1024, kSW),
                     smem_desc(gth + kk * 32, 16, 1024, kSW), idp, kk > 0);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            mma_bf16(tmem + 64, smem_desc(base + PREP_KQ + kk * 2048, 16384, 1024, kSW),
                     smem_desc(gtl + kk * 32, 16, 1024, kSW), idp, 1);
        // R = Aqk T (M = 64): Aqk_hi T_hi + Aqk_hi T_lo + Aqk_lo T_hi
        const uint32_t idr = idesc_bf16_f32(64, 64, false, false);
        const uint32_t ah = base + PREP_AQK, al = base + PREP_AQK + 8192;
        const uint32_t th = base + PREP_KQ + 8192, tl = base + PREP_KQ + 24576;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            mma_bf16(tmem, smem_desc(ah + kk * 32, 16, 1024, kSW), smem_desc(th + kk * 32, 16, 1024, kSW), idr,
                     kk > 0);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            mma_bf16(tmem, smem_desc(ah + kk * 32, 16, 1024, kSW), smem_desc(tl + kk * 32, 16, 1024, kSW), idr, 1);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            mma_bf16(tmem, smem_desc(al + kk * 32, 16, 1024, kSW), smem_desc(th + kk * 32, 16, 1024, kSW), idr, 1);
        mma_commit(&bar_mma);
    }
    if (ok) ok = mbar_wait(&bar_mma, 1);
    ok = __syncthreads_and(ok);
    tc_fence_after();

    if (ok) {
        // P rows: lane d = tid holds P[d][0..63]; written as bf16 hi / lo rows of 128 bytes
        const size_t prow = ((size_t)gc * hv + h) * D + tid;
        uint4 *dh = reinterpret_cast<uint4 *>(ws_phi + prow * C);
        uint4 *dl = reinterpret_cast<uint4 *>(ws_plo + prow * C);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            float v16[16];
            tmem_ld16(tmem + tlane + 64 + c * 16, v16);
#pragma unroll
            for (int q8 = 0; q8 < 2; ++q8) {
                uint32_t hh[4], ll[4];
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    __nv_bfloat16 a0, b0, a1, b1;
                    split_bf16(v16[q8 * 8 + e], a0, b0);
                    split_bf16(v16[q8 * 8 + e + 1], a1, b1);
                    hh[e / 2] = (uint32_t)__bfloat16_as_ushort(a0) | ((uint32_t)__bfloat16_as_ushort(a1) << 16);
                    ll[e / 2] = (uint32_t)__bfloat16_as_ushort(b0) | ((uint32_t)__bfloat16_as_ushort(b1) << 16);
                }
                dh[c * 2 + q8] = make_uint4(hh[0], hh[1], hh[2], hh[3]);
                dl[c * 2 + q8] = make_uint4(ll[0], ll[1], ll[2], ll[3]);
            }
        }
        // R rows (M = 64 accumulator): row 16*warp + lane sits in lane 32*warp + lane for lane < 16
        const int r = 16 * warp + lane;
        const size_t rrow = ((size_t)gc * hv + h) * C + r;
        uint4 *rh = reinterpret_cast<uint4 *>(ws_rhi + rrow * C);
        uint4 *rl = reinterpret_cast<uint4 *>(ws_rlo + rrow * C);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            float v16[16];
            tmem_ld16(tmem + tlane + c * 16, v16);
            if (lane < 16) {
#pragma unroll
                for (int q8 = 0; q8 < 2; ++q8) {
                    uint32_t hh[4], ll[4];
#pragma unroll
                    for (int e = 0; e < 8; e += 2) {
                        __nv_bfloat16 a0, b0, a1, b1;
                        split_bf16(v16[q8 * 8 + e], a0, b0);
                        split_bf16(v16[q8 * 8 + e + 1], a1, b1);
                        hh[e / 2] = (uint32_t)__bfloat16_as_ushort(a0) | ((uint32_t)__bfloat16_as_ushort(a1) << 16);
                        ll[e / 2] = (uint32_t)__bfloat16_as_ushort(b0) | ((uint32_t)__bfloat16_as_ushort(b1) << 16);
                    }
                    rh[c * 2 + q8] = make_uint4(hh[0], hh[1], hh[2], hh[3]);
                    rl[c * 2 + q8] = make_uint4(ll[0], ll[1], ll[2], ll[3]);
                }
            }
        }
    } else if (tid == 0) {
        raise_error(err, kErrTimeout);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, PREP_TMEM_COLS);
}

// ============================================================================
// Kernel 2: state passing + outputs (sequential over chunks)
// ============================================================================
// One pipeline stage: Q|K 32 KiB, P_hi 16, P_lo 16, R_hi 16, R_lo 16 KiB (the R tiles hold 64 rows
// loaded per chunk and 64 zero rows, so that R feeds an M = 128 MMA whose upper rows are unused).
constexpr uint32_t PASS_STAGE = 98304;
constexpr uint32_t ST_QK = 0, ST_PH = 32768, ST_PL = 49152, ST_RH = 65536, ST_RL = 81920;
constexpr uint32_t PASS_SOP = 2 * PASS_STAGE;      // [S_hi ; S_lo] tile, 2 k-blocks x 8 KiB
constexpr uint32_t PASS_XOP = PASS_SOP + 16384;    // [X_hi ; X_lo] tile [64 x 64] bf16
constexpr uint32_t PASS_SMEM = PASS_XOP + 8192 + 1024;
constexpr uint32_t kStageTx = 32768 + 16384 + 16384 + 8192 + 8192;
constexpr uint32_t PASS_TMEM_COLS = 256;

__device__ __forceinline__ void pass_issue_loads(uint8_t *st, uint64_t *bar, const CUtensorMap *qmap,
                                                 const CUtensorMap *kmap, const CUtensorMap *phmap,
                                                 const CUtensorMap *plmap, const CUtensorMap *rhmap,
                                                 const CUtensorMap *rlmap, int hq, int t0, int gc, int hv, int h) {
    mbar_arrive_expect_tx(bar, kStageTx);
#pragma unroll
    for (int kb = 0; kb < 2; ++kb) {
        tma_load_2d(st + ST_QK + kb * 16384, qmap, bar, hq * D + kb * 64, t0);
        tma_load_2d(st + ST_QK + kb * 16384 + 8192, kmap, bar, hq * D + kb * 64, t0);
    }
    const int prow = (gc * hv + h) * D;
    tma_load_2d(st + ST_PH, phmap, bar, 0, prow);
    tma_load_2d(st + ST_PL, plmap, bar, 0, prow);
    tma_load_2d(st + ST_RH, rhmap, bar, 0, (gc * hv + h) * C);
    tma_load_2d(st + ST_RL, rlmap, bar, 0, (gc * hv + h) * C);
}

// Per-chunk inputs that are read with plain loads (gates, beta, this thread's v
// row); loaded one chunk ahead so that their latency is off the state chain.
struct ChunkInputs {
    float la0, la1;   // log_alpha of tokens 2*lane, 2*lane+1 (raw; 0 past the end)
    float b;          // beta of this thread's token row (warps 2, 3)
    uint4 v[DS / 8];  // 32 bf16 of this thread's v row slice (warps 2, 3)
};

__device__ __forceinline__ void load_chunk_inputs(ChunkInputs &in, const float *__restrict__ log_alpha,
                                                  const float *__restrict__ beta, const __nv_bfloat16 *__restrict__ v,
                                                  int t0, int L, int hv, int h, int row0, int lane, int warp, int i) {
    const int i0 = 2 * lane, i1 = 2 * lane + 1;
    in.la0 = i0 < L ? log_alpha[(size_t)(t0 + i0) * hv + h] : 0.f;
    in.la1 = i1 < L ? log_alpha[(size_t)(t0 + i1) * hv + h] : 0.f;
    in.b = 0.f;
#pragma unroll
    for (int q4 = 0; q4 < DS / 8; ++q4) in.v[q4] = make_uint4(0, 0, 0, 0);
    if (warp >= 2 && i < L) {
        in.b = beta[(size_t)(t0 + i) * hv + h];
        const uint4 *vp = reinterpret_cast<const uint4 *>(v + ((size_t)(t0 + i) * hv + h) * D + row0);
#pragma unroll
        for (int q4 = 0; q4 < DS / 8; ++q4) in.v[q4] = vp[q4];
    }
}

// Inclusive cumulative log-decay from already loaded pairs (see chunk_cumsum).
__device__ __forceinline__ float2 cumsum_pairs(float la0_raw, float la1_raw, int len, int lane) {
    const int i0 = 2 * lane, i1 = 2 * lane + 1;
    const float la0 = i0 < len ? fminf(clamp_log_alpha(la0_raw), 0.f) : 0.f;
    const float la1 = i1 < len ? fminf(clamp_log_alpha(la1_raw), 0.f) : 0.f;
    const float pair = la0 + la1;
    float incl = pair;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    const float excl = incl - pair;
    return make_float2(excl + la0, excl + la0 + la1);
}

// Outputs of one chunk: O_i = e^{g_i} (Q S^T)_i (in qs) + (R X)_i (TMEM columns 128..191).
__device__ __forceinline__ void store_outputs(float (&qs)[DS], uint32_t tmem_row, int i, int L, int t0, int hv,
                                              int h, int row0, void *__restrict__ out, int out_f32) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        float a[16], b[16];
        tmem_ld16(tmem_row + 128 + half * 16, a);   // R_hi X_hi + R_lo X_hi
        tmem_ld16(tmem_row + 160 + half * 16, b);   // R_hi X_lo
#pragma unroll
        for (int e = 0; e < 16; ++e) qs[half * 16 + e] += a[e] + b[e];
    }
    if (i < L) {
        const size_t o = ((size_t)(t0 + i) * hv + h) * D + row0;
        if (out_f32) {
            float4 *op = reinterpret_cast<float4 *>(reinterpret_cast<float *>(out) + o);
#pragma unroll
            for (int e = 0; e < DS / 4; ++e) op[e] = make_float4(qs[4 * e], qs[4 * e + 1], qs[4 * e + 2], qs[4 * e + 3]);
        } else {
            uint4 *op = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(out) + o);
#pragma unroll
            for (int e = 0; e < DS / 8; ++e)
                op[e] = make_uint4(pack_bf16(qs[8 * e], qs[8 * e + 1]), pack_bf16(qs[8 * e + 2], qs[8 * e + 3]),
                                   pack_bf16(qs[8 * e + 4], qs[8 * e + 5]), pack_bf16(qs[8 * e + 6], qs[8 * e + 7]));
        }
    }
}

__global__ void __launch_bounds__(kThreads)
state_pass_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                  const __grid_constant__ CUtensorMap phmap, const __grid_constant__ CUtensorMap plmap,
                  const __grid_constant__ CUtensorMap rhmap, const __grid_constant__ CUtensorMap rlmap,
                  const __nv_bfloat16 *__restrict__ v,
                  const float *__restrict__ log_alpha, const float *__restrict__ beta,
                  const float *__restrict__ init_state, const int32_t *__restrict__ cu, int n_seqs, int total,
                  int nch, int hk, int hv, void *__restrict__ out, int out_f32, float *__restrict__ final_state,
                  unsigned int *err) {
    extern __shared__ uint8_t pass_raw[];
    uint8_t *sm = align1024(pass_raw);
    __shared__ uint64_t bar_tma[2], bar_mma;
    __shared__ uint32_t tmem_slot;

    constexpr int SLICES = D / DS;
    const int slice = blockIdx.x % SLICES;
    const int h = (blockIdx.x / SLICES) % hv;
    const int n = blockIdx.x / (SLICES * hv);
    const int hq = h / (hv / hk);
    const int row0 = slice * DS;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int i = tid & 63;   // token row of this thread in the D1 / D4 accumulators
    const uint32_t base = smem_u32(sm);

    int ta, tb;
    seq_range(cu, n, total, ta, tb);
    const int nchunks = (tb - ta + C - 1) / C;
    const int gc0 = first_chunk_of(cu, n, total);
    bool ok = gc0 + nchunks <= nch;
    if (!ok && tid == 0) raise_error(err, kErrInternal);

    if (warp == 0) {
        tmem_alloc(&tmem_slot, PASS_TMEM_COLS);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&bar_tma[0], 1);
        mbar_init(&bar_tma[1], 1);
        mbar_init(&bar_mma, 1);
        fence_mbar_init();
        if (ok && nchunks > 0) {
            tma_prefetch_desc(&qmap);
            tma_prefetch_desc(&kmap);
            tma_prefetch_desc(&phmap);
            tma_prefetch_desc(&plmap);
            tma_prefetch_desc(&rhmap);
            tma_prefetch_desc(&rlmap);
            pass_issue_loads(sm, &bar_tma[0], &qmap, &kmap, &phmap, &plmap, &rhmap, &rlmap, hq, ta, gc0, hv, h);
        }
    }
    ChunkInputs nxt;
    if (ok && nchunks > 0) load_chunk_inputs(nxt, log_alpha, beta, v, ta, min(C, tb - ta), hv, h, row0, lane, warp, i);

    // state columns: thread d = tid holds S[row0 + r][d] for r < 32
    const int d = tid;
    float S[DS];
    const size_t sbase = (((size_t)n * hv + h) * D + row0) * D + d;
#pragma unroll
    for (int r = 0; r < DS; ++r) S[r] = init_state ? init_state[sbase + (size_t)r * D] : 0.f;

    // zero the padding rows of the R tiles once (rows 64..127 feed only unused accumulator rows)
    for (int x = tid; x < 4 * 512; x += kThreads) {
        const int st = x / 1024, t = (x / 512) & 1, o = x % 512;
        reinterpret_cast<uint4 *>(sm + st * PASS_STAGE + (t ? ST_RL : ST_RH) + 8192)[o] = make_uint4(0, 0, 0, 0);
    }

    auto write_sop = [&]() {
        const int kb = d >> 6, col = d & 63;
        uint8_t *t = sm + PASS_SOP + kb * 8192;
#pragma unroll
        for (int r = 0; r < DS; ++r) {
            __nv_bfloat16 hi, lo;
            split_bf16(S[r], hi, lo);
            *reinterpret_cast<__nv_bfloat16 *>(t + sw128_offset(r, col)) = hi;
            *reinterpret_cast<__nv_bfloat16 *>(t + sw128_offset(DS + r, col)) = lo;
        }
    };
    write_sop();
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    const uint32_t tlane = (uint32_t)(32 * warp) << 16;

    float qs[DS];
    int c = 0, prev_t0 = 0, prev_L = 0;
    for (; ok && c < nchunks; ++c) {
        const int s = c & 1;
        const int t0 = ta + c * C, L = min(C, tb - t0);
        const int gc = gc0 + c;
        const ChunkInputs cur = nxt;

        if (tid == 0 && c + 1 < nchunks)
            pass_issue_loads(sm + (s ^ 1) * PASS_STAGE, &bar_tma[s ^ 1], &qmap, &kmap, &phmap, &plmap, &rhmap,
                             &rlmap, hq, t0 + C, gc + 1, hv, h);
        if (c + 1 < nchunks)
            load_chunk_inputs(nxt, log_alpha, beta, v, t0 + C, min(C, tb - t0 - C), hv, h, row0, lane, warp, i);

        ok = mbar_wait(&bar_tma[s], (c >> 1) & 1);
        ok = __syncthreads_and(ok);
        if (!ok) break;
        if (tid == 0) {
            // D1[128 x 64] = [Q ; K] [S_hi ; S_lo]^T
            const uint32_t idesc = idesc_bf16_f32(128, 64, false, false);
            const uint32_t qk = base + s * PASS_STAGE + ST_QK, sop = base + PASS_SOP;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_bf16(tmem, smem_desc(qk + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024, kSW),
                         smem_desc(sop + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024, kSW), idesc, kk > 0);
            mma_commit(&bar_mma);
        }
        // outputs of the previous chunk, while this chunk's first MMA runs
        if (c > 0 && warp < 2) store_outputs(qs, tmem + tlane, i, prev_L, prev_t0, hv, h, row0, out, out_f32);

        const float2 g2 = cumsum_pairs(cur.la0, cur.la1, L, lane);
        const float gL = g_of(g2, L - 1);
        const float gi = g_of(g2, i);

        ok = mbar_wait(&bar_mma, 0);
        tc_fence_before();
        ok = __syncthreads_and(ok);
        if (!ok) break;
        tc_fence_after();

        {
            float a[16], b[16];
            const float eg = expf(gi);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                tmem_ld16(tmem + tlane + half * 16, a);         // x S_hi^T
                tmem_ld16(tmem + tlane + 32 + half * 16, b);    // x S_lo^T
#pragma unroll
                for (int e = 0; e < 16; ++e) qs[half * 16 + e] = a[e] + b[e];
            }
            if (warp >= 2) {
                // X_i = beta_i (v_i - e^{g_i} (K S^T)_i), split into bf16 hi/lo, column i of the X tile
                const float bi = cur.b, be = cur.b * eg;
#pragma unroll
                for (int q4 = 0; q4 < DS / 8; ++q4) {
                    const uint4 x = cur.v[q4];
                    const float vv[8] = {bf16_lo(x.x), bf16_hi(x.x), bf16_lo(x.y), bf16_hi(x.y),
                                         bf16_lo(x.z), bf16_hi(x.z), bf16_lo(x.w), bf16_hi(x.w)};
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int r = q4 * 8 + e;
                        const float xv = bi * vv[e] - be * qs[r];
                        __nv_bfloat16 hi, lo;
                        split_bf16(xv, hi, lo);
                        *reinterpret_cast<__nv_bfloat16 *>(sm + PASS_XOP + sw128_offset(r, i)) = hi;
                        *reinterpret_cast<__nv_bfloat16 *>(sm + PASS_XOP + sw128_offset(DS + r, i)) = lo;
                    }
                }
            } else {
#pragma unroll
                for (int r = 0; r < DS; ++r) qs[r] *= eg;       // e^{g_i} (Q S^T)_i
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();

        if (tid == 0) {
            const uint32_t ph = base + s * PASS_STAGE + ST_PH, pl = base + s * PASS_STAGE + ST_PL;
            const uint32_t rh = base + s * PASS_STAGE + ST_RH, rl = base + s * PASS_STAGE + ST_RL;
            const uint32_t xop = base + PASS_XOP;
            const uint32_t id64 = idesc_bf16_f32(128, 64, false, false);
            const uint32_t id32 = idesc_bf16_f32(128, 32, false, false);
            // D3[dk x 64] = P_hi [X_hi ; X_lo]^T  (+ P_lo X_hi^T into the first 32 columns)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16(tmem + 64, smem_desc(ph + kk * 32, 16, 1024, kSW), smem_desc(xop + kk * 32, 16, 1024, kSW),
                         id64, kk > 0);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16(tmem + 64, smem_desc(pl + kk * 32, 16, 1024, kSW), smem_desc(xop + kk * 32, 16, 1024, kSW),
                         id32, 1);
            // D4[64(+64 pad) x 64] = R_hi [X_hi ; X_lo]^T  (+ R_lo X_hi^T into the first 32 columns)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16(tmem + 128, smem_desc(rh + kk * 32, 16, 1024, kSW), smem_desc(xop + kk * 32, 16, 1024, kSW),
                         id64, kk > 0);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16(tmem + 128, smem_desc(rl + kk * 32, 16, 1024, kSW), smem_desc(xop + kk * 32, 16, 1024, kSW),
                         id32, 1);
            mma_commit(&bar_mma);
        }
        ok = mbar_wait(&bar_mma, 1);
        ok = __syncthreads_and(ok);
        if (!ok) break;
        tc_fence_after();

        // state: S[r][d] <- e^{g_L} S[r][d] + D3[d][r] + D3[d][32 + r]
        const float eL = expf(gL);
        {
            float a[16], b[16];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                tmem_ld16(tmem + tlane + 64 + half * 16, a);
                tmem_ld16(tmem + tlane + 96 + half * 16, b);
#pragma unroll
                for (int e = 0; e < 16; ++e) S[half * 16 + e] = fmaf(eL, S[half * 16 + e], a[e] + b[e]);
            }
        }
        write_sop();
        prev_t0 = t0;
        prev_L = L;
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }

    if (!ok) {
        if (tid == 0) {
            raise_error(err, kErrTimeout);
            // let a prefetch that may still be in flight land before the CTA exits
            if (c + 1 < nchunks) mbar_wait(&bar_tma[(c + 1) & 1], ((c + 1) >> 1) & 1);
        }
    } else {
        if (nchunks > 0 && warp < 2) store_outputs(qs, tmem + tlane, i, prev_L, prev_t0, hv, h, row0, out, out_f32);
        if (final_state) {
#pragma unroll
            for (int r = 0; r < DS; ++r) final_state[sbase + (size_t)r * D] = S[r];
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, PASS_TMEM_COLS);
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 2-D bf16 view [rows, cols] with row pitch `pitch_elems`, box [box_rows, 64], 128B swizzle.
bool make_map(CUtensorMap *m, const void *ptr, uint64_t rows, uint64_t cols, uint64_t pitch_elems,
              uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {pitch_elems * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

long total_chunks(int n_seqs, const int32_t *cu_host) {
    long nch = 0;
    for (int n = 0; n < n_seqs; ++n) nch += (cu_host[n + 1] - cu_host[n] + C - 1) / C;
    return nch;
}

}  // namespace

size_t chunked_workspace_bytes(int n_seqs, const int32_t *cu_host, int hv, int d) {
    if (d != D) return 0;
    const long nch = total_chunks(n_seqs, cu_host);
    return (size_t)nch * hv * (2 * kPTile + 2 * kRTile);
}

cudaError_t launch_chunked_prefill(const PrefillProblem &p, int phases) {
    if (p.d != D) return cudaErrorNotSupported;
    const long nch = total_chunks(p.n_seqs, p.cu_seqlens_host);
    if (nch > 0x7fffffffL / (p.hv * D)) return cudaErrorInvalidValue;
    // workspace: P_hi | P_lo  [nch][hv][D][C]  then R_hi | R_lo  [nch][hv][C][C]  (bf16)
    __nv_bfloat16 *phi = static_cast<__nv_bfloat16 *>(p.workspace);
    __nv_bfloat16 *plo = phi + (size_t)nch * p.hv * D * C;
    __nv_bfloat16 *rhi = plo + (size_t)nch * p.hv * D * C;
    __nv_bfloat16 *rlo = rhi + (size_t)nch * p.hv * C * C;

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static bool attrs_set[128] = {};
    if (dev < 128 && !attrs_set[dev]) {
        e = cudaFuncSetAttribute(chunk_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, PREP_SMEM);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(state_pass_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, PASS_SMEM);
        if (e != cudaSuccess) return e;
        attrs_set[dev] = true;
    }

    CUtensorMap qmap{}, kmap{}, phmap{}, plmap{}, rhmap{}, rlmap{};
    if (p.total_tokens > 0 && nch > 0) {
        const uint64_t T = (uint64_t)p.total_tokens;
        const uint64_t rows_p = (uint64_t)nch * p.hv * D, rows_r = (uint64_t)nch * p.hv * C;
        if (!make_map(&qmap, p.q, T, (uint64_t)p.hk * D, (uint64_t)p.hk * D, 64) ||
            !make_map(&kmap, p.k, T, (uint64_t)p.hk * D, (uint64_t)p.hk * D, 64) ||
            !make_map(&phmap, phi, rows_p, C, C, 128) || !make_map(&plmap, plo, rows_p, C, C, 128) ||
            !make_map(&rhmap, rhi, rows_r, C, C, 64) || !make_map(&rlmap, rlo, rows_r, C, C, 64))
            return cudaErrorInvalidValue;
    }

    if ((phases & 1) && nch > 0) {
        dim3 grid((unsigned)nch, (unsigned)p.hv);
        chunk_prep_kernel<<<grid, kThreads, PREP_SMEM, p.stream>>>(qmap, kmap, p.log_alpha, p.beta, p.cu_seqlens,
                                                                   p.n_seqs, p.total_tokens, p.hk, p.hv, phi, plo,
                                                                   rhi, rlo, p.err);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (phases & 2) {
        const unsigned grid2 = (unsigned)(p.n_seqs * p.hv * (D / DS));
        state_pass_kernel<<<grid2, kThreads, PASS_SMEM, p.stream>>>(
            qmap, kmap, phmap, plmap, rhmap, rlmap, p.v, p.log_alpha, p.beta, p.init_state, p.cu_seqlens, p.n_seqs,
            p.total_tokens, (int)nch, p.hk, p.hv, p.out, p.out_f32, p.final_state, p.err);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace gdn
