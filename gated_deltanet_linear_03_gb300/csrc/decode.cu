// Batch decode step: one token for each of n independent Gated DeltaNet states.
//
// "Optimizing on-device inference for Apple Silicon", section "Decode:
// minimise the bytes moved per token" notes that batch-1 decode is bound by
// the bytes moved per token; for this layer those bytes are the fp32 state,
// read once and written once.  The kernel therefore streams every state row
// exactly once: a row of dk fp32 values is spread over dk/4 lanes (one 16-byte
// load each), the two dot products S k and S q of a row are finished with warp
// shuffles, and the updated row is written back from the same registers.  For
// a row s (one value index i) of one head:
//     sk = s.k,  sq = s.q
//     u  = beta (v_i - alpha sk)                 (delta)
//     s' = alpha s + u k                         (new row)
//     o_i = s'.q = alpha sq + u (k.q)            (output after the update)
// With query/key preparation (qk_norm, q_scale) k and q stand for f_k k and f_q q, where f_k = 1/|k| and
// f_q = q_scale/|q| (or 1 and q_scale); the factors are applied to the reduced dot products and to the
// update coefficient (s' = alpha s + (u f_k) k), never element by element.
// The section "Reduce intermediate and state traffic" asks for exactly this
// fusion: the temporaries never leave registers.
#include "gdn_internal.cuh"
#include "sm100.cuh"

namespace gdn {
namespace {

using sm100::cluster_sync;
using sm100::ld_dsmem_f32;

constexpr int kRowsPerGroup = 8;   // rows each lane group carries at once
constexpr int kThreads = 128;

// Threads of a decode CTA: 128 (32 rows at d = 128), except that with the output normalisation a d = 128 head
// is one CTA of 512 threads, so that its sum of squares is a CTA reduction (at d = 32 and 64 a 128-thread CTA
// already holds whole heads).  Both keep 32 warps per SM.
template <int D, bool NORM>
__host__ __device__ constexpr int decode_threads() { return (NORM && D == 128) ? 512 : kThreads; }

// Reduce 16 per-lane partial sums over groups of LPR lanes by recursive
// halving: each round a lane keeps half of its values and receives the
// partner's partials for that half.  Afterwards lane `g` of a group holds the
// complete sums of indices [g*16/LPR, g*16/LPR + max(1, 16/LPR)).
template <int LPR>
__device__ __forceinline__ void reduce16(float (&v)[16], int lane) {
    int n = 16;
#pragma unroll
    for (int off = LPR / 2; off >= 1; off >>= 1) {
        if (n > 1) {
            const int half = n / 2;
            const bool upper = (lane & off) != 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (i < half) {
                    const float send = upper ? v[i] : v[i + half];
                    const float keep = upper ? v[i + half] : v[i];
                    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
                }
            }
            n = half;
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
        }
    }
}

// NORM: fuse the output normalisation o <- o / sqrt(mean_head(o^2) + eps) * w.  Each warp's rows belong to
// one head; a head is one warp (d = 32) or one CTA (d = 64: 128 threads; d = 128: 512 threads), so the
// head's sum of squares is a warp or CTA reduction.  (A d = 128 head used to span a cluster of four
// 128-thread CTAs, whose two cluster barrier rounds per step cost 0.2 of the HBM rate.)
// PREP: query/key preparation (qk_norm, or q_scale != 1); the plain instantiation has none of its arithmetic.
// GATE: the gates are formed from raw inputs (gdn.h: gate_scale, gate_bias); the plain instantiation has no
// gate code.
template <int D, bool PREP, bool NORM, bool GATE>
__global__ void __launch_bounds__(decode_threads<D, NORM>())
decode_step_kernel(int total_rows, int hk, int hv, float *__restrict__ state,
                   const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                   const __nv_bfloat16 *__restrict__ v, const float *__restrict__ log_alpha,
                   const float *__restrict__ beta, void *__restrict__ out, int out_f32, int qk_norm,
                   float q_scale, const float *__restrict__ norm_w, float norm_eps,
                   const float *__restrict__ gate_c, const float *__restrict__ gate_b, unsigned int *err) {
    constexpr int LPR = D / 4;                  // lanes per row
    constexpr int GROUPS = 32 / LPR;            // lane groups per warp
    constexpr int WARP_ROWS = GROUPS * kRowsPerGroup;
    constexpr int NT = decode_threads<D, NORM>();
    constexpr int PER = (16 / LPR) > 0 ? (16 / LPR) : 1;  // sums held per lane after reduce16

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int group = lane / LPR, gl = lane % LPR;
    const long row0 = ((long)blockIdx.x * (NT / 32) + warp) * WARP_ROWS + group * kRowsPerGroup;
    // whole group out of range (8 | D keeps groups in one head).  With NORM and d >= 64 the grid covers the
    // rows exactly (the host checks), so no thread of a CTA that meets a barrier below leaves early.
    if (row0 >= total_rows) return;

    const long head = row0 / D;                 // flat (n, h)
    const int h = (int)(head % hv);
    const long nb = head / hv;
    const int hq = h / (hv / hk);
    const int row_in_head = (int)(row0 % D);

    // extents (elements) of the buffers, for the bounds-checking build
    const long n_states = (long)total_rows / ((long)hv * D);
    const long state_n = (long)total_rows * D, qk_n = n_states * hk * D, v_n = n_states * hv * D;
    (void)state_n; (void)qk_n; (void)v_n;

    // q, k slice of this lane: 4 bf16 = 8 bytes
    const size_t qk_off = ((size_t)nb * hk + hq) * D + gl * 4;
    const bool qk_ok = GDN_INB(qk_off + 3, qk_n, err);
    const uint2 kraw = qk_ok ? *reinterpret_cast<const uint2 *>(k + qk_off) : make_uint2(0, 0);
    const uint2 qraw = qk_ok ? *reinterpret_cast<const uint2 *>(q + qk_off) : make_uint2(0, 0);
    const float kv[4] = {bf16_lo(kraw.x), bf16_hi(kraw.x), bf16_lo(kraw.y), bf16_hi(kraw.y)};
    const float qv[4] = {bf16_lo(qraw.x), bf16_hi(qraw.x), bf16_lo(qraw.y), bf16_hi(qraw.y)};

    float4 s[kRowsPerGroup];
    float4 *srow = reinterpret_cast<float4 *>(state + (size_t)row0 * D) + gl;
    const bool state_ok = GDN_INB((row0 + kRowsPerGroup - 1) * D + gl * 4 + 3, state_n, err);
#pragma unroll
    for (int i = 0; i < kRowsPerGroup; ++i)
        s[i] = state_ok ? __ldcs(srow + (size_t)i * (D / 4)) : make_float4(0.f, 0.f, 0.f, 0.f);

    // k.q over the head (same for every row of the group), and the preparation factors of k and q
    float kq = kv[0] * qv[0] + kv[1] * qv[1] + kv[2] * qv[2] + kv[3] * qv[3];
    float fk = 1.f, fq = PREP ? q_scale : 1.f;
    if (PREP && qk_norm) {
        float kk = kv[0] * kv[0] + kv[1] * kv[1] + kv[2] * kv[2] + kv[3] * kv[3];
        float qq = qv[0] * qv[0] + qv[1] * qv[1] + qv[2] * qv[2] + qv[3] * qv[3];
#pragma unroll
        for (int off = LPR / 2; off >= 1; off >>= 1) {
            kq += __shfl_xor_sync(0xffffffffu, kq, off);
            kk += __shfl_xor_sync(0xffffffffu, kk, off);
            qq += __shfl_xor_sync(0xffffffffu, qq, off);
        }
        fk = qk_inv_norm(kk, 1);
        fq = q_scale * qk_inv_norm(qq, 1);
    } else {
#pragma unroll
        for (int off = LPR / 2; off >= 1; off >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, off);
    }
    if (PREP) kq *= fk * fq;

    const bool gate_ok = GDN_INB(head, n_states * hv, err);
    float la_raw = gate_ok ? log_alpha[head] : 0.f, b = gate_ok ? beta[head] : 0.f;
    if (GATE) {
        la_raw = gate_log_alpha(la_raw, gate_c, gate_b, h);
        b = gate_beta(b, gate_c);
    }
    const float alpha = __expf(clamp_log_alpha(la_raw));

    float part[16];
#pragma unroll
    for (int i = 0; i < kRowsPerGroup; ++i) {
        part[i] = s[i].x * kv[0] + s[i].y * kv[1] + s[i].z * kv[2] + s[i].w * kv[3];
        part[8 + i] = s[i].x * qv[0] + s[i].y * qv[1] + s[i].z * qv[2] + s[i].w * qv[3];
    }
    reduce16<LPR>(part, lane);

    // v values of the group's rows, one per holder lane
    const __nv_bfloat16 *vrow = v + (size_t)head * D + row_in_head;
    const int my_base = gl * 16 / LPR;
    const int group_lane0 = group * LPR;
    float u[kRowsPerGroup];
#pragma unroll
    for (int i = 0; i < kRowsPerGroup; ++i) {
        // holder of sum index i (sk_i) and 8 + i (sq_i) within the group
        const int src_k = group_lane0 + (i * LPR) / 16;
        float mine = 0.f;
#pragma unroll
        for (int j = 0; j < PER; ++j)
            if (my_base + j == i) mine = part[j];
        const float sk = (PREP ? fk : 1.f) * __shfl_sync(0xffffffffu, mine, src_k);
        const float vi = GDN_INB(head * D + row_in_head + i, v_n, err) ? __bfloat162float(vrow[i]) : 0.f;
        u[i] = b * (vi - alpha * sk);
    }

    // write the updated rows
#pragma unroll
    for (int i = 0; i < kRowsPerGroup; ++i) {
        const float uk = PREP ? u[i] * fk : u[i];
        float4 o;
        o.x = alpha * s[i].x + uk * kv[0];
        o.y = alpha * s[i].y + uk * kv[1];
        o.z = alpha * s[i].z + uk * kv[2];
        o.w = alpha * s[i].w + uk * kv[3];
        if (state_ok) __stcs(srow + (size_t)i * (D / 4), o);
    }

    // outputs: the holder lane of sq_i writes o_i (with 32 lanes per row two
    // lanes hold each sum; the even one writes)
    const bool writer = LPR != 32 || (lane & 1) == 0;
    float ov[PER];
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const int idx = my_base + j;
        ov[j] = 0.f;
        if (idx >= 8 && idx < 16) {
            ov[j] = (PREP ? alpha * fq : alpha) * part[j] + u[idx - 8] * kq;
            if (writer) ss = fmaf(ov[j], ov[j], ss);
        }
    }
    float scale = 1.f;
    if (NORM) {
        __shared__ float warp_ss[NT / 32];
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        float head_ss = ss;   // d = 32: the warp is the head
        if (D >= 64) {        // d = 64, 128: the CTA is the head
            if (lane == 0) warp_ss[warp] = ss;
            __syncthreads();
            head_ss = 0.f;
#pragma unroll
            for (int w = 0; w < NT / 32; ++w) head_ss += warp_ss[w];
        }
        scale = rsqrtf(head_ss * (1.f / D) + norm_eps);
    }
    if (!writer) return;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const int idx = my_base + j;
        if (idx >= 8 && idx < 16) {
            const int i = idx - 8;
            const float o = NORM ? ov[j] * scale * norm_w[row_in_head + i] : ov[j];
            const size_t oi = (size_t)head * D + row_in_head + i;
            if (!GDN_INB(oi, v_n, err)) continue;
            if (out_f32) reinterpret_cast<float *>(out)[oi] = o;
            else reinterpret_cast<__nv_bfloat16 *>(out)[oi] = __float2bfloat16_rn(o);
        }
    }
}

// Short-sequence prefill: the decode step's row streaming applied to every token of a short sequence
// (a speculative verify, a prompt segment of a few tokens).  Each state row is read once, carried through
// the sequence's tokens in registers and written once; the tokens' q, k, v and gates are staged in shared
// memory up front.  One CTA covers kShortRows(D) value rows of one (sequence, head); the per-token math
// is the decode step's:  sk = s.k, sq = s.q, u = beta (v - alpha sk), s' = alpha s + u k, o = alpha sq + u (k.q).
constexpr int kShortMaxTokens = kShortScanTokens;

template <int D>
__host__ __device__ constexpr int short_warps() { return D == 32 ? 1 : 4; }
template <int D>
__host__ __device__ constexpr int short_rows() { return short_warps<D>() * (32 / (D / 4)) * kRowsPerGroup; }   // 32, 64, 32

template <int D, bool NORM>
struct __align__(16) ShortSmem {
    __nv_bfloat16 k[kShortMaxTokens][D];
    __nv_bfloat16 q[kShortMaxTokens][D];
    __nv_bfloat16 v[kShortMaxTokens][short_rows<D>()];
    float alpha[kShortMaxTokens];
    float beta[kShortMaxTokens];
    float kq[kShortMaxTokens];   // prepared k.q
    float fk[kShortMaxTokens];   // preparation factors of k and q
    float fq[kShortMaxTokens];
    float o[NORM ? kShortMaxTokens : 1][short_rows<D>()];   // outputs, held back for the output normalisation
    float ps[NORM ? kShortMaxTokens : 1];   // per-token sum of squares of this CTA's outputs, then the scale
};

template <int D, bool NORM>
__global__ void __launch_bounds__(short_warps<D>() * 32)
short_prefill_kernel(int total_tokens, int hk, int hv, const __nv_bfloat16 *__restrict__ q,
                     const __nv_bfloat16 *__restrict__ k, const __nv_bfloat16 *__restrict__ v,
                     const float *__restrict__ log_alpha, const float *__restrict__ beta,
                     const float *__restrict__ init_state, const int32_t *__restrict__ cu_seqlens,
                     void *__restrict__ out, int out_f32, float *__restrict__ final_state, int qk_norm,
                     float q_scale, const float *__restrict__ norm_w, float norm_eps,
                     const float *__restrict__ gate_c, const float *__restrict__ gate_b, int n_seqs,
                     unsigned int *err) {
    constexpr int LPR = D / 4, GROUPS = 32 / LPR, ROWS = short_rows<D>(), SLICES = D / ROWS;
    constexpr int NT = short_warps<D>() * 32;
    constexpr int PER = (16 / LPR) > 0 ? (16 / LPR) : 1;
    __shared__ ShortSmem<D, NORM> sm;

    const int slice = blockIdx.x % SLICES;
    const int h = (blockIdx.x / SLICES) % hv;
    const int n = blockIdx.x / (SLICES * hv);
    const int hq = h / (hv / hk);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int group = lane / LPR, gl = lane % LPR;
    const int row_in_head = slice * ROWS + (warp * GROUPS + group) * kRowsPerGroup;   // first of 8 rows
    const long tbeg = min(max((long)cu_seqlens[n], 0L), (long)total_tokens);
    const long tend = min(max((long)cu_seqlens[n + 1], tbeg), (long)total_tokens);
    const int L = (int)min(tend - tbeg, (long)kShortMaxTokens);   // the host sends only L <= kShortMaxTokens

    // extents (elements) of the buffers, for the bounds-checking build
    const long qk_n = (long)total_tokens * hk * D, v_n = (long)total_tokens * hv * D, g_n = (long)total_tokens * hv;
    const long state_n = (long)n_seqs * hv * D * D;
    (void)qk_n; (void)v_n; (void)g_n; (void)state_n; (void)n_seqs;

    // stage the tokens: q, k rows of head hq (16-byte pieces), v of this CTA's rows, gates
    for (int i = tid; i < L * (D / 8); i += NT) {
        const int t = i / (D / 8), c = i % (D / 8);
        const size_t g = ((size_t)(tbeg + t) * hk + hq) * D + c * 8;
        const bool ok = GDN_INB(g + 7, qk_n, err);
        *reinterpret_cast<uint4 *>(&sm.k[t][c * 8]) = ok ? *reinterpret_cast<const uint4 *>(k + g) : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4 *>(&sm.q[t][c * 8]) = ok ? *reinterpret_cast<const uint4 *>(q + g) : make_uint4(0, 0, 0, 0);
    }
    for (int i = tid; i < L * (ROWS / 8); i += NT) {
        const int t = i / (ROWS / 8), c = i % (ROWS / 8);
        const size_t g = ((size_t)(tbeg + t) * hv + h) * D + slice * ROWS + c * 8;
        *reinterpret_cast<uint4 *>(&sm.v[t][c * 8]) =
            GDN_INB(g + 7, v_n, err) ? *reinterpret_cast<const uint4 *>(v + g) : make_uint4(0, 0, 0, 0);
    }
    for (int t = tid; t < L; t += NT) {
        const size_t g = (size_t)(tbeg + t) * hv + h;
        const bool ok = GDN_INB(g, g_n, err);
        sm.alpha[t] = __expf(clamp_log_alpha(ok ? gate_log_alpha(log_alpha[g], gate_c, gate_b, h) : 0.f));
        sm.beta[t] = ok ? gate_beta(beta[g], gate_c) : 0.f;
    }

    // this lane group's 8 state rows, 4 columns per lane
    const size_t head = (size_t)n * hv + h;
    float4 s[kRowsPerGroup];
    const bool state_ok = GDN_INB((head * D + row_in_head + kRowsPerGroup - 1) * D + gl * 4 + 3, state_n, err);
    float4 *srow = final_state && state_ok
                       ? reinterpret_cast<float4 *>(final_state + (head * D + row_in_head) * D) + gl
                       : nullptr;
    if (init_state && state_ok) {
        const float4 *irow = reinterpret_cast<const float4 *>(init_state + (head * D + row_in_head) * D) + gl;
#pragma unroll
        for (int i = 0; i < kRowsPerGroup; ++i) s[i] = irow[(size_t)i * (D / 4)];
    } else {
#pragma unroll
        for (int i = 0; i < kRowsPerGroup; ++i) s[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncthreads();
    // k.q and |k|^2, |q|^2 of every token, one lane group per token (all warps run the same number of rounds)
    for (int t0 = 0; t0 < L; t0 += short_warps<D>() * GROUPS) {
        const int t = t0 + warp * GROUPS + group;
        float x = 0.f, kk = 0.f, qq = 0.f;
        if (t < L) {
            const uint2 kr = *reinterpret_cast<const uint2 *>(&sm.k[t][gl * 4]);
            const uint2 qr = *reinterpret_cast<const uint2 *>(&sm.q[t][gl * 4]);
            const float k4[4] = {bf16_lo(kr.x), bf16_hi(kr.x), bf16_lo(kr.y), bf16_hi(kr.y)};
            const float q4[4] = {bf16_lo(qr.x), bf16_hi(qr.x), bf16_lo(qr.y), bf16_hi(qr.y)};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                x = fmaf(k4[e], q4[e], x);
                kk = fmaf(k4[e], k4[e], kk);
                qq = fmaf(q4[e], q4[e], qq);
            }
        }
#pragma unroll
        for (int off = LPR / 2; off >= 1; off >>= 1) {
            x += __shfl_xor_sync(0xffffffffu, x, off);
            kk += __shfl_xor_sync(0xffffffffu, kk, off);
            qq += __shfl_xor_sync(0xffffffffu, qq, off);
        }
        if (gl == 0 && t < L) {
            const float fk = qk_inv_norm(kk, qk_norm), fq = q_scale * qk_inv_norm(qq, qk_norm);
            sm.fk[t] = fk;
            sm.fq[t] = fq;
            sm.kq[t] = x * fk * fq;
        }
    }
    __syncthreads();

    const int my_base = gl * 16 / LPR;
    const int group_lane0 = group * LPR;
    const int vrow0 = (warp * GROUPS + group) * kRowsPerGroup;   // within the CTA's rows
    for (int t = 0; t < L; ++t) {
        const uint2 kr = *reinterpret_cast<const uint2 *>(&sm.k[t][gl * 4]);
        const uint2 qr = *reinterpret_cast<const uint2 *>(&sm.q[t][gl * 4]);
        const float kv[4] = {bf16_lo(kr.x), bf16_hi(kr.x), bf16_lo(kr.y), bf16_hi(kr.y)};
        const float qv[4] = {bf16_lo(qr.x), bf16_hi(qr.x), bf16_lo(qr.y), bf16_hi(qr.y)};
        const float alpha = sm.alpha[t], b = sm.beta[t], kq = sm.kq[t], fk = sm.fk[t], fq = sm.fq[t];
        float part[16];
#pragma unroll
        for (int i = 0; i < kRowsPerGroup; ++i) {
            part[i] = s[i].x * kv[0] + s[i].y * kv[1] + s[i].z * kv[2] + s[i].w * kv[3];
            part[8 + i] = s[i].x * qv[0] + s[i].y * qv[1] + s[i].z * qv[2] + s[i].w * qv[3];
        }
        reduce16<LPR>(part, lane);
        float u[kRowsPerGroup];
#pragma unroll
        for (int i = 0; i < kRowsPerGroup; ++i) {
            const int src_k = group_lane0 + (i * LPR) / 16;
            float mine = 0.f;
#pragma unroll
            for (int j = 0; j < PER; ++j)
                if (my_base + j == i) mine = part[j];
            const float sk = fk * __shfl_sync(0xffffffffu, mine, src_k);
            u[i] = b * (__bfloat162float(sm.v[t][vrow0 + i]) - alpha * sk);
        }
#pragma unroll
        for (int i = 0; i < kRowsPerGroup; ++i) {
            const float uk = u[i] * fk;
            s[i].x = alpha * s[i].x + uk * kv[0];
            s[i].y = alpha * s[i].y + uk * kv[1];
            s[i].z = alpha * s[i].z + uk * kv[2];
            s[i].w = alpha * s[i].w + uk * kv[3];
        }
        // the holder lane of sq_i writes o_i (with 32 lanes per row two lanes hold each sum: the even one)
        if (LPR != 32 || (lane & 1) == 0) {
#pragma unroll
            for (int j = 0; j < PER; ++j) {
                const int idx = my_base + j;
                if (idx >= 8 && idx < 16) {
                    const int i = idx - 8;
                    const float o = alpha * fq * part[j] + u[i] * kq;
                    const size_t oi = ((size_t)(tbeg + t) * hv + h) * D + row_in_head + i;
                    if (NORM) sm.o[t][vrow0 + i] = o;
                    else if (!GDN_INB(oi, v_n, err)) continue;
                    else if (out_f32) reinterpret_cast<float *>(out)[oi] = o;
                    else reinterpret_cast<__nv_bfloat16 *>(out)[oi] = __float2bfloat16_rn(o);
                }
            }
        }
    }
    if (srow) {
#pragma unroll
        for (int i = 0; i < kRowsPerGroup; ++i) srow[(size_t)i * (D / 4)] = s[i];
    }
    if (NORM) {
        // Output normalisation over the head's d rows: per token, the sum of squares of this CTA's rows; with
        // d = 128 the head's four CTAs form a cluster and add theirs through distributed shared memory.
        __syncthreads();
        for (int t = tid; t < L; t += NT) {
            float x = 0.f;
            for (int j = 0; j < ROWS; ++j) x = fmaf(sm.o[t][j], sm.o[t][j], x);
            sm.ps[t] = x;
        }
        float scale_t[(kShortMaxTokens + NT - 1) / NT];
        if (SLICES > 1) {
            cluster_sync();
#pragma unroll
            for (int m = 0; m < (kShortMaxTokens + NT - 1) / NT; ++m) {
                const int t = tid + m * NT;
                float x = 0.f;
                if (t < L)
                    for (int rk = 0; rk < SLICES; ++rk) x += ld_dsmem_f32(&sm.ps[t], rk);
                scale_t[m] = x;
            }
            cluster_sync();   // every peer has read this CTA's sums
        } else {
            __syncthreads();
#pragma unroll
            for (int m = 0; m < (kShortMaxTokens + NT - 1) / NT; ++m) {
                const int t = tid + m * NT;
                scale_t[m] = t < L ? sm.ps[t] : 0.f;
            }
        }
        __syncthreads();
#pragma unroll
        for (int m = 0; m < (kShortMaxTokens + NT - 1) / NT; ++m) {
            const int t = tid + m * NT;
            if (t < L) sm.ps[t] = rsqrtf(scale_t[m] * (1.f / D) + norm_eps);
        }
        __syncthreads();
        for (int i = tid; i < L * ROWS; i += NT) {
            const int t = i / ROWS, j = i % ROWS;
            const float o = sm.o[t][j] * sm.ps[t] * norm_w[slice * ROWS + j];
            const size_t oi = ((size_t)(tbeg + t) * hv + h) * D + slice * ROWS + j;
            if (!GDN_INB(oi, v_n, err)) continue;
            if (out_f32) reinterpret_cast<float *>(out)[oi] = o;
            else reinterpret_cast<__nv_bfloat16 *>(out)[oi] = __float2bfloat16_rn(o);
        }
    }
}

template <int D, bool NORM>
cudaError_t launch_short_dn(const PrefillProblem &p) {
    constexpr int SLICES = D / short_rows<D>();   // CTAs per head; a cluster when the output is normalised
    const unsigned grid = (unsigned)(p.n_seqs * p.hv * SLICES);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = SLICES;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(short_warps<D>() * 32);
    cfg.stream = p.stream;
    cfg.attrs = attr;
    cfg.numAttrs = (NORM && SLICES > 1) ? 1 : 0;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, short_prefill_kernel<D, NORM>, p.total_tokens, p.hk, p.hv, p.q, p.k, p.v,
                                             p.log_alpha, p.beta, p.init_state, p.cu_seqlens, p.out, p.out_f32,
                                             p.final_state, p.qk_norm, p.q_scale, p.norm_w, p.norm_eps, p.gate_c,
                                             p.gate_b, p.n_seqs, p.err);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <int D>
cudaError_t launch_short_d(const PrefillProblem &p) {
    return p.norm_w ? launch_short_dn<D, true>(p) : launch_short_dn<D, false>(p);
}

}  // namespace

cudaError_t launch_short_prefill(const PrefillProblem &p) {
    if (p.n_seqs == 0) return cudaSuccess;
    switch (p.d) {
        case 32: return launch_short_d<32>(p);
        case 64: return launch_short_d<64>(p);
        case 128: return launch_short_d<128>(p);
        default: return cudaErrorInvalidValue;
    }
}

namespace {

template <int D, bool PREP, bool NORM, bool GATE>
cudaError_t launch_decode_dg(const DecodeProblem &p) {
    constexpr int NT = decode_threads<D, NORM>();
    constexpr long rows_per_block = (long)(NT / 32) * (32 / (D / 4)) * kRowsPerGroup;
    const long total_rows = (long)p.n * p.hv * p.d;
    // with the output normalisation a CTA holds whole heads (d >= 64) or whole warps do (d = 32): no CTA may
    // end early, so the rows must fill the grid exactly (always true: rows_per_block divides hv * d)
    if (NORM && D >= 64 && total_rows % rows_per_block) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((total_rows + rows_per_block - 1) / rows_per_block));
    cfg.blockDim = dim3(NT);
    cfg.stream = p.stream;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, decode_step_kernel<D, PREP, NORM, GATE>, (int)((long)p.n * p.hv * p.d), p.hk,
                                             p.hv, p.state, p.q, p.k, p.v, p.log_alpha, p.beta, p.out, p.out_f32,
                                             p.qk_norm, p.q_scale, p.norm_w, p.norm_eps, p.gate_c, p.gate_b, p.err);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <int D, bool PREP, bool NORM>
cudaError_t launch_decode_d(const DecodeProblem &p) {
    return p.gate_c ? launch_decode_dg<D, PREP, NORM, true>(p) : launch_decode_dg<D, PREP, NORM, false>(p);
}

template <int D, bool PREP>
cudaError_t launch_decode_prep(const DecodeProblem &p) {
    return p.norm_w ? launch_decode_d<D, PREP, true>(p) : launch_decode_d<D, PREP, false>(p);
}

template <int D>
cudaError_t launch_decode_norm(const DecodeProblem &p) {
    return (p.qk_norm || p.q_scale != 1.f) ? launch_decode_prep<D, true>(p) : launch_decode_prep<D, false>(p);
}

}  // namespace

cudaError_t launch_decode(const DecodeProblem &p) {
    if ((long)p.n * p.hv * p.d == 0) return cudaSuccess;
    switch (p.d) {
        case 32: return launch_decode_norm<32>(p);
        case 64: return launch_decode_norm<64>(p);
        case 128: return launch_decode_norm<128>(p);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gdn
