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
// sequential over chunks, in `state_pass_kernel` (which, when the output
// normalisation is fused, runs as clusters of the four slice CTAs of a head
// that exchange the per-token sums of squares).
//
// Tensor-core use (tcgen05.mma, bf16 operands, fp32 accumulation in TMEM,
// operands staged by TMA in 128B-swizzled shared memory):
//   prep:  [K;Q] K^T (exact: q/k are bf16), P = K^T (Gamma T) and R = Aqk T with
//          Gamma T, T and Aqk split into bf16 hi + lo parts; P and R are stored
//          as bf16 hi + lo pairs
//   pass:  [Q;K] [S_hi;S_lo]^T, (P_hi + P_lo) [X_hi;X_lo]^T, (R_hi + R_lo) [X_hi;X_lo]^T
// Everything that feeds the carried state is either an exact bf16 input or a
// value split into two bf16 terms (about 16 significant bits), so the state
// error stays far below the fp32-state tolerance; the output-only terms use
// one bf16 pass.  The triangular solve runs in fp32 on the CUDA cores.
#include <cudaTypedefs.h>

#include <algorithm>
#include <vector>

#include "gdn_internal.cuh"
#include "sm100.cuh"

namespace gdn {
namespace {

using namespace sm100;

constexpr int D = 128;          // head size of the chunked path
constexpr int C = kChunk;       // 64 tokens per chunk
constexpr int DS = 32;          // value rows per state-passing CTA
constexpr uint32_t kSW = kLayoutSwizzle128B;

constexpr size_t kPTile = (size_t)D * C * 2;     // P_hi or P_lo of one (chunk, head): 16 KiB
constexpr size_t kRTile = (size_t)C * C * 2;     // R of one (chunk, head): 8 KiB
constexpr size_t kNormBytes = 2 * C * 4;         // q/k preparation factors of one (chunk, head): f_k [64], f_q [64]

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

// A position in the chunks of a run of consecutive sequences: sequence n (tokens [ta, tb), nk chunks), its
// chunk k.  Past the run, n = end and the chunk is empty.
struct ChunkCursor {
    int n, ta, tb, k, nk;
    __device__ __forceinline__ int t0() const { return ta + k * C; }
    __device__ __forceinline__ int len() const { return min(C, tb - ta - k * C); }
    __device__ __forceinline__ bool last_of_seq() const { return k == nk - 1; }
};

__device__ __forceinline__ void cursor_at_seq(ChunkCursor &cc, const int32_t *cu, int n_seqs, int total, int n) {
    cc.n = n;
    cc.k = 0;
    if (n_seqs == 1) {   // the host checked cu_seqlens = {0, total}
        cc.ta = 0;
        cc.tb = total;
    } else {
        seq_range(cu, n, total, cc.ta, cc.tb);
    }
    cc.nk = (cc.tb - cc.ta + C - 1) / C;
}

// The first chunk of the first sequence in [m, end) that has tokens; on_empty(m') is called for every sequence
// without tokens passed over.
template <typename F>
__device__ __forceinline__ void cursor_seek(ChunkCursor &cc, const int32_t *cu, int n_seqs, int total, int m,
                                            int end, F on_empty) {
    for (; m < end; ++m) {
        cursor_at_seq(cc, cu, n_seqs, total, m);
        if (cc.nk > 0) return;
        on_empty(m);
    }
    cc.n = end;
    cc.k = cc.nk = 0;
    cc.ta = cc.tb = total;
}

// The next chunk of the run: the next one of this sequence, else the first of the next sequence with tokens.
template <typename F>
__device__ __forceinline__ void cursor_next(ChunkCursor &cc, const int32_t *cu, int n_seqs, int total, int end,
                                            F on_empty) {
    if (++cc.k < cc.nk) return;
    cursor_seek(cc, cu, n_seqs, total, cc.n + 1, end, on_empty);
}

// Sequence buckets of the plain state pass: CTA (bucket b, head, row slice) carries the state through the
// sequences [seq[b], seq[b+1]) one after another, which are the global chunks [chunk[b], chunk[b+1])
// (sequences are packed, and their chunks numbered, in order).  The host balances the buckets by chunks.
// With per_seq, bucket b is sequence b and its first chunk is found from cu_seqlens (any number of sequences).
constexpr int kMaxPassBuckets = 64;
struct PassBuckets {
    int per_seq;
    int seq[kMaxPassBuckets + 1];
    int chunk[kMaxPassBuckets + 1];
};

// The next 1 KiB boundary of a dynamic shared-memory pointer.  Pointer arithmetic (no integer round trip)
// keeps the shared address space visible to the compiler, so accesses through the result compile to
// shared-memory instructions instead of generic ones.
__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
    return p + ((1024u - (smem_u32(p) & 1023u)) & 1023u);
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(a));
    const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(b));
    return lo | (hi << 16);
}

// Split 8 floats into bf16 hi and lo parts packed as two 16-byte vectors (x = hi + lo to ~16 bits).  hi is
// x with its low 16 bits dropped (a byte permute, no conversion); x - hi is then exact in fp32 and only lo
// is rounded to bf16, which bounds the split's relative error by 2^-17.
__device__ __forceinline__ void split8_bf16(const float *x, uint4 &hi, uint4 &lo) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const uint32_t a = __float_as_uint(x[2 * e]), b = __float_as_uint(x[2 * e + 1]);
        h[e] = __byte_perm(a, b, 0x7632);
        const __nv_bfloat162 ll = __floats2bfloat162_rn(x[2 * e] - __uint_as_float(a & 0xffff0000u),
                                                        x[2 * e + 1] - __uint_as_float(b & 0xffff0000u));
        l[e] = *reinterpret_cast<const uint32_t *>(&ll);
    }
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
}


// Inclusive cumulative log-decay of a chunk for this warp: lane l holds the raw log_alpha of tokens 2l
// and 2l+1 (anything for tokens at or beyond `len`, which contribute 0, so their g equals g_{len-1}).
// log_alpha is clamped to [-20, 0].  Returns the two g values of the lane.
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

// g_i of token i from the per-lane pairs produced by cumsum_pairs.
__device__ __forceinline__ float g_of(float2 g2, int i) {
    const float a = __shfl_sync(0xffffffffu, g2.x, i >> 1);
    const float b = __shfl_sync(0xffffffffu, g2.y, i >> 1);
    return (i & 1) ? b : a;
}


// ============================================================================
// Kernel 1: per-chunk preparation (parallel over chunks x value heads)
// ============================================================================
// Shared memory (offsets from a 1 KiB-aligned base):
constexpr uint32_t PREP_KQ = 0;        // kb0: K rows | Q rows, kb1: K rows | Q rows (32 KiB).  Once [K;Q]K^T
                                       // is done the Q halves hold T (fp32), then the T^T hi / lo tiles.
constexpr uint32_t PREP_A = 32768;     // fp32 A [64][68]; later (Gamma T)^T hi / lo, then R hi / lo
constexpr int A_LD = 68;
constexpr uint32_t PREP_AQK = PREP_A + 64 * A_LD * 4;   // 50176: Aqk hi, Aqk lo tiles [64 x 64] bf16
constexpr uint32_t PREP_Y = PREP_AQK + 16384;           // fp32 scratch [4][16][16]
constexpr uint32_t PREP_G = PREP_Y + 4 * 256 * 4;       // g [64], beta [64], Gamma = e^{g_L - g} [64],
                                                        // the q/k preparation factors f_k [64], f_q [64],
                                                        // then alpha = e^{log_alpha} [64]
constexpr uint32_t PREP_SMEM = PREP_G + 1536 + 1024;    // + alignment slack: 3 CTAs per SM
constexpr uint32_t PREP_TMEM_COLS = 128;

// Row ii of T (fp32, 64 columns): rows 0-31 over the Q half of k-block 0, rows 32-63 over that of k-block 1.
__device__ __forceinline__ float *t_row(uint8_t *sm, int ii) {
    return reinterpret_cast<float *>(sm + PREP_KQ + (ii < 32 ? 8192 : 24576)) + (ii & 31) * 64;
}

constexpr int kPrepThreads = 256;   // 8 warps: warps w and w + 4 share TMEM lane quadrant w % 4

// T = (I + A)^-1 for the strictly lower fp32 A (row stride A_LD), by 16 x 16 blocks, kPrepThreads threads:
//   diagonal blocks  T_II = (I + A_II)^-1      forward substitution by threads 0-127, two per column: the
//                                              first takes rows 0-7 of its block, the second rows 8-15
//                                              once those are in shared memory (rows of A read as 16-byte
//                                              words)
//   below them       by recursive doubling on block pairs: T_10 and T_32 together, then the lower-left
//                                              32 x 32 block from the two 32 x 32 diagonal halves (four
//                                              barriers; level by level in the block row it took six, and
//                                              the preparation 60.6 against 57.8 us at the 4K layer)
// In the block products each thread owns a strip of two adjacent columns of one row: four consecutive
// elements of the left factor come in one 16-byte load (the same address for the lanes of a row) and each
// row of the right factor in one 8-byte load, so a pair of FMAs costs about one shared-memory load.
// T must be zero on entry.  Ends with the block synchronised.
__device__ __forceinline__ void solve_unit_lower_blocked(const float *__restrict__ A, uint8_t *sm,
                                                         float *__restrict__ Y, int tid) {
    {
        const int j = tid & 63, second = (tid >> 6) & 1, b = j >> 4, jj = j & 15;
        const float *Ab = A + (16 * b) * A_LD + 16 * b;
        float tc[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) tc[r] = (8 * second + r == jj) ? 1.f : 0.f;
        if (tid < 64) {   // rows 0-7, left-looking; each row's A entries come as 16-byte loads
#pragma unroll
            for (int r = 1; r < 8; ++r) {
                float acc = tc[r];
#pragma unroll
                for (int k4 = 0; k4 < r; k4 += 4) {
                    const float4 a4 = *reinterpret_cast<const float4 *>(Ab + r * A_LD + k4);
                    const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (k4 + e < r) acc = fmaf(-av[e], tc[k4 + e], acc);
                }
                tc[r] = acc;
            }
#pragma unroll
            for (int r = 0; r < 8; ++r) t_row(sm, 16 * b + r)[j] = tc[r];
        }
        __syncthreads();
        if (tid >= 64 && tid < 128) {   // rows 8-15: the terms of rows 0-7, then left-looking among themselves
            float top[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) top[r] = t_row(sm, 16 * b + r)[j];
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const float *arow = Ab + (8 + r) * A_LD;
                const float4 a0 = *reinterpret_cast<const float4 *>(arow);
                const float4 a1 = *reinterpret_cast<const float4 *>(arow + 4);
                float acc0 = tc[r], acc1 = 0.f;
                acc0 = fmaf(-a0.x, top[0], acc0);
                acc1 = fmaf(-a0.y, top[1], acc1);
                acc0 = fmaf(-a0.z, top[2], acc0);
                acc1 = fmaf(-a0.w, top[3], acc1);
                acc0 = fmaf(-a1.x, top[4], acc0);
                acc1 = fmaf(-a1.y, top[5], acc1);
                acc0 = fmaf(-a1.z, top[6], acc0);
                acc1 = fmaf(-a1.w, top[7], acc1);
#pragma unroll
                for (int k4 = 0; k4 < r; k4 += 4) {
                    const float4 a4 = *reinterpret_cast<const float4 *>(arow + 8 + k4);
                    const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (k4 + e < r) acc0 = fmaf(-av[e], tc[k4 + e], acc0);
                }
                tc[r] = acc0 + acc1;
            }
#pragma unroll
            for (int r = 0; r < 8; ++r) t_row(sm, 16 * b + 8 + r)[j] = tc[r];
        }
    }
    __syncthreads();
    // Below the diagonal blocks, by recursive doubling on block pairs (16 block products, four barriers):
    //   level 1  T_10 = -T_11 (A_10 T_00)  and  T_32 = -T_33 (A_32 T_22)
    //   level 2  the lower-left 32 x 32 block  T_lh = -T_h (A_hl T_l),  T_l = [T_00 0; T_10 T_11], T_h = [T_22 0; T_32 T_33]
    // Threads 0-127 and 128-255 (par) take balanced halves of each step; in a block product each thread owns a
    // strip of two adjacent columns of one row (the same loads as the level-by-level form).
    const int par = tid >> 7, r = (tid >> 3) & 15, c = (tid & 7) * 2;
    // y += (row r of the 16-block of `left` at rows 16 I, columns 16 K) x (16-block of T at rows 16 K, columns 16 J)
    auto acc_AT = [&](int I, int K, int J, float &y0, float &y1) {
        const float *arow = A + (16 * I + r) * A_LD + 16 * K;
        const float *tb = t_row(sm, 16 * K) + 16 * J + c;
        float z0 = 0.f, z1 = 0.f;
#pragma unroll
        for (int k4 = 0; k4 < 16; k4 += 4) {
            const float4 a4 = *reinterpret_cast<const float4 *>(arow + k4);
            const float2 t0 = *reinterpret_cast<const float2 *>(tb + (k4 + 0) * 64);
            const float2 t1 = *reinterpret_cast<const float2 *>(tb + (k4 + 1) * 64);
            const float2 t2 = *reinterpret_cast<const float2 *>(tb + (k4 + 2) * 64);
            const float2 t3 = *reinterpret_cast<const float2 *>(tb + (k4 + 3) * 64);
            y0 = fmaf(a4.x, t0.x, y0);
            y1 = fmaf(a4.x, t0.y, y1);
            z0 = fmaf(a4.y, t1.x, z0);
            z1 = fmaf(a4.y, t1.y, z1);
            y0 = fmaf(a4.z, t2.x, y0);
            y1 = fmaf(a4.z, t2.y, y1);
            z0 = fmaf(a4.w, t3.x, z0);
            z1 = fmaf(a4.w, t3.y, z1);
        }
        y0 += z0;
        y1 += z1;
    };
    // y += (row r of the 16-block of T at rows 16 I, columns 16 K) x (Y block yb)
    auto acc_TY = [&](int I, int K, const float *yb, float &y0, float &y1) {
        const float *trow = t_row(sm, 16 * I + r) + 16 * K;
        float z0 = 0.f, z1 = 0.f;
#pragma unroll
        for (int k4 = 0; k4 < 16; k4 += 4) {
            const float4 a4 = *reinterpret_cast<const float4 *>(trow + k4);
            const float2 t0 = *reinterpret_cast<const float2 *>(yb + (k4 + 0) * 16 + c);
            const float2 t1 = *reinterpret_cast<const float2 *>(yb + (k4 + 1) * 16 + c);
            const float2 t2 = *reinterpret_cast<const float2 *>(yb + (k4 + 2) * 16 + c);
            const float2 t3 = *reinterpret_cast<const float2 *>(yb + (k4 + 3) * 16 + c);
            y0 = fmaf(a4.x, t0.x, y0);
            y1 = fmaf(a4.x, t0.y, y1);
            z0 = fmaf(a4.y, t1.x, z0);
            z1 = fmaf(a4.y, t1.y, z1);
            y0 = fmaf(a4.z, t2.x, y0);
            y1 = fmaf(a4.z, t2.y, y1);
            z0 = fmaf(a4.w, t3.x, z0);
            z1 = fmaf(a4.w, t3.y, z1);
        }
        y0 += z0;
        y1 += z1;
    };
    auto put = [&](float *dst, float y0, float y1) { *reinterpret_cast<float2 *>(dst) = make_float2(y0, y1); };
    {   // level 1: par 0 the pair (0, 1), par 1 the pair (2, 3)
        const int lo = 2 * par;
        float y0 = 0.f, y1 = 0.f;
        acc_AT(lo + 1, lo, lo, y0, y1);                      // Y = A_{lo+1,lo} T_{lo,lo}
        put(Y + par * 256 + r * 16 + c, y0, y1);
        __syncthreads();
        float t0 = 0.f, t1 = 0.f;
        acc_TY(lo + 1, lo + 1, Y + par * 256, t0, t1);       // T_{lo+1,lo} = -T_{lo+1,lo+1} Y
        put(t_row(sm, 16 * (lo + 1) + r) + 16 * lo + c, -t0, -t1);
        __syncthreads();
    }
    {   // level 2: Y_ab = sum_k A_ak (T_l)_kb for a in {2, 3}, b in {0, 1}; par 0 rows a = 2, par 1 a = 3
        const int a = 2 + par;
        float y0 = 0.f, y1 = 0.f, w0 = 0.f, w1 = 0.f;
        acc_AT(a, 0, 0, y0, y1);                             // Y_a0 = A_a0 T_00 + A_a1 T_10
        acc_AT(a, 1, 0, y0, y1);
        acc_AT(a, 1, 1, w0, w1);                             // Y_a1 = A_a1 T_11
        put(Y + (2 * par) * 256 + r * 16 + c, y0, y1);
        put(Y + (2 * par + 1) * 256 + r * 16 + c, w0, w1);
        __syncthreads();
        // T_2b = -T_22 Y_2b, T_3b = -(T_32 Y_2b + T_33 Y_3b); par 0 columns b = 0, par 1 b = 1
        const int b = par;
        float u0 = 0.f, u1 = 0.f, v0 = 0.f, v1 = 0.f;
        acc_TY(2, 2, Y + (0 + b) * 256, u0, u1);
        acc_TY(3, 2, Y + (0 + b) * 256, v0, v1);
        acc_TY(3, 3, Y + (2 + b) * 256, v0, v1);
        put(t_row(sm, 32 + r) + 16 * b + c, -u0, -u1);
        put(t_row(sm, 48 + r) + 16 * b + c, -v0, -v1);
        __syncthreads();
    }
}

// PREP: query/key preparation (qk_norm, or q_scale != 1); the plain instantiation has none of its arithmetic.
// GATE: the gates are formed from raw inputs (gdn.h: gate_scale, gate_bias).
template <bool PREP, bool GATE>
__global__ void __launch_bounds__(kPrepThreads, 3)
chunk_prep_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                  const __grid_constant__ CUtensorMap phmap, const __grid_constant__ CUtensorMap plmap,
                  const __grid_constant__ CUtensorMap rhmap, const __grid_constant__ CUtensorMap rlmap,
                  const float *__restrict__ log_alpha, const float *__restrict__ beta,
                  const int32_t *__restrict__ cu, int n_seqs, int total, int hk, int hv, float *__restrict__ norms,
                  int qk_norm, float q_scale, const float *__restrict__ gate_c, const float *__restrict__ gate_b,
                  unsigned int *err) {
    extern __shared__ uint8_t prep_raw[];
    uint8_t *sm = align1024(prep_raw);
    __shared__ uint64_t bar_tma, bar_mma;
    __shared__ uint32_t tmem_slot;

    // chunk-major, last chunk first: the state pass reads the first chunks first, so they are the ones written
    // last, the most likely to be still in L2 when it starts
    const int nch = (int)(gridDim.x / hv);
    const int h = (int)(blockIdx.x % hv);
    const int gc = nch - 1 - (int)(blockIdx.x / hv);
    const int hq = h / (hv / hk);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, half = warp >> 2;   // TMEM lane quadrant; which column half the warp takes
    ChunkLoc loc;
    if (n_seqs == 1) {   // one sequence (the host checked cu_seqlens = {0, total}): chunk gc starts at 64 gc
        if (gc * C >= total) return;
        loc.seq = 0;
        loc.t0 = gc * C;
        loc.len = min(C, total - loc.t0);
    } else if (!locate_chunk(cu, n_seqs, total, gc, loc)) {
        return;   // uniform for the CTA
    }
    const int t0 = loc.t0, L = loc.len;
    const uint32_t base = smem_u32(sm);
    const uint32_t tlane = (uint32_t)(32 * quad) << 16;
    // the state pass may start its prologue (and its first chunk's products, which need no workspace) on SMs
    // this grid has left; it waits for this grid before reading the workspace
    if (tid == 0) grid_launch_dependents();

    // Thread 0 requests the tiles first (their latency is the longest); warp 2 allocates TMEM meanwhile.
    if (tid == 0) {
        mbar_init(&bar_tma, 1);
        mbar_init(&bar_mma, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(&bar_tma, 32768);
        // (bounds-checking build: the tile's columns inside the q/k rows, its first token inside the tokens)
        if (GDN_INB(hq * D + 127, hk * D, err) && GDN_INB(t0, total, err)) {
#pragma unroll
            for (int kb = 0; kb < 2; ++kb) {
                tma_load_2d(sm + PREP_KQ + kb * 16384, &kmap, &bar_tma, hq * D + kb * 64, t0);
                tma_load_2d(sm + PREP_KQ + kb * 16384 + 8192, &qmap, &bar_tma, hq * D + kb * 64, t0);
            }
        }
    }
    if (warp == 2) {
        tmem_alloc(&tmem_slot, PREP_TMEM_COLS);
        tmem_relinquish();
    }
    float *g_s = reinterpret_cast<float *>(sm + PREP_G);  // [64]
    float *b_s = g_s + 64;                                // [64]
    float *gam_s = g_s + 128;                             // [64], 0 past the chunk's end
    float *kf_s = g_s + 192, *qf_s = g_s + 256;           // [64] each: f_k = 1/|k| (or 1), f_q = q_scale/|q| (or q_scale)
    float *al_s = g_s + 320;                              // [64] per-token decay e^{log_alpha} (1 past the chunk's end)
    // warp 1 loads this chunk's gates now; their cumulative sum is formed while the TMA and MMA run
    float la0 = 0.f, la1 = 0.f, bt0 = 0.f, bt1 = 0.f;
    if (warp == 1) {
        const int i0 = 2 * lane, i1 = 2 * lane + 1;
        if (i0 < L && GDN_INB((size_t)(t0 + i0) * hv + h, (long)total * hv, err)) {
            la0 = log_alpha[(size_t)(t0 + i0) * hv + h];
            bt0 = beta[(size_t)(t0 + i0) * hv + h];
        }
        if (i1 < L && GDN_INB((size_t)(t0 + i1) * hv + h, (long)total * hv, err)) {
            la1 = log_alpha[(size_t)(t0 + i1) * hv + h];
            bt1 = beta[(size_t)(t0 + i1) * hv + h];
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    // shared-memory descriptors of every MMA operand (uniform values, built outside divergent code)
    const uint64_t dkq = smem_desc(base + PREP_KQ, 16, 1024, kSW);          // [K;Q] K-major
    const uint64_t dk_mn = smem_desc(base + PREP_KQ, 16384, 1024, kSW);     // K read MN-major
    const uint64_t dgth = smem_desc(base + PREP_A, 16, 1024, kSW);          // (Gamma T)^T hi
    const uint64_t dgtl = smem_desc(base + PREP_A + 8192, 16, 1024, kSW);   //                lo
    const uint64_t dah = smem_desc(base + PREP_AQK, 16, 1024, kSW);         // Aqk hi
    const uint64_t dal = smem_desc(base + PREP_AQK + 8192, 16, 1024, kSW);  //     lo
    const uint64_t dth = smem_desc(base + PREP_KQ + 8192, 16, 1024, kSW);   // T^T hi
    const uint64_t dtl = smem_desc(base + PREP_KQ + 24576, 16, 1024, kSW);  //     lo

    bool ok = mbar_wait(&bar_tma, 0);
    ok = __syncthreads_and(ok);
    if (ok && tid == 0) {
        // D0[128 x 64] = [K ; Q] K^T  (rows 0-63: K K^T, rows 64-127: Q K^T), exact products
        constexpr uint32_t idesc = idesc_bf16_f32(128, 64, false, false);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const uint64_t off = (uint64_t)(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
            mma_bf16(tmem, dkq + off, dkq + off, idesc, kk > 0);
        }
        mma_commit(&bar_mma);
    }
    if (PREP && tid < 128) {   // Query/key preparation factors of the 64 k rows (threads 0-63) and 64 q rows (64-127), from the staged
        // tiles (which the MMA above only reads).  The products use raw q and k; the factors scale rows and
        // columns of [K;Q]K^T and the rows of P = K^T diag(f_k) Gamma T.  The state pass reads them from the
        // workspace.
        const int r = tid & 63;
        const bool isq = tid >= 64;
        float f = isq ? q_scale : 1.f;
        if (qk_norm) {
            float ss = 0.f;
#pragma unroll
            for (int kb = 0; kb < 2; ++kb) {
#pragma unroll
                for (int c = 0; c < 64; c += 8) {
                    const uint4 x =
                        *reinterpret_cast<const uint4 *>(sm + PREP_KQ + kb * 16384 + (isq ? 8192 : 0) + sw128_offset(r, c));
                    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        ss = fmaf(bf16_lo(w[e]), bf16_lo(w[e]), ss);
                        ss = fmaf(bf16_hi(w[e]), bf16_hi(w[e]), ss);
                    }
                }
            }
            f *= qk_inv_norm(ss, 1);
        }
        (isq ? qf_s : kf_s)[r] = f;
        if (ok && qk_norm && GDN_INB(((size_t)gc * hv + h) * 128 + tid, (long)nch * hv * 128, err))
            norms[((size_t)gc * hv + h) * 128 + tid] = f;   // read by the pass only with qk_norm
    }
    if (warp == 1) {
        if (GATE) {   // the gates from raw inputs, formed while the loads' latency was covered by the MMA wait
            if (2 * lane < L) {
                la0 = gate_log_alpha(la0, gate_c, gate_b, h);
                bt0 = gate_beta(bt0, gate_c);
            }
            if (2 * lane + 1 < L) {
                la1 = gate_log_alpha(la1, gate_c, gate_b, h);
                bt1 = gate_beta(bt1, gate_c);
            }
        }
        const float2 g2 = cumsum_pairs(la0, la1, L, lane);
        const float gl = g_of(g2, L - 1);
        g_s[2 * lane] = g2.x;
        g_s[2 * lane + 1] = g2.y;
        b_s[2 * lane] = bt0;
        b_s[2 * lane + 1] = bt1;
        gam_s[2 * lane] = 2 * lane < L ? __expf(gl - g2.x) : 0.f;
        gam_s[2 * lane + 1] = 2 * lane + 1 < L ? __expf(gl - g2.y) : 0.f;
        al_s[2 * lane] = 2 * lane < L ? __expf(fminf(clamp_log_alpha(la0), 0.f)) : 1.f;
        al_s[2 * lane + 1] = 2 * lane + 1 < L ? __expf(fminf(clamp_log_alpha(la1), 0.f)) : 1.f;
    }
    if (ok) ok = mbar_wait(&bar_mma, 0);
    ok = __syncthreads_and(ok);
    tc_fence_after();
    if (PREP && qk_norm && tid < 64) gam_s[tid] *= kf_s[tid];   // P = K^T diag(f_k Gamma) T (read after the solve's barriers)
    {   // T (over the Q rows, which [K;Q]K^T no longer needs) starts at zero; its upper blocks stay zero
        float4 *t0q = reinterpret_cast<float4 *>(sm + PREP_KQ + 8192);
        float4 *t1q = reinterpret_cast<float4 *>(sm + PREP_KQ + 24576);
        for (int x = tid; x < 512; x += kPrepThreads) {
            t0q[x] = make_float4(0.f, 0.f, 0.f, 0.f);
            t1q[x] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }

    // Quadrants 0-1 build A (fp32) from the K K^T rows, quadrants 2-3 the Aqk tiles (split into bf16 hi/lo)
    // from the Q K^T rows; the two warps of a quadrant split the columns.  Then all warps solve for T and
    // write the T operand tiles.  Rows 0-31 have nothing left of the diagonal past column 31: their warps
    // take 16 columns each of 0-31, those of rows 32-63 32 columns each.  The solve never reads A on or
    // above the diagonal, so A is written only below it (rows past the chunk's end get zeros through their
    // row factor); the Aqk tiles feed an MMA and are written in full (zeros above the diagonal).
    {
        const int i = 32 * (quad & 1) + lane;
        const bool low_rows = (quad & 1) == 0;    // rows 0-31 (warp-uniform)
        const int c0 = low_rows ? 16 * half : 32 * half, ncol = low_rows ? 16 : 32;
        float vals[32];
        {
            float a16[16], b16[16];
            if (low_rows) {
                tmem_ld16(tmem + tlane + c0, a16);
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) vals[jj] = a16[jj];
            } else {
                tmem_ld16x2(tmem + tlane + c0, tmem + tlane + c0 + 16, a16, b16);
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                    vals[jj] = a16[jj];
                    vals[16 + jj] = b16[jj];
                }
            }
        }
        if (PREP && qk_norm) {
#pragma unroll
            for (int jj = 0; jj < 32; ++jj)
                if (jj < ncol) vals[jj] *= kf_s[c0 + jj];   // column factor f_k,j
        }
        // Decays e^{g_i - g_j} for this thread's columns, j <= i: one exponential at the highest such column,
        // then down the row d(i, j - 1) = d(i, j) alpha_j, so that the special-function unit (which shares
        // the shared-memory instruction queue) runs one exponential per thread instead of one per element.
        {
            const int jstar = min(i, c0 + ncol - 1);
            float dcy = jstar >= c0 ? __expf(g_s[i] - g_s[jstar]) : 0.f;
#pragma unroll
            for (int j4 = 28; j4 >= 0; j4 -= 4) {   // the per-token decays four at a time (one 16-byte load)
                if (j4 >= ncol) continue;
                const float4 al4 = *reinterpret_cast<const float4 *>(al_s + c0 + j4);
                const float al[4] = {al4.x, al4.y, al4.z, al4.w};
#pragma unroll
                for (int e = 3; e >= 0; --e) {
                    const int jj = j4 + e, j = c0 + jj;
                    vals[jj] = j <= jstar ? vals[jj] * dcy : 0.f;
                    if (j <= jstar) dcy *= al[e];
                }
            }
        }
        const bool row_ok = ok && i < L;
        if (quad < 2) {
            const float bi = row_ok ? (PREP ? b_s[i] * kf_s[i] : b_s[i]) : 0.f;   // row factor f_k,i beta_i
            float *arow = reinterpret_cast<float *>(sm + PREP_A) + i * A_LD + c0;
#pragma unroll
            for (int jj = 0; jj < 32; jj += 4) {
                if (jj >= ncol) break;
                float4 a;
                a.x = (c0 + jj + 0 < i) ? bi * vals[jj + 0] : 0.f;
                a.y = (c0 + jj + 1 < i) ? bi * vals[jj + 1] : 0.f;
                a.z = (c0 + jj + 2 < i) ? bi * vals[jj + 2] : 0.f;
                a.w = (c0 + jj + 3 < i) ? bi * vals[jj + 3] : 0.f;
                *reinterpret_cast<float4 *>(arow + jj) = a;
            }
        } else {
            const float fqi = row_ok ? (PREP ? qf_s[i] : 1.f) : 0.f;   // row factor f_q,i
#pragma unroll
            for (int jj = 0; jj < 32; jj += 8) {
                if (jj >= ncol) break;
                float x[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = fqi * vals[jj + e];   // zero above the diagonal already
                uint4 hi, lo;
                split8_bf16(x, hi, lo);
                const uint32_t off = sw128_offset(i, c0 + jj);
                *reinterpret_cast<uint4 *>(sm + PREP_AQK + off) = hi;
                *reinterpret_cast<uint4 *>(sm + PREP_AQK + 8192 + off) = lo;
            }
            if (low_rows) {   // columns 32-63 of rows 0-31 are zero: 16 of them per warp
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const uint32_t off = sw128_offset(i, 32 + 16 * half + 8 * q);
                    *reinterpret_cast<uint4 *>(sm + PREP_AQK + off) = make_uint4(0, 0, 0, 0);
                    *reinterpret_cast<uint4 *>(sm + PREP_AQK + 8192 + off) = make_uint4(0, 0, 0, 0);
                }
            }
        }
    }
    __syncthreads();

    solve_unit_lower_blocked(reinterpret_cast<const float *>(sm + PREP_A), sm, reinterpret_cast<float *>(sm + PREP_Y),
                             tid);
    // (A is no longer read: its space takes the (Gamma T)^T tiles.)

    // Operand tiles: row j of T^T (for R) and of (Gamma T)^T (for P) is column j of T, split into bf16 hi/lo.
    // Thread t covers row j = t % 64, columns i in [16 (t / 64), 16 (t / 64) + 16) (the lanes of a warp read
    // 32 consecutive words of a row of T).  T is read into registers first, because the T^T tiles then
    // overwrite it.
    {
        const int j = tid & 63, i0 = (tid >> 6) * 16;
        float tv[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) tv[e] = t_row(sm, i0 + e)[j];
        __syncthreads();
        if (ok) {
            uint8_t *tth = sm + PREP_KQ + 8192, *ttl = sm + PREP_KQ + 24576;   // over T
            uint8_t *gth = sm + PREP_A, *gtl = sm + PREP_A + 8192;
#pragma unroll
            for (int c8 = 0; c8 < 16; c8 += 8) {
                float g8[8];
#pragma unroll
                for (int e4 = 0; e4 < 8; e4 += 4) {
                    const float4 gm = *reinterpret_cast<const float4 *>(gam_s + i0 + c8 + e4);
                    g8[e4] = gm.x * tv[c8 + e4];
                    g8[e4 + 1] = gm.y * tv[c8 + e4 + 1];
                    g8[e4 + 2] = gm.z * tv[c8 + e4 + 2];
                    g8[e4 + 3] = gm.w * tv[c8 + e4 + 3];
                }
                const uint32_t off = sw128_offset(j, i0 + c8);
                uint4 hi, lo;
                split8_bf16(tv + c8, hi, lo);
                *reinterpret_cast<uint4 *>(tth + off) = hi;
                *reinterpret_cast<uint4 *>(ttl + off) = lo;
                split8_bf16(g8, hi, lo);
                *reinterpret_cast<uint4 *>(gth + off) = hi;
                *reinterpret_cast<uint4 *>(gtl + off) = lo;
            }
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (ok && tid == 0) {
        // P = K^T (Gamma T): A = K tile read MN-major (M = dk = 128), B = (Gamma T)^T hi then lo
        constexpr uint32_t idp = idesc_bf16_f32(128, 64, true, false);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) mma_bf16(tmem + 64, dk_mn + 128 * kk, dgth + 2 * kk, idp, kk > 0);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) mma_bf16(tmem + 64, dk_mn + 128 * kk, dgtl + 2 * kk, idp, 1);
        // R = Aqk T (M = 64): Aqk_hi T_hi + Aqk_hi T_lo + Aqk_lo T_hi
        constexpr uint32_t idr = idesc_bf16_f32(64, 64, false, false);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) mma_bf16(tmem, dah + 2 * kk, dth + 2 * kk, idr, kk > 0);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) mma_bf16(tmem, dah + 2 * kk, dtl + 2 * kk, idr, 1);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) mma_bf16(tmem, dal + 2 * kk, dth + 2 * kk, idr, 1);
        mma_commit(&bar_mma);
    }
    if (ok) ok = mbar_wait(&bar_mma, 1);
    ok = __syncthreads_and(ok);
    tc_fence_after();

    // Stage P (rows d = TMEM lane, 64 columns), then R (rows 16 quad + lane for lane < 16, M = 64 accumulator),
    // as bf16 hi / lo tiles in the same 128B-swizzled layout the TMA maps use, over operand tiles that the
    // finished MMAs no longer read; each tile leaves with one bulk tensor store, P's while R is staged.  The
    // two warps of a quadrant take 32 columns each.
    const int cb = 32 * half;
    if (ok) {
        uint8_t *sph = sm + PREP_KQ, *spl = sm + PREP_KQ + 16384;     // 16 KiB each
        float a[16], b[16];
        tmem_ld16x2(tmem + tlane + 64 + cb, tmem + tlane + 64 + cb + 16, a, b);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint4 hi, lo;
            split8_bf16(q < 2 ? a + 8 * q : b + 8 * (q - 2), hi, lo);
            const uint32_t off = sw128_offset(32 * quad + lane, cb + 8 * q);
            *reinterpret_cast<uint4 *>(sph + off) = hi;
            *reinterpret_cast<uint4 *>(spl + off) = lo;
        }
        fence_proxy_async_smem();
    }
    __syncthreads();
    if (ok && tid == 0) {
        const int prow = (gc * hv + h) * D;
        if (GDN_INB((long)prow + D - 1, (long)nch * hv * D, err)) {
            tma_store_2d(&phmap, sm + PREP_KQ, 0, prow);
            tma_store_2d(&plmap, sm + PREP_KQ + 16384, 0, prow);
        }
        tma_store_commit();
    }
    if (ok) {
        uint8_t *srh = sm + PREP_A, *srl = sm + PREP_A + 8192;        // 8 KiB each
        const int r = 16 * quad + lane;
        float a[16], b[16];
        tmem_ld16x2(tmem + tlane + cb, tmem + tlane + cb + 16, a, b);
        if (lane < 16) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint4 hi, lo;
                split8_bf16(q < 2 ? a + 8 * q : b + 8 * (q - 2), hi, lo);
                const uint32_t off = sw128_offset(r, cb + 8 * q);
                *reinterpret_cast<uint4 *>(srh + off) = hi;
                *reinterpret_cast<uint4 *>(srl + off) = lo;
            }
        }
        fence_proxy_async_smem();
    }
    __syncthreads();
    if (ok && tid == 0) {
        const int rrow = (gc * hv + h) * C;
        if (GDN_INB((long)rrow + C - 1, (long)nch * hv * C, err)) {
            tma_store_2d(&rhmap, sm + PREP_A, 0, rrow);
            tma_store_2d(&rlmap, sm + PREP_A + 8192, 0, rrow);
        }
        tma_store_commit();
        tma_store_wait_read();
    } else if (tid == 0) {
        raise_error(err, kErrTimeout);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 2) tmem_dealloc(tmem, PREP_TMEM_COLS);
}

// ============================================================================
// Kernel 2: state passing + outputs (sequential over chunks)
// ============================================================================
// One pipeline stage: Q|K 32 KiB, P_hi 16, P_lo 16, R_hi 8, R_lo 8 KiB.  R feeds M = 128 MMAs whose upper 64
// accumulator rows are unused: the group on R_hi reads R_lo as its upper rows, the accumulating group on R_lo
// reads whatever follows it (the next stage's Q|K, or the state operand), so the valid rows hold
// (R_hi + R_lo) X and the upper ones anything (never read).
constexpr uint32_t PASS_STAGE = 81920;
constexpr uint32_t ST_QK = 0, ST_PH = 32768, ST_PL = 49152, ST_RH = 65536, ST_RL = 73728;
constexpr uint32_t PASS_SOP = 2 * PASS_STAGE;      // [S_hi ; S_lo] tile, 2 k-blocks x 8 KiB
constexpr uint32_t PASS_XOP = PASS_SOP + 16384;    // [X_hi ; X_lo] tile(s) [64 x 64] bf16 (state_pass_kernel: by chunk parity)
constexpr uint32_t PASS_SMEM = PASS_XOP + 2 * 8192 + 1024;
constexpr uint32_t kQkTx = 32768;                                   // Q|K of a stage
constexpr uint32_t PASS_TMEM_COLS = 256;
// TMEM columns (each accumulator 64 columns: 32 for the S_hi / X_hi part, 32 for the S_lo / X_lo part):
//   [Q;K] [S_hi;S_lo]^T  (M = 128 token rows: Q rows in lanes 0-63, K rows in 64-127);
//   P X                  (M = 128 = dk), P_hi X and P_lo X accumulated together;
//   R X                  (M = 128, rows 0-63 valid), double-buffered by chunk parity so that a chunk's
//                        outputs can be read while the next chunk's R X is computed.
// A chain of MMAs into one accumulator runs as fast as independent ones, so each product has one.
constexpr uint32_t TM_D1 = 0, TM_PX = 64, TM_RX = 128;

// Q and K rows of the chunk starting at token t0 (q/k head hq) into a stage (the caller arms the barrier).
__device__ __forceinline__ void pass_load_qk(uint8_t *st, uint64_t *bar, const CUtensorMap *qmap,
                                             const CUtensorMap *kmap, int hq, int t0, int hk, int total,
                                             unsigned int *err) {
    // (bounds-checking build: the tile's columns inside the q/k rows, its first token inside the tokens)
    if (!GDN_INB(hq * D + 127, hk * D, err) || !GDN_INB(t0, total, err)) return;
    (void)hk; (void)total; (void)err;
#pragma unroll
    for (int kb = 0; kb < 2; ++kb) {
        tma_load_2d(st + ST_QK + kb * 16384, qmap, bar, hq * D + kb * 64, t0);
        tma_load_2d(st + ST_QK + kb * 16384 + 8192, kmap, bar, hq * D + kb * 64, t0);
    }
}

// 8 warps: warps w and w + 4 share TMEM lane quadrant w % 4 and split the CTA's 32 value rows (NG row groups).
// 128 and 512 threads (32 and 8 rows per thread) measured 119 and 146 us against 115 us at the 4K layer.
constexpr int kPassThreads = 256;
constexpr int NG = kPassThreads / 128;

constexpr int DG = DS / NG;         // state rows per thread

// Per-chunk inputs that are read with plain loads (gates, beta, this thread's v
// row piece); loaded one chunk ahead so that their latency is off the state chain.
struct ChunkInputs {
    float la0, la1;   // log_alpha of tokens 2*lane, 2*lane+1 (raw; 0 past the end)
    float f;          // q/k preparation factor of this thread's token row (f_k for K rows, f_q for Q rows)
    float b;          // beta of this thread's token row (K-row threads)
    uint4 v[DG / 8];  // DG bf16 of this thread's v row piece (K-row threads)
};

__device__ __forceinline__ void load_chunk_inputs(ChunkInputs &in, const float *__restrict__ log_alpha,
                                                  const float *__restrict__ beta, const __nv_bfloat16 *__restrict__ v,
                                                  const float *__restrict__ norms, float q_scale, int gcx, int t0,
                                                  int L, int hv, int h, int rowg, int lane, bool krow, int i,
                                                  int total, int nch, unsigned int *err) {
    const int i0 = 2 * lane, i1 = 2 * lane + 1;
    const long g_n = (long)total * hv;
    (void)g_n; (void)nch; (void)err;
    // norms is null without qk_norm: the factors are then 1 (k) and q_scale (q)
    const size_t fi = ((size_t)gcx * hv + h) * 128 + (krow ? i : 64 + i);
    in.f = norms ? (GDN_INB(fi, (long)nch * hv * 128, err) ? norms[fi] : 0.f) : (krow ? 1.f : q_scale);
    in.la0 = i0 < L && GDN_INB((size_t)(t0 + i0) * hv + h, g_n, err) ? log_alpha[(size_t)(t0 + i0) * hv + h] : 0.f;
    in.la1 = i1 < L && GDN_INB((size_t)(t0 + i1) * hv + h, g_n, err) ? log_alpha[(size_t)(t0 + i1) * hv + h] : 0.f;
    in.b = 0.f;
#pragma unroll
    for (int q4 = 0; q4 < DG / 8; ++q4) in.v[q4] = make_uint4(0, 0, 0, 0);
    const size_t vi = ((size_t)(t0 + i) * hv + h) * D + rowg;
    if (krow && i < L && GDN_INB(vi + DG - 1, g_n * D, err)) {
        in.b = beta[(size_t)(t0 + i) * hv + h];
        const uint4 *vp = reinterpret_cast<const uint4 *>(v + vi);
#pragma unroll
        for (int q4 = 0; q4 < DG / 8; ++q4) in.v[q4] = vp[q4];
    }
}


// GATE: the gates of a chunk from raw inputs, formed when the chunk is used (one chunk after its loads were
// issued, so their latency stays hidden): log_alpha of tokens 2 lane and 2 lane + 1, beta of this thread's
// token.  Positions past the chunk's end keep their zeros.
template <bool GATE>
__device__ __forceinline__ void finish_gates(ChunkInputs &in, int L, int lane, bool krow, int i,
                                             const float *__restrict__ gate_c, const float *__restrict__ gate_b,
                                             int h) {
    if (!GATE) return;
    if (2 * lane < L) in.la0 = gate_log_alpha(in.la0, gate_c, gate_b, h);
    if (2 * lane + 1 < L) in.la1 = gate_log_alpha(in.la1, gate_c, gate_b, h);
    if (krow && i < L) in.b = gate_beta(in.b, gate_c);
}

// Outputs of one chunk for this thread's token and 16 value rows (Q-row threads):
// O_i = e^{g_i} (Q S^T)_i (in qs) + (R X)_i ((R_hi + R_lo) X_hi, and (R_hi + R_lo) X_lo).
// outputs_begin adds R X into qs (`valid` false skips TMEM); outputs_end writes them.
__device__ __forceinline__ void outputs_begin(float (&qs)[DG], uint32_t tmem_rx, int grp, bool valid) {
    if (valid) {
        float a[DG], b[DG];
        tmem_ldx2<DG>(tmem_rx + grp * DG, tmem_rx + 32 + grp * DG, a, b);
#pragma unroll
        for (int e = 0; e < DG; ++e) qs[e] += a[e] + b[e];
    }
}

__device__ __forceinline__ void outputs_end(const float (&qs)[DG], int i, int L, int t0, int hv, int h, int rowg,
                                            void *__restrict__ out, int out_f32, bool valid, long out_n,
                                            unsigned int *err) {
    (void)out_n;
    if (valid && i < L && GDN_INB(((size_t)(t0 + i) * hv + h) * D + rowg + DG - 1, out_n, err)) {
        const size_t o = ((size_t)(t0 + i) * hv + h) * D + rowg;
        if (out_f32) {
            float4 *op = reinterpret_cast<float4 *>(reinterpret_cast<float *>(out) + o);
#pragma unroll
            for (int e = 0; e < DG / 4; ++e) op[e] = make_float4(qs[4 * e], qs[4 * e + 1], qs[4 * e + 2], qs[4 * e + 3]);
        } else {
            uint4 *op = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(out) + o);
#pragma unroll
            for (int e = 0; e < DG / 8; ++e)
                op[e] = make_uint4(pack_bf16(qs[8 * e], qs[8 * e + 1]), pack_bf16(qs[8 * e + 2], qs[8 * e + 3]),
                                   pack_bf16(qs[8 * e + 4], qs[8 * e + 5]), pack_bf16(qs[8 * e + 6], qs[8 * e + 7]));
        }
    }
}

// Thread roles (320 threads).  Warps 0-7 compute: TMEM lane quadrant quad = warp % 4, row group grp = warp / 4
// (which DG = 16 of the CTA's 32 value rows).  Lane l of quadrant quad is accumulator row 32 quad + l: for
// [Q;K] S^T and R X that row is a token (Q rows for quad 0-1, K rows for quad 2-3); for P X it is state
// column d.  Lane 0 of warp 8 issues every MMA and lane 0 of warp 9 every tensor load.  The compute warps never wait behind an
// issuing thread (a tensor load's issue can stall its thread for thousands of cycles when memory is busy):
// they meet the issuers through mbarriers only, two per chunk.
//   bar_x[b]  X buffer b written (128 arrivals, the K-row threads)              -> P X, later R X
//   bar_s     state operand of the next chunk written (256 arrivals, after the state update) -> [Q;K] S^T
// Per chunk c the MMA thread waits for the chunk's Q|K and bar_s, issues [Q;K] S^T (commit bar_d1), then chunk
// c - 1's R X (the pipe runs it while the X values are computed), waits for P and bar_x and issues P X
// (commit bar_px).  The tensor pipe runs small MMAs one after another, so the state chain's two groups never
// queue behind R X.
// Tiles: Q|K, P and R each have a full barrier (landed) and a free barrier per stage (the MMA thread commits
// it once its reads of that stage are complete); the load thread refills a stage part only after its free
// barrier.  Every wait is on a phase that cannot be overtaken before the waiter acts (each barrier's next
// phase depends on work the waiter has still to do), so parities never alias.
// The four waits of the state chain (state operand and X buffer written; [Q;K] S^T and P X complete) spin on
// mbarrier.test_wait instead of try_wait, which may suspend the waiting thread: 109 against 113 us at the
// 4K layer.
constexpr int kWsThreads = kPassThreads + 64;
constexpr int kMmaWarp = kPassThreads / 32, kTmaWarp = kMmaWarp + 1;
constexpr uint32_t kPTx = 16384 + 16384, kRTx = 8192 + 8192;

// MULTI: a CTA may carry several sequences (buckets of more than one); without it each bucket is one sequence
// and the chunk loop has none of the sequence-boundary code.
// NORM: the output normalisation o <- o / sqrt(mean_head(o^2) + eps) * w over the head's 128 rows, which the
// four slice CTAs of a (bucket, head) hold 32 each; they form a cluster.  Per chunk every Q-row thread writes
// its token's sum of squares over its 16 rows into its CTA's block of the slot array (two slot sets by chunk
// parity); the last of the 128 Q-row threads to count itself in (a shared counter) sends the block (512 bytes)
// to the same place in each peer CTA with a bulk copy that completes on the peer's norm barrier, and arms its
// own barrier for the three peers' blocks.  After the state update every Q-row thread waits on its own barrier
// and adds its token's eight sums.  Only the Q-row threads take part, so the MMA and tile warps never wait on
// the cluster, and the wait is off the state chain.  A slot set is
// written again two chunks later: by then the peers have received this CTA's block of the chunk in between,
// which it sends only after reading; the barrier's phases advance the same way, so they never alias.
template <bool GATE, bool MULTI, bool NORM>
__global__ void __launch_bounds__(kWsThreads, 1)
state_pass_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                  const __grid_constant__ CUtensorMap phmap, const __grid_constant__ CUtensorMap plmap,
                  const __grid_constant__ CUtensorMap rhmap, const __grid_constant__ CUtensorMap rlmap,
                  const __nv_bfloat16 *__restrict__ v, const float *__restrict__ norms, float q_scale,
                  const float *__restrict__ log_alpha, const float *__restrict__ beta,
                  const float *__restrict__ init_state, const int32_t *__restrict__ cu, int n_seqs, int total,
                  int nch, int hk, int hv, void *__restrict__ out, int out_f32, float *__restrict__ final_state,
                  const float *__restrict__ gate_c, const float *__restrict__ gate_b, unsigned int *err,
                  const __grid_constant__ PassBuckets bk, const float *__restrict__ norm_w, float norm_eps) {
    extern __shared__ uint8_t pass_raw[];
    uint8_t *sm = align1024(pass_raw);
    __shared__ uint64_t bar_qk[2], bar_p[2], bar_r[2], bar_qkf[2], bar_pf[2], bar_rf[2];
    __shared__ uint64_t bar_s, bar_x[2], bar_d1, bar_px, bar_rx[2];
    __shared__ uint64_t bar_norm[2];   // (NORM) the peers' sums of a chunk have landed, by chunk parity
    __shared__ uint32_t nsum_count;    // (NORM) Q-row threads that have written their sums, over all chunks so far
    // [chunk parity][cluster rank][row group][token]; the bulk copies need 16-byte aligned blocks
    __shared__ __align__(128) float norm_part[NORM ? 2 * 4 * NG * 64 : 4];
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int abort_flag;   // set by any thread whose wait ran out; everyone stops at the next check
    __shared__ int warp_chunks[kWsThreads / 32];

    constexpr int SLICES = D / DS;
    const int slice = blockIdx.x % SLICES;
    const int h = (blockIdx.x / SLICES) % hv;
    const int bucket = blockIdx.x / (SLICES * hv);
    const int hq = h / (hv / hk);
    const int row0 = slice * DS;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t base = smem_u32(sm);

    // this CTA's sequences [sa, sb) and their chunks [gc0, gc0 + nchunks), carried one after another
    const int sa = bk.per_seq ? bucket : bk.seq[bucket], sb = bk.per_seq ? bucket + 1 : bk.seq[bucket + 1];
    const int gc0 = bk.per_seq ? (n_seqs > 1 && bucket < n_seqs ? first_chunk_of(cu, bucket, total) : 0)
                               : bk.chunk[bucket];
    int nchunks = bk.per_seq ? 0 : bk.chunk[bucket + 1] - gc0;   // per_seq: counted below
    const bool table_ok = sa >= 0 && sa <= sb && sb <= n_seqs && gc0 >= 0 && nchunks >= 0 && gc0 + nchunks <= nch;
    {   // the chunks the device's cu_seqlens gives these sequences, counted by all threads (summed below)
        int cnt = 0;
        if (table_ok) {
            if (n_seqs == 1) {
                if (tid == 0) cnt = (total + C - 1) / C;
            } else {
                for (int m = sa + tid; m < sb; m += kWsThreads) {
                    int a, b;
                    seq_range(cu, m, total, a, b);
                    cnt += (b - a + C - 1) / C;
                }
            }
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, off);
        if (lane == 0) warp_chunks[warp] = cnt;
    }
    auto no_op = [](int) {};

    if (warp == 0) {
        tmem_alloc(&tmem_slot, PASS_TMEM_COLS);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bar_qk[b], 1);
            mbar_init(&bar_p[b], 1);
            mbar_init(&bar_r[b], 1);
            mbar_init(&bar_qkf[b], 1);
            mbar_init(&bar_pf[b], 1);
            mbar_init(&bar_rf[b], 1);
            mbar_init(&bar_x[b], 128);
            mbar_init(&bar_rx[b], 1);
        }
        mbar_init(&bar_s, kPassThreads);
        mbar_init(&bar_d1, 1);
        mbar_init(&bar_px, 1);
        if (NORM) {
            mbar_init(&bar_norm[0], 1);
            mbar_init(&bar_norm[1], 1);
        }
        abort_flag = 0;
        nsum_count = 0;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (NORM) cluster_sync();   // every CTA's norm barrier is initialised before any peer arrives on it
    const uint32_t tmem = tmem_slot;
    // the planned chunks must be the ones the device's sequence table gives (a host copy that disagrees with it
    // would send the loads past the planned range): otherwise record the error and run nothing
    int dev_chunks = 0;
#pragma unroll
    for (int w = 0; w < kWsThreads / 32; ++w) dev_chunks += warp_chunks[w];
    if (bk.per_seq) nchunks = dev_chunks;
    const bool range_ok = table_ok && dev_chunks == nchunks && gc0 + nchunks <= nch;
    if (!range_ok && tid == 0) raise_error(err, kErrInternal);
    const bool started = range_ok && nchunks > 0;

    // Shared-memory descriptors (the same for every thread, built outside divergent code); a K step adds a
    // byte offset >> 4 to the start field (all tiles sit far below 256 KiB, so the 14-bit field never carries).
    const uint64_t dQK0 = smem_desc(base + ST_QK, 16, 1024, kSW);
    const uint64_t dPH0 = smem_desc(base + ST_PH, 16, 1024, kSW);
    const uint64_t dPL0 = smem_desc(base + ST_PL, 16, 1024, kSW);
    const uint64_t dRH0 = smem_desc(base + ST_RH, 16, 1024, kSW);
    const uint64_t dRL0 = smem_desc(base + ST_RL, 16, 1024, kSW);
    const uint64_t dSOP = smem_desc(base + PASS_SOP, 8192, 1024, kSW);
    const uint64_t dXOP = smem_desc(base + PASS_XOP, 8192, 1024, kSW);   // + parity * (8192 >> 4)
    constexpr uint64_t kStageStep = PASS_STAGE >> 4;
    constexpr uint32_t idb = idesc_bf16_f32(128, 64, false, true);
    auto ph = [](int cc) { return (uint32_t)((cc >> 1) & 1); };   // phase parity of chunk cc on a per-stage barrier
    auto stop = [&]() { return abort_flag != 0; };
    auto fail = [&]() { abort_flag = 1; };

    if (warp == kMmaWarp) {
        if (lane == 0 && started) {
            // R X of chunk cc (64 valid rows x 64) = (R_hi + R_lo) [X_hi ; X_lo]^T into TMEM buffer cc & 1
            auto issue_rx = [&](int cc) -> bool {
                const int sc = cc & 1;
                if (!mbar_wait(&bar_r[sc], ph(cc))) return false;
                const uint64_t soc = sc * kStageStep, dx = dXOP + sc * (8192 >> 4);
                const uint32_t rx = tmem + TM_RX + 64 * sc;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) mma_bf16(rx, dRH0 + soc + 2 * kk, dx + 128 * kk, idb, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) mma_bf16(rx, dRL0 + soc + 2 * kk, dx + 128 * kk, idb, 1);
                mma_commit(&bar_rx[sc]);
                mma_commit(&bar_rf[sc]);
                return true;
            };
            bool ok = true;
            for (int c = 0; ok && c < nchunks; ++c) {
                if (stop()) break;
                const int s = c & 1;
                const uint64_t so = s * kStageStep;
                // D1[128 x 64] = [Q ; K] [S_hi ; S_lo]^T once this chunk's Q|K and the state operand are in place
                // (tiles first: they land early, the state operand is the chain)
                ok = mbar_wait(&bar_qk[s], ph(c)) && mbar_spin(&bar_s, (uint32_t)(c & 1));
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t off = (uint64_t)(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
                    mma_bf16(tmem + TM_D1, dQK0 + so + off, dSOP + 128 * kk, idb, kk > 0);
                }
                mma_commit(&bar_d1);
                mma_commit(&bar_qkf[s]);
                if (c > 0 && !(ok = issue_rx(c - 1))) break;   // X of chunk c - 1 is complete: its P X ran
                // P X (dk x 64) = P_hi [X_hi ; X_lo]^T + P_lo [X_hi ; X_lo]^T once this chunk's P and X are in place
                ok = mbar_wait(&bar_p[s], ph(c)) && mbar_spin(&bar_x[s], ph(c));
                if (!ok) break;
                const uint64_t dx = dXOP + s * (8192 >> 4);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    mma_bf16(tmem + TM_PX, dPH0 + so + 2 * kk, dx + 128 * kk, idb, kk > 0);
                    mma_bf16(tmem + TM_PX, dPL0 + so + 2 * kk, dx + 128 * kk, idb, 1);
                }
                mma_commit(&bar_px);
                mma_commit(&bar_pf[s]);
            }
            // the last chunk's R X, once its X is written
            if (ok && !stop()) ok = mbar_wait(&bar_x[(nchunks - 1) & 1], ph(nchunks - 1)) && issue_rx(nchunks - 1);
            if (!ok) fail();
        }
        __syncwarp();
    } else if (warp == kTmaWarp) {
        if (lane == 0 && started) {
            tma_prefetch_desc(&qmap);
            tma_prefetch_desc(&kmap);
            tma_prefetch_desc(&phmap);
            tma_prefetch_desc(&plmap);
            tma_prefetch_desc(&rhmap);
            tma_prefetch_desc(&rlmap);
            // Q|K, P and R of chunk cc into stage cc & 1; the Q|K requests go in chunk order, following the
            // run's token rows with a cursor
            ChunkCursor qc;
            cursor_seek(qc, cu, n_seqs, total, sa, sb, no_op);
            auto load_qk = [&](int cc) {
                mbar_arrive_expect_tx(&bar_qk[cc & 1], kQkTx);
                pass_load_qk(sm + (cc & 1) * PASS_STAGE, &bar_qk[cc & 1], &qmap, &kmap, hq, qc.t0(), hk, total, err);
                cursor_next(qc, cu, n_seqs, total, sb, no_op);
            };
            auto load_p = [&](int cc) {
                uint8_t *st = sm + (cc & 1) * PASS_STAGE;
                const int prow = ((gc0 + cc) * hv + h) * D;
                mbar_arrive_expect_tx(&bar_p[cc & 1], kPTx);
                if (!GDN_INB((long)prow + D - 1, (long)nch * hv * D, err)) return;
                tma_load_2d(st + ST_PH, &phmap, &bar_p[cc & 1], 0, prow);
                tma_load_2d(st + ST_PL, &plmap, &bar_p[cc & 1], 0, prow);
            };
            auto load_r = [&](int cc) {
                uint8_t *st = sm + (cc & 1) * PASS_STAGE;
                const int rrow = ((gc0 + cc) * hv + h) * C;
                mbar_arrive_expect_tx(&bar_r[cc & 1], kRTx);
                if (!GDN_INB((long)rrow + C - 1, (long)nch * hv * C, err)) return;
                tma_load_2d(st + ST_RH, &rhmap, &bar_r[cc & 1], 0, rrow);
                tma_load_2d(st + ST_RL, &rlmap, &bar_r[cc & 1], 0, rrow);
            };
            // both stages start empty; Q|K come from the inputs, P and R from the preparation, which may still
            // be finishing (programmatic dependent launch)
            int nq = min(2, nchunks), np = nq, nr = nq;   // chunks < nq (np, nr) have had Q|K (P, R) requested
            for (int cc = 0; cc < nq; ++cc) load_qk(cc);
            grid_dependency_wait();
            for (int cc = 0; cc < nq; ++cc) {
                load_p(cc);
                load_r(cc);
            }
            // stage c & 1 takes chunk c + 2 once chunk c has finished with it: Q|K after [Q;K] S^T, P after
            // P X, R after R X (which runs during chunk c + 1)
            bool ok = true;
            for (int c = 0; c + 2 < nchunks; ++c) {
                if (stop()) break;
                const int s = c & 1;
                if (!(ok = mbar_wait(&bar_qkf[s], ph(c)))) break;
                load_qk(c + 2);
                nq = c + 3;
                if (!(ok = mbar_wait(&bar_pf[s], ph(c)))) break;
                load_p(c + 2);
                np = c + 3;
                if (!(ok = mbar_wait(&bar_rf[s], ph(c)))) break;
                load_r(c + 2);
                nr = c + 3;
            }
            if (!ok) fail();
            // every requested tile has landed before the CTA can end (normally all were consumed); each
            // barrier has at most one phase outstanding, the last one armed
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                const int aq = (nq - b + 1) / 2, ap = (np - b + 1) / 2, ar = (nr - b + 1) / 2;
                if (aq > 0) mbar_wait(&bar_qk[b], (uint32_t)((aq - 1) & 1));
                if (ap > 0) mbar_wait(&bar_p[b], (uint32_t)((ap - 1) & 1));
                if (ar > 0) mbar_wait(&bar_r[b], (uint32_t)((ar - 1) & 1));
            }
        }
        __syncwarp();
    } else {
        // compute warps
        const int quad = warp & 3, grp = warp >> 2;
        const int lrow = 32 * quad + lane;
        const int d = lrow;
        const int i = lrow & 63;
        const bool krow = quad >= 2;
        const int rowg = row0 + grp * DG;
        const uint32_t tlane = (uint32_t)(32 * quad) << 16;

        // this thread's state elements S[rowg + r][d] of sequence m start at sbase_of(m) + r D
        auto sbase_of = [&](int m) { return (((size_t)m * hv + h) * D + rowg) * D + d; };
        auto state_in_range = [&](size_t sbase) {
            return GDN_INB(sbase + (size_t)(DG - 1) * D, (long)n_seqs * hv * D * D, err);
        };
        // a sequence without tokens returns its initial state
        auto copy_empty = [&](int m) {
            const size_t sbm = sbase_of(m);
            if (!final_state || !state_in_range(sbm)) return;
#pragma unroll
            for (int r = 0; r < DG; ++r) final_state[sbm + (size_t)r * D] = init_state ? init_state[sbm + (size_t)r * D] : 0.f;
        };
        if (norms) grid_dependency_wait();   // the q/k preparation factors come from the preparation
        // cur_c: chunk c; pre_c: the chunk whose inputs are loaded next.  Per-chunk inputs are loaded two chunks
        // ahead: under the pass's tile traffic a global load can take longer than one chunk (one chunk ahead left
        // the K-row threads waiting on them at the top of the loop).
        ChunkCursor cur_c;
        if (!range_ok) cursor_seek(cur_c, cu, n_seqs, total, 0, 0, no_op);   // nothing (the bucket table is invalid)
        else if (MULTI) cursor_seek(cur_c, cu, n_seqs, total, sa, sb, copy_empty);
        else cursor_at_seq(cur_c, cu, n_seqs, total, sa);
        ChunkCursor pre_c = cur_c;
        ChunkInputs nxt, nxt2;
        if (started) {
            load_chunk_inputs(nxt, log_alpha, beta, v, norms, q_scale, gc0, pre_c.t0(), pre_c.len(), hv, h, rowg,
                              lane, krow, i, total, nch, err);
            cursor_next(pre_c, cu, n_seqs, total, sb, no_op);
            if (nchunks > 1) {
                load_chunk_inputs(nxt2, log_alpha, beta, v, norms, q_scale, gc0 + 1, pre_c.t0(), pre_c.len(), hv, h,
                                  rowg, lane, krow, i, total, nch, err);
                cursor_next(pre_c, cu, n_seqs, total, sb, no_op);
            }
        }
        float S[DG];
        size_t sbase = sbase_of(MULTI ? cur_c.n : sa);
        ChunkCursor next_c = cur_c;   // (MULTI) the first chunk of the next sequence, found a chunk early
        bool next_ok = false;         // (MULTI) its initial state is read (fetched into L2 a chunk early)
        // (one sequence per CTA: an empty one returns its initial state through the store after the loop)
        bool state_ok = (MULTI ? started : range_ok) && state_in_range(sbase);
#pragma unroll
        for (int r = 0; r < DG; ++r) S[r] = init_state && state_ok ? init_state[sbase + (size_t)r * D] : 0.f;
        auto write_sop = [&]() {
#pragma unroll
            for (int j = 0; j < DG / 8; ++j) {
                uint4 hi, lo;
                split8_bf16(&S[8 * j], hi, lo);
                *reinterpret_cast<uint4 *>(sm + PASS_SOP + sw128_offset(d, grp * DG + 8 * j)) = hi;
                *reinterpret_cast<uint4 *>(sm + PASS_SOP + sw128_offset(d, DS + grp * DG + 8 * j)) = lo;
            }
        };
        // publish the state operand: generic writes made visible to the tensor cores, TMEM reads of this
        // thread ordered before the MMAs that follow
        auto publish_sop = [&]() {
            write_sop();
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&bar_s);
        };
        if (started) publish_sop();

        float qs[DG], qcur[DG];   // Q-row threads: outputs being finished, and this chunk's e^g f_q Q S^T
        int prev_t0 = 0, prev_L = 0;
        const uint32_t crank = NORM ? cluster_ctarank() : 0u;
        // Outputs of chunk j (Q-row threads; qs holds e^g f_q Q S^T, R X is in TMEM at trx), in two steps so that
        // with NORM the exchange of the head's sums of squares waits off the state chain: send_outputs adds R X
        // and sends this CTA's sums (NORM), finish_outputs (after the state update) waits for the peers' sums,
        // normalises and writes.  finish_outputs is false when the exchange timed out.
        auto send_outputs = [&](int j, uint32_t trx, bool valid) {
            outputs_begin(qs, trx, grp, valid);
            if (NORM) {
                float ss = 0.f;
                if (valid && i < prev_L) {
#pragma unroll
                    for (int e = 0; e < DG; ++e) ss = fmaf(qs[e], qs[e], ss);
                }
                const int np = j & 1;
                constexpr uint32_t kBlock = NG * 64 * 4;   // one CTA's sums of a chunk, bytes
                float *mine = norm_part + (np * 4 + (int)crank) * NG * 64;
                mine[grp * 64 + i] = ss;
                fence_proxy_async_smem();   // read by the bulk copies
                // The last of the 128 Q-row threads to count itself in (acquire-release: every other thread's
                // sums and proxy fence come before) sends.  Nobody waits here: a named barrier would block for
                // good on a thread whose own bounded wait ran out and left the loop, while a missing count only
                // means no send, and the peers' waits, then this CTA's own, run out in turn.
                if (count_in_shared(&nsum_count) == 128u * (uint32_t)(j + 1) - 1u) {
#pragma unroll
                    for (uint32_t rk = 0; rk < 4; ++rk)
                        if (rk != crank) bulk_copy_to_peer(mine, mine, kBlock, &bar_norm[np], rk);
                    mbar_arrive_expect_tx(&bar_norm[np], 3 * kBlock);
                }
            }
        };
        auto finish_outputs = [&](int j, bool valid) -> bool {
            bool got = true;
            if (NORM) {
                const int np = j & 1;
                got = mbar_spin_cluster(&bar_norm[np], (uint32_t)((j >> 1) & 1));
                float tot = 0.f;
#pragma unroll
                for (int rk = 0; rk < 4; ++rk)
#pragma unroll
                    for (int g = 0; g < NG; ++g) tot += norm_part[((np * 4 + rk) * NG + g) * 64 + i];
                const float sc = rsqrtf(tot * (1.f / D) + norm_eps);
#pragma unroll
                for (int e = 0; e < DG; ++e) qs[e] *= sc * norm_w[rowg + e];
            }
            outputs_end(qs, i, prev_L, prev_t0, hv, h, rowg, out, out_f32, valid && got, (long)total * hv * D, err);
            return got;
        };
        bool ok = range_ok;   // an empty sequence runs no chunk and returns its initial state
        int c = 0;
        for (; ok && c < nchunks; ++c) {
            if (stop()) {
                ok = false;
                break;
            }
            const uint32_t par = c & 1;
            const int t0 = cur_c.t0(), L = cur_c.len();
            const bool seq_end = MULTI && cur_c.last_of_seq();
            if (MULTI && seq_end) {
                // the next sequence (sequences without tokens in between return their initial states now) and
                // its initial state, so that neither lookup waits at the sequence boundary
                next_c = cur_c;
                cursor_next(next_c, cu, n_seqs, total, sb, copy_empty);
                const size_t nsb = sbase_of(next_c.n);
                next_ok = c + 1 < nchunks && init_state && state_in_range(nsb);
                if (next_ok) {
#pragma unroll
                    for (int r = 0; r < DG; ++r) prefetch_l2(init_state + nsb + (size_t)r * D);
                }
            }
            ChunkInputs cur = nxt;
            nxt = nxt2;
            finish_gates<GATE>(cur, L, lane, krow, i, gate_c, gate_b, h);
            if (c + 2 < nchunks) {
                load_chunk_inputs(nxt2, log_alpha, beta, v, norms, q_scale, gc0 + c + 2, pre_c.t0(), pre_c.len(), hv,
                                  h, rowg, lane, krow, i, total, nch, err);
                if (MULTI) cursor_next(pre_c, cu, n_seqs, total, sb, no_op);
                else ++pre_c.k;
            }
            const float2 g2 = cumsum_pairs(cur.la0, cur.la1, L, lane);
            const float gL = g_of(g2, L - 1);
            const float eg = __expf(g_of(g2, i));

            if (!mbar_spin(&bar_d1, par)) ok = false;
            tc_fence_after();
            if (krow) {
                // X_i = beta_i (v_i - e^{g_i} (K S^T)_i) into X buffer c & 1, whose last reader (R X of chunk
                // c - 2) must be complete
                if (c > 1 && !mbar_wait(&bar_rx[par], ph(c - 2))) ok = false;
                tc_fence_after();
                float a[DG], b[DG];
                tmem_ldx2<DG>(tmem + tlane + TM_D1 + grp * DG, tmem + tlane + TM_D1 + 32 + grp * DG, a, b);
                const float bi = cur.b, be = cur.b * eg * cur.f;
#pragma unroll
                for (int q4 = 0; q4 < DG / 8; ++q4) {
                    const uint4 x = cur.v[q4];
                    const float vv[8] = {bf16_lo(x.x), bf16_hi(x.x), bf16_lo(x.y), bf16_hi(x.y),
                                         bf16_lo(x.z), bf16_hi(x.z), bf16_lo(x.w), bf16_hi(x.w)};
                    float xv[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) xv[e] = bi * vv[e] - be * (a[q4 * 8 + e] + b[q4 * 8 + e]);
                    uint4 hi, lo;
                    split8_bf16(xv, hi, lo);
                    *reinterpret_cast<uint4 *>(sm + PASS_XOP + par * 8192 + sw128_offset(i, grp * DG + 8 * q4)) = hi;
                    *reinterpret_cast<uint4 *>(sm + PASS_XOP + par * 8192 + sw128_offset(i, DS + grp * DG + 8 * q4)) =
                        lo;
                }
                fence_proxy_async_smem();
                mbar_arrive(&bar_x[par]);
            } else {
                // Q-row threads: e^{g_i} (Q S^T)_i of this chunk (into qcur), and the previous chunk's outputs
                {
                    float a[DG], b[DG];
                    tmem_ldx2<DG>(tmem + tlane + TM_D1 + grp * DG, tmem + tlane + TM_D1 + 32 + grp * DG, a, b);
#pragma unroll
                    for (int r = 0; r < DG; ++r) qcur[r] = (eg * cur.f) * (a[r] + b[r]);
                }
                if (c > 0) {
                    if (!mbar_wait(&bar_rx[par ^ 1], ph(c - 1))) ok = false;
                    tc_fence_after();
                    send_outputs(c - 1, tmem + tlane + TM_RX + 64 * (par ^ 1), ok);
                    if (!NORM) {
                        finish_outputs(c - 1, ok);
#pragma unroll
                        for (int r = 0; r < DG; ++r) qs[r] = qcur[r];
                    }
                } else {
#pragma unroll
                    for (int r = 0; r < DG; ++r) qs[r] = qcur[r];
                }
            }

            // state: S[r][d] <- e^{g_L} S[r][d] + (P X)[d][r] + (P X)[d][32 + r]
            if (!mbar_spin(&bar_px, par)) ok = false;
            tc_fence_after();
            if (!ok) break;
            {
                const float eL = __expf(gL);
                float a[DG], b[DG];
                tmem_ldx2<DG>(tmem + tlane + TM_PX + grp * DG, tmem + tlane + TM_PX + 32 + grp * DG, a, b);
#pragma unroll
                for (int e = 0; e < DG; ++e) S[e] = fmaf(eL, S[e], a[e] + b[e]);
            }
            if (MULTI && seq_end) {   // the sequence's final state; the next one starts from its initial state
                if (final_state && state_ok) {
#pragma unroll
                    for (int r = 0; r < DG; ++r) final_state[sbase + (size_t)r * D] = S[r];
                }
                const size_t nsb = sbase_of(next_c.n);
#pragma unroll
                for (int r = 0; r < DG; ++r) S[r] = next_ok ? init_state[nsb + (size_t)r * D] : 0.f;
            }
            publish_sop();
            if (NORM && !krow && c > 0) {   // the previous chunk's normalised outputs, now off the state chain
                if (!finish_outputs(c - 1, ok)) ok = false;
#pragma unroll
                for (int r = 0; r < DG; ++r) qs[r] = qcur[r];
            }
            prev_t0 = t0;
            prev_L = L;
            if (MULTI && seq_end) {
                cur_c = next_c;
                sbase = sbase_of(cur_c.n);
                state_ok = cur_c.n < sb && state_in_range(sbase);
            } else {
                ++cur_c.k;
            }
        }
        if (!ok && range_ok) fail();
        if (ok) {
            if (!krow && nchunks > 0) {
                const uint32_t lp = (nchunks - 1) & 1;
                const bool done = mbar_wait(&bar_rx[lp], ph(nchunks - 1));
                tc_fence_after();
                if (!done) fail();
                send_outputs(nchunks - 1, tmem + tlane + TM_RX + 64 * lp, done);
                if (!finish_outputs(nchunks - 1, done)) fail();
            }
            if (!MULTI && final_state && state_ok) {
#pragma unroll
                for (int r = 0; r < DG; ++r) final_state[sbase + (size_t)r * D] = S[r];
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (NORM) cluster_sync();   // no CTA leaves while a peer may still write its slots or barriers
    if (tid == 0 && started && abort_flag) raise_error(err, kErrTimeout);
    if (warp == 0) tmem_dealloc(tmem, PASS_TMEM_COLS);
}

// ---------------------------------------------------------------- host side
// The driver's tensor-map encoder, looked up once per process (a function-local static: thread-safe).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        return nullptr;
    }();
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

// Multiprocessors of device dev (cached per device; 1 if the query fails).
int multiprocessors(int dev) {
    static std::atomic<int> cached[kMaxDevices];
    const bool in_table = dev >= 0 && dev < kMaxDevices;
    if (in_table) {
        const int n = cached[dev].load(std::memory_order_relaxed);
        if (n > 0) return n;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
    if (in_table) cached[dev].store(n, std::memory_order_relaxed);
    return n;
}

// Buckets of the plain state pass.  Its CTAs take one SM each, hv * 4 of them per bucket.  One bucket per
// sequence runs short sequences in waves of CTAs that each pay the pass's fixed cost (about two chunk times)
// for one or two chunks: 1024 CTAs for eight sequences at 32 value heads.  A CTA carrying several sequences'
// chunks one after another keeps the tile pipeline full across their boundaries, at ~1.1x per chunk (the
// kernel with sequence boundaries in its loop, measured at 4K).  The candidates are: as many buckets of
// consecutive sequences (with about equal chunks) as run in one wave, or one bucket per sequence, whose CTAs
// run in waves (estimated as max(the longest sequence, all work spread over the SMs, the waves times the
// shortest)).  Measured with eight sequences at 32 value heads, one bucket is faster up to 128 tokens per
// sequence, even at 256 and slower from 512.
int pass_buckets(PassBuckets &bk, int n_seqs, const int32_t *cu_host, long nch, int hv, int sms) {
    constexpr double kCtaCost = 2.0, kMultiCost = 1.1;
    const long per_bucket = (long)hv * (D / DS);
    std::vector<long> first(n_seqs + 1, 0);   // first chunk of each sequence
    for (int n = 0; n < n_seqs; ++n) first[n + 1] = first[n] + (cu_host[n + 1] - cu_host[n] + C - 1) / C;
    // sequence starts of nb buckets: bucket b opens at the first sequence whose first chunk reaches b / nb of
    // the total (strictly after the previous bucket's first sequence); returns the buckets made
    auto split = [&](int nb, int *seq) {
        seq[0] = 0;
        if (nb == n_seqs) {   // one sequence per bucket
            for (int b = 1; b <= nb; ++b) seq[b] = b;
            return nb;
        }
        int made = 1;
        for (int b = 1; b < nb; ++b) {
            const long target = (b * nch + nb - 1) / nb;
            int n = (int)(std::lower_bound(first.begin(), first.end() - 1, target) - first.begin());
            n = std::max(n, seq[made - 1] + 1);
            if (n >= n_seqs) break;
            seq[made++] = n;
        }
        seq[made] = n_seqs;
        return made;
    };
    int seq[kMaxPassBuckets + 1];
    // one wave of buckets carrying several sequences each
    const int one_wave = (int)std::max(1L, std::min<long>(sms / per_bucket, kMaxPassBuckets));
    int best_nb = 1;
    double best_cost = -1.0;
    for (int nb = 1; nb <= std::min(n_seqs, one_wave); ++nb) {
        const int made = split(nb, seq);
        double longest = 0.0;
        for (int b = 0; b < made; ++b)
            longest = std::max(longest, (double)(first[seq[b + 1]] - first[seq[b]]) * (made < n_seqs ? kMultiCost : 1.0));
        if (best_cost < 0.0 || longest + kCtaCost < best_cost) {
            best_cost = longest + kCtaCost;
            best_nb = nb;
        }
    }
    // one bucket per sequence
    bk.per_seq = 0;
    if (n_seqs > one_wave) {
        double longest = 0.0, shortest = 0.0, work = 0.0;
        for (int n = 0; n < n_seqs; ++n) {
            const double t = (double)(first[n + 1] - first[n]) + kCtaCost;
            longest = std::max(longest, t);
            shortest = n == 0 ? t : std::min(shortest, t);
            work += t;
        }
        const double waves = (double)((n_seqs * per_bucket + sms - 1) / sms);
        const double cost = std::max({longest, work * (double)per_bucket / (double)sms, waves * shortest});
        if (cost < best_cost) {
            bk.per_seq = 1;
            return n_seqs;
        }
    }
    const int made = split(best_nb, bk.seq);
    for (int b = 0; b <= made; ++b) bk.chunk[b] = (int)first[bk.seq[b]];
    return made;
}

long total_chunks(int n_seqs, const int32_t *cu_host) {
    long nch = 0;
    for (int n = 0; n < n_seqs; ++n) nch += (cu_host[n + 1] - cu_host[n] + C - 1) / C;
    return nch;
}

}  // namespace

int plan_state_pass(int n_seqs, const int32_t *cu_host, int hv, int sms, int *first_seq, int capacity) {
    PassBuckets bk;
    const int nb = pass_buckets(bk, n_seqs, cu_host, total_chunks(n_seqs, cu_host), hv, sms);
    if (capacity < nb + 1) return -1;
    for (int b = 0; b <= nb; ++b) first_seq[b] = bk.per_seq ? b : bk.seq[b];
    return nb;
}

size_t chunked_workspace_bytes(int n_seqs, const int32_t *cu_host, int hv, int d) {
    if (d != D) return 0;
    const long nch = total_chunks(n_seqs, cu_host);
    return (size_t)nch * hv * (2 * kPTile + 2 * kRTile + kNormBytes);
}

cudaError_t launch_chunked_prefill(const PrefillProblem &p, int phases) {
    if (p.d != D) return cudaErrorNotSupported;
    const long nch = total_chunks(p.n_seqs, p.cu_seqlens_host);
    if (nch > 0x7fffffffL / (p.hv * D)) return cudaErrorInvalidValue;
    // workspace: P_hi | P_lo  [nch][hv][D][C]  then R_hi | R_lo  [nch][hv][C][C]  (bf16), then the q/k
    // preparation factors [nch][hv][2 C] (fp32: f_k of the chunk's 64 k rows, then f_q of its q rows)
    __nv_bfloat16 *phi = static_cast<__nv_bfloat16 *>(p.workspace);
    __nv_bfloat16 *plo = phi + (size_t)nch * p.hv * D * C;
    __nv_bfloat16 *rhi = plo + (size_t)nch * p.hv * D * C;
    __nv_bfloat16 *rlo = rhi + (size_t)nch * p.hv * C * C;
    float *norms = reinterpret_cast<float *>(rlo + (size_t)nch * p.hv * C * C);

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static std::atomic<bool> attrs_set[kMaxDevices];
    const bool cached = dev >= 0 && dev < kMaxDevices;
    if (!cached || !attrs_set[dev].load(std::memory_order_acquire)) {
        const void *prep[] = {(const void *)chunk_prep_kernel<false, false>, (const void *)chunk_prep_kernel<true, false>,
                              (const void *)chunk_prep_kernel<false, true>, (const void *)chunk_prep_kernel<true, true>};
        const void *pass[] = {(const void *)state_pass_kernel<false, false, false>,
                              (const void *)state_pass_kernel<true, false, false>,
                              (const void *)state_pass_kernel<false, true, false>,
                              (const void *)state_pass_kernel<true, true, false>,
                              (const void *)state_pass_kernel<false, false, true>,
                              (const void *)state_pass_kernel<true, false, true>,
                              (const void *)state_pass_kernel<false, true, true>,
                              (const void *)state_pass_kernel<true, true, true>};
        for (const void *f : prep)
            if (e == cudaSuccess) e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, PREP_SMEM);
        for (const void *f : pass)
            if (e == cudaSuccess) e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, PASS_SMEM);
        if (e != cudaSuccess) return e;
        if (cached) attrs_set[dev].store(true, std::memory_order_release);
    }

    CUtensorMap qmap{}, kmap{}, phmap{}, plmap{}, rhmap{}, rlmap{};
    if (p.total_tokens > 0 && nch > 0) {
        const uint64_t T = (uint64_t)p.total_tokens, QK = (uint64_t)p.hk * D;
        const uint64_t rows_p = (uint64_t)nch * p.hv * D, rows_r = (uint64_t)nch * p.hv * C;
        if (!make_map(&qmap, p.q, T, QK, QK, 64) || !make_map(&kmap, p.k, T, QK, QK, 64) ||
            !make_map(&phmap, phi, rows_p, C, C, 128) || !make_map(&plmap, plo, rows_p, C, C, 128) ||
            !make_map(&rhmap, rhi, rows_r, C, C, 64) || !make_map(&rlmap, rlo, rows_r, C, C, 64))
            return cudaErrorInvalidValue;
    }

    const bool prep_qk = p.qk_norm || p.q_scale != 1.f, gate = p.gate_c != nullptr;
    if ((phases & 1) && nch > 0) {
        dim3 grid((unsigned)(nch * p.hv));
        auto prep = prep_qk ? (gate ? chunk_prep_kernel<true, true> : chunk_prep_kernel<true, false>)
                            : (gate ? chunk_prep_kernel<false, true> : chunk_prep_kernel<false, false>);
        prep<<<grid, kPrepThreads, PREP_SMEM, p.stream>>>(qmap, kmap, phmap, plmap, rhmap, rlmap, p.log_alpha,
                                                           p.beta, p.cu_seqlens, p.n_seqs, p.total_tokens, p.hk, p.hv,
                                                           norms, p.qk_norm, p.q_scale, p.gate_c, p.gate_b, p.err);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (phases & 2) {
        const float *nrm = p.qk_norm ? norms : nullptr;
        PassBuckets bk;
        const int nb = pass_buckets(bk, p.n_seqs, p.cu_seqlens_host, nch, p.hv, multiprocessors(dev));
        const bool multi = nb < p.n_seqs;   // some bucket carries more than one sequence
        const bool norm = p.norm_w != nullptr;
        using PassFn = decltype(&state_pass_kernel<false, false, false>);
        const PassFn table[8] = {state_pass_kernel<false, false, false>, state_pass_kernel<true, false, false>,
                                 state_pass_kernel<false, true, false>,  state_pass_kernel<true, true, false>,
                                 state_pass_kernel<false, false, true>,  state_pass_kernel<true, false, true>,
                                 state_pass_kernel<false, true, true>,   state_pass_kernel<true, true, true>};
        const PassFn pass = table[(gate ? 1 : 0) + (multi ? 2 : 0) + (norm ? 4 : 0)];
        // With the output normalisation the four slice CTAs of a (bucket, head) form one cluster.  Right after
        // this call's preparation the pass is its programmatic dependent: its CTAs may start on SMs the
        // preparation has left, run their prologue and first products (which read only the inputs, complete
        // since before the preparation started), and wait for the preparation before reading the workspace.
        // Launched alone it follows the stream as usual.
        cudaLaunchAttribute attr[2];
        int nattr = 0;
        if (norm) {
            attr[nattr].id = cudaLaunchAttributeClusterDimension;
            attr[nattr].val.clusterDim.x = D / DS;
            attr[nattr].val.clusterDim.y = 1;
            attr[nattr].val.clusterDim.z = 1;
            ++nattr;
        }
        if ((phases & 1) && nch > 0) {
            attr[nattr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[nattr].val.programmaticStreamSerializationAllowed = 1;
            ++nattr;
        }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(nb * p.hv * (D / DS)));
        cfg.blockDim = dim3(kWsThreads);
        cfg.dynamicSmemBytes = PASS_SMEM;
        cfg.stream = p.stream;
        cfg.attrs = attr;
        cfg.numAttrs = nattr;
        e = cudaLaunchKernelEx(&cfg, pass, qmap, kmap, phmap, plmap, rhmap, rlmap, p.v, nrm, p.q_scale, p.log_alpha,
                               p.beta, p.init_state, p.cu_seqlens, p.n_seqs, p.total_tokens, (int)nch, p.hk, p.hv,
                               p.out, p.out_f32, p.final_state, p.gate_c, p.gate_b, p.err, bk, p.norm_w,
                               p.norm_eps);
        if (e != cudaSuccess || (e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace gdn
