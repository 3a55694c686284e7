// Chunked backward pass of the ungated recurrence (D_k = D_v = 128), fp32 on
// CUDA cores.
//
// The extended sequence of every (batch, head) is cut into chunks of ct
// whole tokens (R = ct n_h <= 32 rows, padded to 32 with zero rows, which
// are exact no-ops), as in the forward. Per chunk, with S0 the state at its
// start (OSDN paper, App.A.2, write key = read key; DeltaProduct paper,
// Sec.5.1, readout at each token's last row):
//   A = I + tril(diag(beta) K K^T, -1),  T = A^{-1}
//   W = T diag(beta) K,  U = T diag(beta) V,  U' = U - W S0
//   S1 = S0 + K^T U',   O = Q S0 + P U',  P = (Q K^T) masked to s <= last(t)
// and, given dO and dS1 (the gradient at the chunk's end), by the chain rule
//   dU' = P^T dO + K dS1,   dS0 = dS1 + Q^T dO - W^T dU'          (chain)
//   dQ  = dO S0^T + dP K,   dP = (dO U'^T) masked
//   dK  = dP^T Q + U' dS1^T + diag(beta) T^T dW + (B dG) K + (B dG)^T K
//   dV  = diag(beta) T^T dU',  dW = -dU' S0^T,  B = diag(beta)
//   dbeta = rowsum(K o T^T dW) + rowsum(V o T^T dU') + rowsum(dG o K K^T)
//   dT = dW (B K)^T + dU' (B V)^T,  dG = strictly lower part of -T^T dT T^T
// Four launches:
//   cb_prep    every chunk at once: T, W, U, P, K K^T and fp32 K, Q into its
//              record;
//   cb_chains  per (b,h) and 64 value columns, chunk by chunk, two
//              independent CTAs: the forward chain (S <- S + K^T (U - W S))
//              stores S0 and U' of every chunk; the reverse chain (the
//              transposed recurrence above, from the last chunk) stores dS1
//              and dU' of every chunk and dh0. The next chunk's operands are
//              copied in (cp.async) while the current one is processed;
//   cb_grad_s  every chunk at once, the products with the 128 x 128
//              boundary states (60% of the per-chunk arithmetic):
//              dq <- dO S0^T, dk <- U' dS1^T, dW = -dU' S0^T and dP; each
//              thread holds quarter rows of two rows of S0, then of dS1, in
//              registers;
//   cb_grad_r  every chunk at once, the rest: dq += dP K, dk += ..., dv,
//              dbeta.
// The chains carry the only sequential dependency, as 32 x 128 x 128
// products per chunk instead of a matrix-vector product per sub-step.
#include "internal.h"

namespace dp {
namespace {

constexpr int kD = 128;
constexpr int kC = 32;     // rows per chunk (padded)
constexpr int kQ = 16;     // token rows per chunk (padded)
constexpr int kS = 132;    // fp32 row stride of [.][128] tiles: float4-aligned, rows spread over the banks
constexpr int kL = kC + 1; // row stride of [.][32] tiles

// record of one chunk (fp32): W [32][128] | U [32][128] | T [32][32] |
// P [16][32] | K K^T [32][32] | K [32][128] | Q [16][128] (K and Q as fp32
// for the chains), and for gated problems: Kd [32][128] (the keys decayed to
// the chunk's end, (Gamma_C / Gamma_r) k_r, for the chains) | Pr [16][32]
// (Q K^T masked, before the decay; P holds it decayed) | E [32][32]
// (Gamma_r / Gamma_s, s <= r) | Gamma [32] | ratio [32] (Gamma_C /
// Gamma_r) | lg [32] (the rows' log gates) | aux [4] (<dS1, S0>). After the
// chains, cb_grad_s overwrites W with dW and P with dP (before the decay),
// which cb_grad_r reads.
constexpr size_t kRecW = 0, kRecU = kC * kD, kRecT = 2 * kC * kD, kRecP = kRecT + kC * kC;
constexpr size_t kRecKK = kRecP + kQ * kC, kRecK = kRecKK + kC * kC, kRecQ = kRecK + kC * kD;
constexpr size_t kRecKd = kRecQ + kQ * kD, kRecPr = kRecKd + kC * kD, kRecE = kRecPr + kQ * kC;
constexpr size_t kRecGm = kRecE + kC * kC, kRecRt = kRecGm + kC, kRecLg = kRecRt + kC, kRecAux = kRecLg + kC;
constexpr size_t kRecFloats = kRecAux + 4;
// log gates below this are taken as it (a gate of 1.8e-35: the forward's
// chunk path clamps the same way)
constexpr float kMinLogGate = -80.f;
constexpr size_t kStateFloats = (size_t)kD * kD;   // S0 or dS1 of one chunk
constexpr size_t kRowsFloats = (size_t)kC * kD;    // U' or dU' of one chunk

struct CbArgs {
    int B, T, H, nh, ct, nc;            // nc: chunks per (sequence, head) at the longest length
    const int *cu;                      // packed sequences: int32 [B+1] token offsets (NULL: dense)
    int max_T;                          // longest sequence (T for dense calls)
    const void *q, *k, *v, *beta;
    const float *h0;
    const void *d_o;
    const float *dh_final;
    float *dq, *dk, *dv, *dbeta, *dh0;
    float *rec, *S0, *dS1, *Up, *dUp;   // workspace areas, [B*H*nc] chunks each
    const void *g;                      // gates [B,T,H] (gated instantiations)
    float *dg;
    uint32_t *status;
};

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

// bf16 -> fp32 is exact: the bf16 bits are the high half of the fp32 word
__device__ __forceinline__ void unpack8(const uint4 u, float *x)
{
    x[0] = __uint_as_float(u.x << 16), x[1] = __uint_as_float(u.x & 0xffff0000u);
    x[2] = __uint_as_float(u.y << 16), x[3] = __uint_as_float(u.y & 0xffff0000u);
    x[4] = __uint_as_float(u.z << 16), x[5] = __uint_as_float(u.z & 0xffff0000u);
    x[6] = __uint_as_float(u.w << 16), x[7] = __uint_as_float(u.w & 0xffff0000u);
}
// 8 consecutive elements (16-byte aligned) as fp32, from global memory
// (read-only during the kernel)
__device__ __forceinline__ void ldg8(const __nv_bfloat16 *p, float *x) { unpack8(__ldg((const uint4 *)p), x); }
__device__ __forceinline__ void ldg8(const float *p, float *x)
{
    const float4 a = __ldg((const float4 *)p), b = __ldg((const float4 *)p + 1);
    x[0] = a.x, x[1] = a.y, x[2] = a.z, x[3] = a.w, x[4] = b.x, x[5] = b.y, x[6] = b.z, x[7] = b.w;
}
__device__ __forceinline__ float4 ld4(const float *p) { return *(const float4 *)p; }
__device__ __forceinline__ void st4(float *p, float4 v) { *(float4 *)p = v; }
__device__ __forceinline__ float dot4(float4 a, float4 b, float acc)
{
    return fmaf(a.w, b.w, fmaf(a.z, b.z, fmaf(a.y, b.y, fmaf(a.x, b.x, acc))));
}
__device__ __forceinline__ float4 axpy4(float s, float4 x, float4 y)
{
    return make_float4(fmaf(s, x.x, y.x), fmaf(s, x.y, y.y), fmaf(s, x.z, y.z), fmaf(s, x.w, y.w));
}

__device__ __forceinline__ void cp_async16(void *dst, const void *src)
{
    const unsigned s = (unsigned)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }

// The chunk's rows: row r (< 32) = token c*ct + r / nh of its sequence, key
// r % nh; valid while r < R. Packed calls: the sequence's token range from
// the offsets (a sequence that breaks their rules has no tokens).
struct ChunkRows {
    size_t tok0;   // (sequence, first token of the chunk, h) row index of the [.,T,H] layouts
    int nt;        // tokens of the chunk (<= ct; 0 past the sequence's end)
    int R;         // valid extended rows (nt * nh)
    int len;       // tokens of the sequence
    bool ok;       // the sequence's offsets keep the rules
};
__device__ __forceinline__ ChunkRows chunk_rows(const CbArgs &a, int bh, int c)
{
    const int b = bh / a.H, h = bh - b * a.H, t0 = c * a.ct;
    const SeqRange sr = seq_range(a.cu, b, a.B, a.T, a.max_T);
    ChunkRows cr;
    cr.tok0 = ((size_t)sr.b_map * a.T + sr.t0 + t0) * a.H + h;
    cr.nt = max(0, min(a.ct, sr.len - t0));
    cr.R = cr.nt * a.nh;
    cr.len = sr.len;
    cr.ok = sr.ok;
    return cr;
}
// chunks of the (sequence, head) of CTA row bh
__device__ __forceinline__ int seq_chunks(const CbArgs &a, int bh)
{
    return (chunk_rows(a, bh, 0).len + a.ct - 1) / a.ct;
}
__device__ __forceinline__ size_t key_row(const CbArgs &a, const ChunkRows &cr, int r)
{
    const int t = r / a.nh, j = r - t * a.nh;
    return (cr.tok0 + (size_t)t * a.H) * a.nh + j;
}
__device__ __forceinline__ size_t token_row(const CbArgs &a, const ChunkRows &cr, int t)
{
    return cr.tok0 + (size_t)t * a.H;
}

// fp32 [rows][kS] tile of the chunk's key rows (kKeys) or token rows of a
// [.,128] tensor, zero past the valid rows; every thread takes part.
template <bool kKeys, int kRows, typename TIn, int kStride = kS>
__device__ __forceinline__ void stage_f32(const CbArgs &a, const ChunkRows &cr, const TIn *src, float *dst)
{
    for (int i = threadIdx.x; i < kRows * 16; i += blockDim.x) {
        const int r = i >> 4, e = (i & 15) * 8;
        float x[8];
        if (r < (kKeys ? cr.R : cr.nt)) {
            ldg8(src + (kKeys ? key_row(a, cr, r) : token_row(a, cr, r)) * kD + e, x);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) x[j] = 0.f;
        }
        st4(dst + r * kStride + e, make_float4(x[0], x[1], x[2], x[3]));
        st4(dst + r * kStride + e + 4, make_float4(x[4], x[5], x[6], x[7]));
    }
}
template <typename TIn>
__device__ __forceinline__ void stage_betas(const CbArgs &a, const ChunkRows &cr, float *be)
{
    const TIn *beta = (const TIn *)a.beta;
    for (int r = threadIdx.x; r < kC; r += blockDim.x) be[r] = r < cr.R ? to_f(beta[key_row(a, cr, r)]) : 0.f;
}

// ------------------------------------------------------------------ 1. prep
constexpr int kPrepThreads = 256;
constexpr int kPrepSmemFloats = 2 * kC * kS + kQ * kS + 3 * kC * kL + 4 * kC;

// Gated chunks: the rows' log gates lg_r (log g_t at a token's first row,
// clamped below at kMinLogGate; 0 elsewhere and on padding rows) and every
// decay factor as exp of a directly accumulated range sum of them (never a
// difference of prefix sums, so a zero gate cuts the decay exactly):
// E[r][s] = exp(sum_{s < x <= r} lg_x), Gamma_r = exp(sum_{x <= r} lg_x),
// ratio_r = Gamma_C / Gamma_r = exp(sum_{r < x < 32} lg_x). A gate < 0 or
// NaN records a device error.
template <typename TIn>
__device__ __forceinline__ void prep_gates(const CbArgs &a, const ChunkRows &cr, float *lg, float *Gm, float *Rt,
                                           float *E, float *rec)
{
    const int tid = threadIdx.x;
    if (tid < kC) {
        float x = 0.f;
        if (tid < cr.R && tid % a.nh == 0) {
            const float gv = to_f(((const TIn *)a.g)[token_row(a, cr, tid / a.nh)]);
            if (!(gv >= 0.f)) report_bad_sequence(a.status);
            x = gv > 0.f ? fmaxf(logf(gv), kMinLogGate) : kMinLogGate;
        }
        lg[tid] = x;
        rec[kRecLg + tid] = x;
    }
    __syncthreads();
    for (int i = tid; i < kC * kC; i += blockDim.x) {
        const int r = i >> 5, s2 = i & 31;
        float e = 0.f;
        if (s2 <= r) {
            float acc = 0.f;   // sum_{s < x <= r} lg_x
            for (int x2 = s2 + 1; x2 <= r; ++x2) acc += lg[x2];
            e = expf(acc);
        }
        E[r * kL + s2] = e;
        rec[kRecE + i] = e;
    }
    if (tid < kC) {
        const int r = tid;
        float sg = 0.f, sr = 0.f;   // sum_{x <= r} lg_x, sum_{r < x < 32} lg_x
        for (int x2 = 0; x2 <= r; ++x2) sg += lg[x2];
        for (int x2 = r + 1; x2 < kC; ++x2) sr += lg[x2];
        const float gm = expf(sg), rt = expf(sr);
        Gm[r] = gm, Rt[r] = rt;
        rec[kRecGm + r] = gm, rec[kRecRt + r] = rt;
    }
}

template <typename TIn, bool kG>
__global__ void __launch_bounds__(kPrepThreads) cb_prep(const CbArgs a)
{
    extern __shared__ float4 sm_prep[];
    float *Ks = (float *)sm_prep, *Vs = Ks + kC * kS, *Qs = Vs + kC * kS;
    float *KK = Qs + kQ * kS, *Ts = KK + kC * kL, *E = Ts + kC * kL, *be = E + kC * kL;
    float *lg = be + kC, *Gm = lg + kC, *Rt = Gm + kC;
    const int ci = blockIdx.x, bh = ci / a.nc, c = ci - bh * a.nc;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const ChunkRows cr = chunk_rows(a, bh, c);
    if (!cr.ok && c == 0 && threadIdx.x == 0) report_bad_sequence(a.status);
    if (cr.nt == 0) return;   // past the sequence's end (packed calls)
    float *rec = a.rec + (size_t)ci * kRecFloats;
    stage_f32<true, kC, TIn>(a, cr, (const TIn *)a.k, Ks);
    stage_f32<true, kC, TIn>(a, cr, (const TIn *)a.v, Vs);
    stage_f32<false, kQ, TIn>(a, cr, (const TIn *)a.q, Qs);
    stage_betas<TIn>(a, cr, be);
    if (kG) prep_gates<TIn>(a, cr, lg, Gm, Rt, E, rec);
    __syncthreads();
    // fp32 K and Q (zero padding rows included) for the chains; gated: Kd
    for (int i = threadIdx.x; i < (kC + kQ) * kD / 4; i += kPrepThreads) {
        const int r = i >> 5, e = (i & 31) * 4;
        if (r < kC) {
            const float4 k4 = ld4(Ks + r * kS + e);
            st4(rec + kRecK + r * kD + e, k4);
            if (kG) {
                const float f = Rt[r];
                st4(rec + kRecKd + r * kD + e, make_float4(f * k4.x, f * k4.y, f * k4.z, f * k4.w));
            }
        } else {
            st4(rec + kRecQ + (r - kC) * kD + e, ld4(Qs + (r - kC) * kS + e));
        }
    }
    // K K^T rows w, w+8, w+16, w+24 and P rows w, w+8; lane = column s
    {
        float acc[6] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        const float *ks = Ks + lane * kS;
#pragma unroll 4
        for (int d = 0; d < kD; d += 4) {
            const float4 y = ld4(ks + d);
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[i] = dot4(ld4(Ks + (w + 8 * i) * kS + d), y, acc[i]);
#pragma unroll
            for (int i = 0; i < 2; ++i) acc[4 + i] = dot4(ld4(Qs + (w + 8 * i) * kS + d), y, acc[4 + i]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = w + 8 * i;
            rec[kRecKK + r * kC + lane] = acc[i];
            // G = B (K K^T o E), strictly lower: the substitution's operand
            KK[r * kL + lane] = lane < r ? be[r] * acc[i] * (kG ? E[r * kL + lane] : 1.f) : 0.f;
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int t = w + 8 * i, last = t * a.nh + a.nh - 1;
            const float p = lane <= last ? acc[4 + i] : 0.f;
            if (kG) {
                rec[kRecPr + t * kC + lane] = p;
                rec[kRecP + t * kC + lane] = last < kC ? p * E[last * kL + lane] : 0.f;
            } else {
                rec[kRecP + t * kC + lane] = p;
            }
        }
    }
    __syncthreads();
    // T = (I + G)^{-1}: forward substitution, lane = column
    if (w == 0) {
        const int s = lane;
        for (int r = 0; r < kC; ++r) {
            float x = (r == s) ? 1.f : 0.f;
            for (int m = s; m < r; ++m) x = fmaf(-KK[r * kL + m], Ts[m * kL + s], x);
            Ts[r * kL + s] = x;
            rec[kRecT + r * kC + s] = x;
        }
    }
    __syncthreads();
    // W = T diag(beta Gamma) K, U = T diag(beta) V: warp w rows 4w .. 4w+3, lane = 4 columns
    {
        const int d = lane * 4, r0 = 4 * w;
        float4 wa[4], ua[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) wa[i] = ua[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int m = 0; m <= r0 + 3; ++m) {   // T is lower triangular
            const float4 k4 = ld4(Ks + m * kS + d), v4 = ld4(Vs + m * kS + d);
            const float bm = be[m], bg = kG ? bm * Gm[m] : bm;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float t = Ts[(r0 + i) * kL + m];
                wa[i] = axpy4(t * bg, k4, wa[i]);
                ua[i] = axpy4(t * bm, v4, ua[i]);
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            st4(rec + kRecW + (r0 + i) * kD + d, wa[i]);
            st4(rec + kRecU + (r0 + i) * kD + d, ua[i]);
        }
    }
}

// ------------------------------------------------------------------ 2. chains
// CTA: (b,h), 64 value columns (blockIdx.y) and the direction (blockIdx.z),
// 256 threads, one CTA per SM. Every operand a thread reads from shared
// memory feeds several of its FMAs (a 128-bit shared load costs four
// wavefronts even when all lanes read the same address):
//   state owner: warp w, lane = (ro, cq): rows 16w + 8ro .. + 7, columns
//     4cq .. 4cq + 3 (8 x 4 registers); per chunk row r it reads 8 key (W)
//     values and 4 U' (dU') values for 32 FMAs;
//   U' (dU'): thread (kh, rq, cq): rows 4rq .. 4rq + 3, columns 4cq .. +3,
//     half kh of the 128-term contraction (4 x 4 FMAs per 8 values read);
//     the two halves meet in shared memory.
constexpr int kChainThreads = 256;
constexpr int kCols = 64;          // value columns per chain CTA
constexpr int kSS = kCols + 4;     // row stride of the state and U' tiles

struct FwdStage {   // one chunk's operands of the forward chain (fp32; Gamma for gated problems)
    static constexpr size_t kW = (size_t)kC * kD * 4, kK = (size_t)kC * kD * 4, kU = (size_t)kC * kCols * 4;
    static constexpr size_t kG = (size_t)kC * 4;
    static constexpr size_t kBytes = kW + kK + kU + kG;
};
template <typename TDo>
struct BwdStage {   // ... and of the reverse chain
    static constexpr size_t kW = (size_t)kC * kD * 4, kK = (size_t)kC * kD * 4, kQb = (size_t)kQ * kD * 4;
    static constexpr size_t kO = (size_t)kQ * kCols * sizeof(TDo), kP = (size_t)kQ * kC * 4;
    static constexpr size_t kG = (size_t)kC * 4;
    static constexpr size_t kBytes = kW + kK + kQb + kO + kP + kG;
};
// state tile [128][kSS], U' tile [32][kSS], partial sums [128 threads][16]
constexpr size_t kChainShared = (size_t)(kD + kC) * kSS * 4 + (size_t)128 * 16 * 4;
template <typename TDo>
constexpr size_t chain_smem_bytes()
{
    const size_t f = 2 * FwdStage::kBytes, b = 2 * BwdStage<TDo>::kBytes;
    return (f > b ? f : b) + kChainShared;
}

// cp.async of the chunk's token rows of d_o, columns [col0, col0 + kCols), zero rows past nt
template <typename T>
__device__ __forceinline__ void copy_do_rows(const CbArgs &a, const ChunkRows &cr, const T *src, int col0, T *dst)
{
    constexpr int kPer = 16 / sizeof(T), kPerRow = kCols / kPer;
    for (int i = threadIdx.x; i < kQ * kPerRow; i += kChainThreads) {
        const int t = i / kPerRow, e = (i - t * kPerRow) * kPer;
        if (t < cr.nt) cp_async16(dst + t * kCols + e, src + token_row(a, cr, t) * kD + col0 + e);
        else *(uint4 *)(dst + t * kCols + e) = make_uint4(0u, 0u, 0u, 0u);
    }
}
__device__ __forceinline__ void copy_floats(const float *src, float *dst, int n)
{
    for (int i = threadIdx.x * 4; i < n; i += kChainThreads * 4) cp_async16(dst + i, src + i);
}
// 4 consecutive d_o values (8- or 16-byte aligned) as fp32
__device__ __forceinline__ float4 ld4o(const float *p) { return ld4(p); }
__device__ __forceinline__ float4 ld4o(const __nv_bfloat16 *p)
{
    const uint2 u = *(const uint2 *)p;
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u), __uint_as_float(u.y << 16),
                       __uint_as_float(u.y & 0xffff0000u));
}
__device__ __forceinline__ float f4(const float4 v, int j) { return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w; }

// Thread roles of a chain CTA.
struct ChainLanes {
    int sr0, sc0;        // state block: rows sr0 .. sr0 + 7, columns sc0 .. sc0 + 3
    int kh, ur0, uc0;    // U' block: contraction half, rows ur0 .. + 3, columns uc0 .. + 3
    __device__ ChainLanes()
    {
        const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
        sr0 = 16 * w + 8 * (lane >> 4);
        sc0 = 4 * (lane & 15);
        kh = tid >> 7;
        ur0 = 4 * ((tid >> 4) & 7);
        uc0 = 4 * (tid & 15);
    }
};

// the state block into the state tile and global memory (row-major, columns cg + ...)
__device__ __forceinline__ void put_state(const float (*S)[4], float *tile, float *g, const ChainLanes &L, int cg)
{
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float4 v = make_float4(S[i][0], S[i][1], S[i][2], S[i][3]);
        st4(tile + (L.sr0 + i) * kSS + L.sc0, v);
        st4(g + (L.sr0 + i) * kD + cg + L.sc0, v);
    }
}
// acc[i][j] = sum over k in half kh of X[ur0 + i][k] St[k][uc0 + j]
__device__ __forceinline__ void rows_times_state(const float *X, const float *St, const ChainLanes &L,
                                                 float (*acc)[4])
{
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    const int k0 = 64 * L.kh;
#pragma unroll 2
    for (int k = k0; k < k0 + 64; k += 4) {
        float4 x[4], s[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) x[i] = ld4(X + (L.ur0 + i) * kD + k);
#pragma unroll
        for (int q = 0; q < 4; ++q) s[q] = ld4(St + (k + q) * kSS + L.uc0);
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float xv = f4(x[i], q);
                acc[i][0] = fmaf(xv, s[q].x, acc[i][0]);
                acc[i][1] = fmaf(xv, s[q].y, acc[i][1]);
                acc[i][2] = fmaf(xv, s[q].z, acc[i][2]);
                acc[i][3] = fmaf(xv, s[q].w, acc[i][3]);
            }
    }
}
// the second half's partial sums join the first half's (two barriers inside)
__device__ __forceinline__ void join_halves(float (*acc)[4], float *red, const ChainLanes &L)
{
    float *slot = red + (threadIdx.x & 127) * 16;
    if (L.kh == 1) {
#pragma unroll
        for (int i = 0; i < 4; ++i) st4(slot + 4 * i, make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]));
    }
    __syncthreads();
    if (L.kh == 0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 v = ld4(slot + 4 * i);
            acc[i][0] += v.x, acc[i][1] += v.y, acc[i][2] += v.z, acc[i][3] += v.w;
        }
    }
}
// S[i][j] += sgn * sum_r X[r][sr0 + i] Y[r][sc0 + j], r < kN (X stride kD, Y stride kSS)
template <int kN>
__device__ __forceinline__ void update_state(float (*S)[4], const float *X, const float *Y, const ChainLanes &L,
                                             float sgn)
{
#pragma unroll 4
    for (int r = 0; r < kN; ++r) {
        const float4 x0 = ld4(X + r * kD + L.sr0), x1 = ld4(X + r * kD + L.sr0 + 4);
        const float4 y = ld4(Y + r * kSS + L.sc0);
        const float yv[4] = {sgn * y.x, sgn * y.y, sgn * y.z, sgn * y.w};
        const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) S[i][j] = fmaf(xv[i], yv[j], S[i][j]);
    }
}

template <bool kGt>
__device__ __forceinline__ void fwd_chain(const CbArgs &a, char *smem)
{
    using St = FwdStage;
    float *Ssm = (float *)(smem + 2 * St::kBytes), *Usm = Ssm + kD * kSS, *red = Usm + kC * kSS;
    const int bh = blockIdx.x, cg = blockIdx.y * kCols;
    const ChainLanes L;
    auto prefetch = [&](int c) {
        char *base = smem + (c & 1) * St::kBytes;
        const float *rec = a.rec + ((size_t)bh * a.nc + c) * kRecFloats;
        copy_floats(rec + kRecW, (float *)base, kC * kD);
        copy_floats(rec + (kGt ? kRecKd : kRecK), (float *)(base + St::kW), kC * kD);
        if (kGt) copy_floats(rec + kRecGm, (float *)(base + St::kW + St::kK + St::kU), kC);
        float *Ud = (float *)(base + St::kW + St::kK);
        for (int i = threadIdx.x; i < kC * kCols / 4; i += kChainThreads) {
            const int r = i / (kCols / 4), e = (i % (kCols / 4)) * 4;
            cp_async16(Ud + r * kCols + e, rec + kRecU + r * kD + cg + e);
        }
        cp_async_commit();
    };
    float S[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
            S[i][j] = a.h0 ? a.h0[((size_t)bh * kD + L.sr0 + i) * kD + cg + L.sc0 + j] : 0.f;
    const int ncs = seq_chunks(a, bh);
    if (ncs > 0) prefetch(0);
    for (int c = 0; c < ncs; ++c) {
        const size_t ci = (size_t)bh * a.nc + c;
        put_state(S, Ssm, a.S0 + ci * kStateFloats, L, cg);
        cp_async_wait_all();
        __syncthreads();   // chunk c's stage and the state tile are complete; chunk c-1's stage is free
        if (c + 1 < ncs) prefetch(c + 1);
        const char *base = smem + (c & 1) * St::kBytes;
        const float *Wc = (const float *)base, *Kc = (const float *)(base + St::kW);
        const float *Uc = (const float *)(base + St::kW + St::kK);
        // U' = U - W S
        float acc[4][4];
        rows_times_state(Wc, Ssm, L, acc);
        join_halves(acc, red, L);
        if (L.kh == 0) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float4 u = ld4(Uc + (L.ur0 + i) * kCols + L.uc0);
                const float4 v = make_float4(u.x - acc[i][0], u.y - acc[i][1], u.z - acc[i][2], u.w - acc[i][3]);
                st4(Usm + (L.ur0 + i) * kSS + L.uc0, v);
                st4(a.Up + ci * kRowsFloats + (L.ur0 + i) * kD + cg + L.uc0, v);
            }
        }
        __syncthreads();
        if (kGt) {   // S <- Gamma_C S + Kd^T U'
            const float gc = ((const float *)(base + St::kW + St::kK + St::kU))[kC - 1];
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) S[i][j] *= gc;
        }
        update_state<kC>(S, Kc, Usm, L, 1.f);   // S += K^T U'
    }
}

template <typename TDo, bool kGt>
__device__ __forceinline__ void bwd_chain(const CbArgs &a, char *smem)
{
    using St = BwdStage<TDo>;
    float *dSsm = (float *)(smem + 2 * St::kBytes), *dUsm = dSsm + kD * kSS, *red = dUsm + kC * kSS;
    const int bh = blockIdx.x, cg = blockIdx.y * kCols;
    const ChainLanes L;
    auto prefetch = [&](int c) {
        char *base = smem + (c & 1) * St::kBytes;
        const float *rec = a.rec + ((size_t)bh * a.nc + c) * kRecFloats;
        copy_floats(rec + kRecW, (float *)base, kC * kD);
        copy_floats(rec + (kGt ? kRecKd : kRecK), (float *)(base + St::kW), kC * kD);
        copy_floats(rec + kRecQ, (float *)(base + St::kW + St::kK), kQ * kD);
        if (kGt) copy_floats(rec + kRecGm, (float *)(base + St::kW + St::kK + St::kQb + St::kO + St::kP), kC);
        copy_do_rows<TDo>(a, chunk_rows(a, bh, c), (const TDo *)a.d_o, cg,
                          (TDo *)(base + St::kW + St::kK + St::kQb));
        copy_floats(rec + kRecP, (float *)(base + St::kW + St::kK + St::kQb + St::kO), kQ * kC);
        cp_async_commit();
    };
    float dS[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
            dS[i][j] = a.dh_final ? a.dh_final[((size_t)bh * kD + L.sr0 + i) * kD + cg + L.sc0 + j] : 0.f;
    const int ncs = seq_chunks(a, bh);
    if (ncs > 0) prefetch(ncs - 1);
    for (int c = ncs - 1; c >= 0; --c) {
        const size_t ci = (size_t)bh * a.nc + c;
        put_state(dS, dSsm, a.dS1 + ci * kStateFloats, L, cg);
        cp_async_wait_all();
        __syncthreads();
        if (c > 0) prefetch(c - 1);
        const char *base = smem + (c & 1) * St::kBytes;
        const float *Wc = (const float *)base, *Kc = (const float *)(base + St::kW);
        const float *Qc = (const float *)(base + St::kW + St::kK);
        const TDo *Oc = (const TDo *)(base + St::kW + St::kK + St::kQb);
        const float *Pc = (const float *)(base + St::kW + St::kK + St::kQb + St::kO);
        // dU' = K dS1 + P^T dO
        float g[4][4];
        rows_times_state(Kc, dSsm, L, g);
        if (L.kh == 1) {   // the second half also takes P^T dO
#pragma unroll 4
            for (int t = 0; t < kQ; ++t) {
                const float4 p = ld4(Pc + t * kC + L.ur0), o = ld4o(Oc + t * kCols + L.uc0);
                const float pv[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    g[i][0] = fmaf(pv[i], o.x, g[i][0]);
                    g[i][1] = fmaf(pv[i], o.y, g[i][1]);
                    g[i][2] = fmaf(pv[i], o.z, g[i][2]);
                    g[i][3] = fmaf(pv[i], o.w, g[i][3]);
                }
            }
        }
        join_halves(g, red, L);
        if (L.kh == 0) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float4 v = make_float4(g[i][0], g[i][1], g[i][2], g[i][3]);
                st4(dUsm + (L.ur0 + i) * kSS + L.uc0, v);
                st4(a.dUp + ci * kRowsFloats + (L.ur0 + i) * kD + cg + L.uc0, v);
            }
        }
        __syncthreads();
        // dS0 = Gamma_C dS1 + Q^T diag(Gamma_last(t)) dO - W^T dU'
        const float *Gc = (const float *)(base + St::kW + St::kK + St::kQb + St::kO + St::kP);
        if (kGt) {
            const float gc = Gc[kC - 1];
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) dS[i][j] *= gc;
        }
#pragma unroll 4
        for (int t = 0; t < kQ; ++t) {
            const float4 x0 = ld4(Qc + t * kD + L.sr0), x1 = ld4(Qc + t * kD + L.sr0 + 4);
            const float4 o = ld4o(Oc + t * kCols + L.sc0);
            const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
            float gq = 1.f;
            if (kGt) {
                const int last = t * a.nh + a.nh - 1;
                gq = last < kC ? Gc[last] : 0.f;
            }
            const float ov[4] = {gq * o.x, gq * o.y, gq * o.z, gq * o.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) dS[i][j] = fmaf(xv[i], ov[j], dS[i][j]);
        }
        update_state<kC>(dS, Wc, dUsm, L, -1.f);
    }
    if (a.dh0) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            st4(a.dh0 + ((size_t)bh * kD + L.sr0 + i) * kD + cg + L.sc0,
                make_float4(dS[i][0], dS[i][1], dS[i][2], dS[i][3]));
    }
}

template <typename TDo, bool kGt>
__global__ void __launch_bounds__(kChainThreads, 1) cb_chains(const CbArgs a)
{
    extern __shared__ float4 sm_chain[];
    if (blockIdx.z == 0) fwd_chain<kGt>(a, (char *)sm_chain);
    else bwd_chain<TDo, kGt>(a, (char *)sm_chain);
}

// ------------------------------------------------------------------ 3. per-chunk gradients
constexpr int kGradThreads = 512;

// sum over the 4 lanes of a quad (all four get it)
__device__ __forceinline__ float quad_sum(float x)
{
    x += __shfl_xor_sync(0xffffffffu, x, 1);
    return x + __shfl_xor_sync(0xffffffffu, x, 2);
}

// 3a. products with the boundary states. Thread (256 per CTA): rows kk and
// kk + 64 of S0 (then of dS1), kk = tid / 4, float4 columns 16 i + 4 qq
// (qq = tid % 4), i = 0 .. 7; a row of the left operand times those rows is
// a dot product over the quad, each value read feeding both rows.
constexpr int kGradSThreads = 256;
constexpr int kGradSSmemFloats = (kQ + 2 * kC) * kS;

template <typename TDo, bool kG>
__global__ void __launch_bounds__(kGradSThreads, 2) cb_grad_s(const CbArgs a)
{
    extern __shared__ float4 sm_grad_s[];
    __shared__ float wsum[kGradSThreads / 32];
    float *dOs = (float *)sm_grad_s, *Ups = dOs + kQ * kS, *dUps = Ups + kC * kS;
    const int ci = blockIdx.x, bh = ci / a.nc, c = ci - bh * a.nc;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5, kk = tid >> 2, qq = tid & 3;
    const ChunkRows cr = chunk_rows(a, bh, c);
    if (cr.nt == 0) return;   // past the sequence's end (packed calls)
    float *rec = a.rec + (size_t)ci * kRecFloats;
    float4 sa[8], sb[8];
    auto load_rows = [&](const float *m) {
        const float *p0 = m + (size_t)ci * kStateFloats + kk * kD + 4 * qq, *p1 = p0 + 64 * kD;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            sa[i] = __ldg((const float4 *)(p0 + 16 * i));
            sb[i] = __ldg((const float4 *)(p1 + 16 * i));
        }
    };
    load_rows(a.S0);
    stage_f32<false, kQ, TDo>(a, cr, (const TDo *)a.d_o, dOs);
    {
        const float *up = a.Up + (size_t)ci * kRowsFloats, *dup = a.dUp + (size_t)ci * kRowsFloats;
        for (int i = tid; i < kC * kD / 4; i += kGradSThreads) {
            const int r = i >> 5, e = (i & 31) * 4;
            st4(Ups + r * kS + e, __ldg((const float4 *)(up + r * kD + e)));
            st4(dUps + r * kS + e, __ldg((const float4 *)(dup + r * kD + e)));
        }
    }
    __syncthreads();
    // dP = (dO U'^T) masked: rows t = w, w + 8, column s = lane -> the record's P slot
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int t = w + 8 * h;
        float acc = 0.f;
        const float *x = dOs + t * kS, *y = Ups + lane * kS;
#pragma unroll 8
        for (int d = 0; d < kD; d += 4) acc = dot4(ld4(x + d), ld4(y + d), acc);
        rec[kRecP + t * kC + lane] = lane <= t * a.nh + a.nh - 1 ? acc : 0.f;
    }
    auto row_dot2 = [&](const float *x, float &v0, float &v1) {
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 xv = ld4(x + 16 * i + 4 * qq);
            a0 = dot4(xv, sa[i], a0);
            a1 = dot4(xv, sb[i], a1);
        }
        v0 = quad_sum(a0);
        v1 = quad_sum(a1);
    };
    // dq <- dO S0^T, dW = -dU' S0^T (the record's W slot)
#pragma unroll 2
    for (int t = 0; t < kQ; ++t) {
        float v0, v1;
        row_dot2(dOs + t * kS, v0, v1);
        if (qq == 0 && t < cr.nt) {
            float *dq = a.dq + token_row(a, cr, t) * kD;
            dq[kk] = v0;
            dq[kk + 64] = v1;
        }
    }
#pragma unroll 2
    for (int r = 0; r < kC; ++r) {
        float v0, v1;
        row_dot2(dUps + r * kS, v0, v1);
        if (qq == 0) {
            rec[kRecW + r * kD + kk] = -v0;
            rec[kRecW + r * kD + kk + 64] = -v1;
        }
    }
    // dk <- U' dS1^T (gated: the decayed keys' gradient, and <dS1, S0> into aux)
    if (kG) {
        const float *p0 = a.dS1 + (size_t)ci * kStateFloats + kk * kD + 4 * qq, *p1 = p0 + 64 * kD;
        float part = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 x = __ldg((const float4 *)(p0 + 16 * i)), y = __ldg((const float4 *)(p1 + 16 * i));
            part = dot4(x, sa[i], dot4(y, sb[i], part));
            sa[i] = x, sb[i] = y;
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        if (lane == 0) wsum[w] = part;
        __syncthreads();
        if (tid == 0) {
            float tot = 0.f;
            for (int i = 0; i < kGradSThreads / 32; ++i) tot += wsum[i];
            rec[kRecAux] = tot;
        }
    } else {
        load_rows(a.dS1);
    }
#pragma unroll 2
    for (int r = 0; r < kC; ++r) {
        float v0, v1;
        row_dot2(Ups + r * kS, v0, v1);
        if (qq == 0 && r < cr.R) {
            float *dk = a.dk + key_row(a, cr, r) * kD;
            dk[kk] = v0;
            dk[kk + 64] = v1;
        }
    }
}

// 3b. the rest of the chunk's gradients. K and V tiles use a row stride of
// 136 floats: in the dT product a quarter-warp reads rows m, m + 2 of them
// at four interleaved column chunks, which then fall in distinct banks.
constexpr int kSR = kD + 8;
constexpr int kGradRSmemFloats =
    2 * kC * kSR + 2 * kC * kS + kQ * kS + 5 * kC * kL + 2 * kQ * kL + 6 * kC + kQ;

template <typename TIn, bool kG>
__global__ void __launch_bounds__(kGradThreads, 2) cb_grad_r(const CbArgs a)
{
    extern __shared__ float4 sm_grad_r[];
    float *Ks = (float *)sm_grad_r, *Vs = Ks + kC * kSR, *dUps = Vs + kC * kSR, *dWs = dUps + kC * kS;
    float *Qs = dWs + kC * kS;
    float *Ts = Qs + kQ * kS, *KKs = Ts + kC * kL, *dTs = KKs + kC * kL, *Xs = dTs + kC * kL, *Es = Xs + kC * kL;
    float *dPs = Es + kC * kL, *dEq = dPs + kQ * kL;
    float *be = dEq + kQ * kL, *Gm = be + kC, *Rt = Gm + kC, *lg = Rt + kC, *dGm = lg + kC, *dRt = dGm + kC;
    float *dGq = dRt + kC;
    const int ci = blockIdx.x, bh = ci / a.nc, c = ci - bh * a.nc;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const ChunkRows cr = chunk_rows(a, bh, c);
    if (cr.nt == 0) return;   // past the sequence's end (packed calls)
    const float *rec = a.rec + (size_t)ci * kRecFloats;
    const float *dup = a.dUp + (size_t)ci * kRowsFloats;
    for (int i = tid; i < kC * kD / 4; i += kGradThreads) {
        const int r = i >> 5, e = (i & 31) * 4;
        st4(Ks + r * kSR + e, __ldg((const float4 *)(rec + kRecK + r * kD + e)));
        st4(dUps + r * kS + e, __ldg((const float4 *)(dup + r * kD + e)));
        st4(dWs + r * kS + e, __ldg((const float4 *)(rec + kRecW + r * kD + e)));
        if (r < kQ) st4(Qs + r * kS + e, __ldg((const float4 *)(rec + kRecQ + r * kD + e)));
    }
    stage_f32<true, kC, TIn, kSR>(a, cr, (const TIn *)a.v, Vs);
    stage_betas<TIn>(a, cr, be);
    for (int i = tid; i < kC * kC; i += kGradThreads) {
        const int r = i >> 5, s2 = i & 31;
        Ts[r * kL + s2] = rec[kRecT + i];
        KKs[r * kL + s2] = rec[kRecKK + i];
        if (kG) Es[r * kL + s2] = rec[kRecE + i];
        if (i < kQ * kC) {
            // dP of the decayed scores P o Eq, and (gated) the gradient of Eq
            const float dpe = rec[kRecP + i];
            if (kG) {
                const int last = r * a.nh + a.nh - 1;
                dPs[r * kL + s2] = last < kC ? dpe * rec[kRecE + last * kC + s2] : 0.f;
                dEq[r * kL + s2] = dpe * rec[kRecPr + i];
            } else {
                dPs[r * kL + s2] = dpe;
            }
        }
    }
    if (kG && tid < kC) {
        Gm[tid] = rec[kRecGm + tid], Rt[tid] = rec[kRecRt + tid], lg[tid] = rec[kRecLg + tid];
        dGm[tid] = 0.f, dRt[tid] = 0.f;
        if (tid < kQ) dGq[tid] = 0.f;
    }
    __syncthreads();

    // dq = Gamma_last(t) dQ0 + dP K (row t = w, columns 4 lane .. 4 lane + 3);
    // gated: dGq_t = q_t . dQ0_t
    {
        const int d = 4 * lane;
        if (w < cr.nt) {   // warp-uniform
            float *dq = a.dq + token_row(a, cr, w) * kD + d;
            const float4 q0 = ld4(dq);
            float4 acc = q0;
            if (kG) {
                const int last = w * a.nh + a.nh - 1;
                const float gq = Gm[last];
                acc = make_float4(gq * q0.x, gq * q0.y, gq * q0.z, gq * q0.w);
                float pg = dot4(ld4(Qs + w * kS + d), q0, 0.f);
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) pg += __shfl_xor_sync(0xffffffffu, pg, o);
                if (lane == 0) dGq[w] = pg;
            }
#pragma unroll 8
            for (int s2 = 0; s2 < kC; ++s2) acc = axpy4(dPs[w * kL + s2], ld4(Ks + s2 * kSR + d), acc);
            st4(dq, acc);
        }
    }
    // dT = dW (diag(beta Gamma) K)^T + dU' (diag(beta) V)^T. Thread: columns
    // m = 2 mp, 2 mp + 1, rows 4 rq .. 4 rq + 3, float4 column chunks
    // j = dq (mod 4) of the 128-term contraction; the four quarters meet by
    // quad shuffles.
    {
        const int dq = tid & 3, mp = (tid >> 2) & 15, rq = tid >> 6;
        const float g0 = kG ? Gm[2 * mp] : 1.f, g1 = kG ? Gm[2 * mp + 1] : 1.f;
        float t[4][2];
#pragma unroll
        for (int i = 0; i < 4; ++i) t[i][0] = t[i][1] = 0.f;
#pragma unroll 2
        for (int jj = 0; jj < 8; ++jj) {
            const int d = 4 * (4 * jj + dq);
            float4 k0 = ld4(Ks + (2 * mp) * kSR + d), k1 = ld4(Ks + (2 * mp + 1) * kSR + d);
            if (kG) {   // the W term's keys carry Gamma_m
                k0 = make_float4(g0 * k0.x, g0 * k0.y, g0 * k0.z, g0 * k0.w);
                k1 = make_float4(g1 * k1.x, g1 * k1.y, g1 * k1.z, g1 * k1.w);
            }
            const float4 v0 = ld4(Vs + (2 * mp) * kSR + d), v1 = ld4(Vs + (2 * mp + 1) * kSR + d);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float4 x = ld4(dWs + (4 * rq + i) * kS + d), y = ld4(dUps + (4 * rq + i) * kS + d);
                t[i][0] = dot4(y, v0, dot4(x, k0, t[i][0]));
                t[i][1] = dot4(y, v1, dot4(x, k1, t[i][1]));
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 2; ++j) t[i][j] = quad_sum(t[i][j]);
        // lane dq stores row 4 rq + dq
        const int r = 4 * rq + dq;
        float o0 = t[0][0], o1 = t[0][1];
#pragma unroll
        for (int i = 1; i < 4; ++i)
            if (dq == i) o0 = t[i][0], o1 = t[i][1];
        dTs[r * kL + 2 * mp] = o0 * be[2 * mp];
        dTs[r * kL + 2 * mp + 1] = o1 * be[2 * mp + 1];
    }
    __syncthreads();
    // X = dT T^T: rows 2w, 2w+1, column m = lane
    {
        float x0 = 0.f, x1 = 0.f;
#pragma unroll 8
        for (int j = 0; j < kC; ++j) {
            const float tm = Ts[lane * kL + j];
            x0 = fmaf(dTs[2 * w * kL + j], tm, x0);
            x1 = fmaf(dTs[(2 * w + 1) * kL + j], tm, x1);
        }
        Xs[2 * w * kL + lane] = x0;
        Xs[(2 * w + 1) * kL + lane] = x1;
    }
    __syncthreads();
    // dG = strictly lower part of -T^T X (into dT's tile): rows 2w, 2w+1, column s = lane
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int r = 2 * w + i;
        float g = 0.f;
        for (int j = r; j < kC; ++j) g = fmaf(-Ts[j * kL + r], Xs[j * kL + lane], g);   // T[j][r] = 0 for j < r
        dTs[r * kL + lane] = lane < r ? g : 0.f;
    }
    __syncthreads();
    if (kG) {
        // dG o E into dT's tile; into X's tile the coefficient of E[r][s]
        // (s < r): beta_r dG[r][s] (K K^T)[r][s], plus dEq[t][s] on the row
        // r = last(t) of token t
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int r = 2 * w + i, s2 = lane;
            const float g = dTs[r * kL + s2];
            float x = be[r] * g * KKs[r * kL + s2];
            const int t = r / a.nh;
            if (r - t * a.nh == a.nh - 1 && t < kQ && s2 < r) x += dEq[t * kL + s2];
            Xs[r * kL + s2] = s2 < r ? x : 0.f;
            dTs[r * kL + s2] = g * Es[r * kL + s2];
        }
        __syncthreads();
    }
    // rows m0 = 2w, m1 = 2w + 1 together (every loaded row feeds both),
    // columns 4 lane .. 4 lane + 3:
    //   dk = ratio dKd + dP^T Q + diag(beta Gamma) T^T dW + B (dG o E) K + (B (dG o E))^T K
    //   dv = B T^T dU'
    //   dbeta = Gamma (K o T^T dW) + V o T^T dU' + (dG o E o K K^T), each summed over a row
    // (T and dG are lower triangular, so the joint ranges add only zeros;
    // ungated: Gamma = ratio = E = 1)
    const int m0 = 2 * w, m1 = m0 + 1;
    if (m0 < cr.R) {   // warp-uniform
        const int d = 4 * lane;
        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
        // gt: (B dG)^T K + dP^T Q, the terms of dk outside the beta Gamma (...) group
        float4 tw0 = z, tw1 = z, tu0 = z, tu1 = z, gk0 = z, gk1 = z, gt0 = z, gt1 = z;
        for (int r = m0; r < kC; ++r) {
            const float4 x = ld4(dWs + r * kS + d), y = ld4(dUps + r * kS + d);
            const float t0 = Ts[r * kL + m0], t1 = Ts[r * kL + m1];
            tw0 = axpy4(t0, x, tw0), tw1 = axpy4(t1, x, tw1);
            tu0 = axpy4(t0, y, tu0), tu1 = axpy4(t1, y, tu1);
        }
        for (int s2 = 0; s2 < m1; ++s2) {
            const float4 k4 = ld4(Ks + s2 * kSR + d);
            gk0 = axpy4(dTs[m0 * kL + s2], k4, gk0), gk1 = axpy4(dTs[m1 * kL + s2], k4, gk1);
        }
        for (int r = m1; r < kC; ++r) {
            const float4 k4 = ld4(Ks + r * kSR + d);
            gt0 = axpy4(be[r] * dTs[r * kL + m0], k4, gt0), gt1 = axpy4(be[r] * dTs[r * kL + m1], k4, gt1);
        }
#pragma unroll 4
        for (int t = 0; t < kQ; ++t) {
            const float4 q4 = ld4(Qs + t * kS + d);
            gt0 = axpy4(dPs[t * kL + m0], q4, gt0), gt1 = axpy4(dPs[t * kL + m1], q4, gt1);
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int m = m0 + i;
            const float4 tw = i ? tw1 : tw0, tu = i ? tu1 : tu0, gk = i ? gk1 : gk0, gt = i ? gt1 : gt0;
            const float bm = be[m], gm = kG ? Gm[m] : 1.f, rt = kG ? Rt[m] : 1.f;
            const size_t row = key_row(a, cr, m < cr.R ? m : 0);
            float *dkp = a.dk + row * kD + d;
            const float4 km = ld4(Ks + m * kSR + d);
            const float4 k0 = m < cr.R ? ld4(dkp) : z;   // dKd (gated) or U' dS1^T
            // ungated: rest carries the whole dbeta (gm = 1, dbg unused)
            float dbg = kG ? dot4(km, tw, 0.f) : 0.f;
            float rest = dot4(ld4(Vs + m * kSR + d), tu, kG ? 0.f : dot4(km, tw, 0.f));
            if (lane < m) rest = fmaf(dTs[m * kL + lane], KKs[m * kL + lane], rest);
            float drt = kG ? dot4(km, k0, 0.f) : 0.f;
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) {
                rest += __shfl_xor_sync(0xffffffffu, rest, o);
                if (kG) {
                    dbg += __shfl_xor_sync(0xffffffffu, dbg, o);
                    drt += __shfl_xor_sync(0xffffffffu, drt, o);
                }
            }
            if (m < cr.R) {
                const float bg = bm * gm;
                st4(dkp, make_float4(rt * k0.x + bg * tw.x + bm * gk.x + gt.x, rt * k0.y + bg * tw.y + bm * gk.y + gt.y,
                                     rt * k0.z + bg * tw.z + bm * gk.z + gt.z, rt * k0.w + bg * tw.w + bm * gk.w + gt.w));
                st4(a.dv + row * kD + d, make_float4(bm * tu.x, bm * tu.y, bm * tu.z, bm * tu.w));
                if (lane == 0) {
                    a.dbeta[row] = fmaf(dbg, gm, rest);
                    if (kG) dGm[m] = dbg * bm, dRt[m] = drt;
                }
            }
        }
    }
    if (!kG) return;
    __syncthreads();
    // dg of token gi (warp gi, lane = row r; the gate sits on row r' = gi n_h):
    // the sum over every decay factor that contains gamma_r' of its
    // coefficient times the factor without gamma_r' (an exp of a range sum
    // that skips r'), so no division by the gate.
    const int gi = w, rp = gi * a.nh;
    if (rp < cr.R) {   // warp-uniform
        const int r = lane;
        float term = 0.f;
        if (r >= rp) {
            const int t = r / a.nh;
            const float cg = dGm[r] + ((r - t * a.nh == a.nh - 1 && t < kQ) ? dGq[t] : 0.f);
            float sg = 0.f;   // sum_{x <= r, x != r'} lg
            for (int x = 0; x <= r; ++x) sg += x == rp ? 0.f : lg[x];
            term = cg * expf(sg);
            float acc = 0.f;  // sum_{s < x <= r, x != r'} lg, s from r' - 1 down
            for (int x = rp + 1; x <= r; ++x) acc += lg[x];
            for (int s2 = rp - 1; s2 >= 0; --s2) {
                term = fmaf(Xs[r * kL + s2], expf(acc), term);
                acc += lg[s2];
            }
        } else {
            float sr = 0.f;   // sum_{r < x < 32, x != r'} lg
            for (int x = r + 1; x < kC; ++x) sr += x == rp ? 0.f : lg[x];
            term = dRt[r] * expf(sr);
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) term += __shfl_xor_sync(0xffffffffu, term, o);
        if (lane == 0) {
            float sc = 0.f;   // sum_{x < 32, x != r'} lg
            for (int x = 0; x < kC; ++x) sc += x == rp ? 0.f : lg[x];
            a.dg[token_row(a, cr, gi)] = fmaf(rec[kRecAux], expf(sc), term);
        }
    }
}

template <typename TIn, typename TDo, bool kG>
cudaError_t launch_typed(const BwdProblem &p, const CbArgs &a)
{
    const size_t n_chunks = (size_t)p.B * p.H * a.nc;
    cudaError_t e;
    const int chain_smem = (int)chain_smem_bytes<TDo>();
    if ((e = cudaFuncSetAttribute(cb_chains<TDo, kG>, cudaFuncAttributeMaxDynamicSharedMemorySize, chain_smem)) !=
        cudaSuccess)
        return e;
    const dim3 chain_grid(p.B * p.H, kD / kCols, 2);
    if (n_chunks == 0) {   // T = 0: dh0 = dh_final (the reverse chains only)
        cb_chains<TDo, kG><<<chain_grid, kChainThreads, chain_smem, p.stream>>>(a);
        return cudaGetLastError();
    }
    const int prep_smem = (int)(kPrepSmemFloats * sizeof(float));
    if ((e = cudaFuncSetAttribute(cb_prep<TIn, kG>, cudaFuncAttributeMaxDynamicSharedMemorySize, prep_smem)) !=
        cudaSuccess)
        return e;
    cb_prep<TIn, kG><<<(unsigned)n_chunks, kPrepThreads, prep_smem, p.stream>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    cb_chains<TDo, kG><<<chain_grid, kChainThreads, chain_smem, p.stream>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const int gs_smem = (int)(kGradSSmemFloats * sizeof(float));
    if ((e = cudaFuncSetAttribute(cb_grad_s<TDo, kG>, cudaFuncAttributeMaxDynamicSharedMemorySize, gs_smem)) !=
        cudaSuccess)
        return e;
    cb_grad_s<TDo, kG><<<(unsigned)n_chunks, kGradSThreads, gs_smem, p.stream>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const int gr_smem = (int)(kGradRSmemFloats * sizeof(float));
    if ((e = cudaFuncSetAttribute(cb_grad_r<TIn, kG>, cudaFuncAttributeMaxDynamicSharedMemorySize, gr_smem)) !=
        cudaSuccess)
        return e;
    cb_grad_r<TIn, kG><<<(unsigned)n_chunks, kGradThreads, gr_smem, p.stream>>>(a);
    return cudaGetLastError();
}

template <typename TIn, typename TDo>
cudaError_t launch_gated_or_not(const BwdProblem &p, const CbArgs &a)
{
    return p.g ? launch_typed<TIn, TDo, true>(p, a) : launch_typed<TIn, TDo, false>(p, a);
}

int chunk_tokens(int nh) { return (kC / nh < kQ) ? kC / nh : kQ; }

}  // namespace

bool backward_chunk_shape_ok(const BwdProblem &p)
{
    return p.Dk == kD && p.Dv == kD && p.nh >= 1 && p.nh <= kC;
}

bool backward_chunk_supported(const BwdProblem &p) { return backward_chunk_shape_ok(p); }

size_t backward_chunk_scratch_bytes(const BwdProblem &p)
{
    if (!backward_chunk_shape_ok(p)) return 0;
    const int ct = chunk_tokens(p.nh);
    const size_t nc = (size_t)(p.max_T + ct - 1) / ct, n = (size_t)p.B * p.H * nc;
    return n * (kRecFloats + 2 * kStateFloats + 2 * kRowsFloats) * sizeof(float);
}

cudaError_t launch_backward_chunk(const BwdProblem &p)
{
    CbArgs a;
    a.B = p.B; a.T = p.T; a.H = p.H; a.nh = p.nh;
    a.ct = chunk_tokens(p.nh);
    a.cu = p.cu;
    a.max_T = p.max_T;
    a.nc = (p.max_T + a.ct - 1) / a.ct;
    a.q = p.q; a.k = p.k; a.v = p.v; a.beta = p.beta; a.h0 = p.h0;
    a.d_o = p.d_o; a.dh_final = p.dh_final;
    a.dq = p.dq; a.dk = p.dk; a.dv = p.dv; a.dbeta = p.dbeta; a.dh0 = p.dh0;
    const size_t n = (size_t)p.B * p.H * a.nc;
    a.rec = (float *)p.scratch;
    a.S0 = a.rec + n * kRecFloats;
    a.dS1 = a.S0 + n * kStateFloats;
    a.Up = a.dS1 + n * kStateFloats;
    a.dUp = a.Up + n * kRowsFloats;
    a.g = p.g; a.dg = p.dg; a.status = p.status;
    if (p.dtype == DP_F32) return launch_gated_or_not<float, float>(p, a);
    return p.do_dtype == DP_F32 ? launch_gated_or_not<__nv_bfloat16, float>(p, a)
                                : launch_gated_or_not<__nv_bfloat16, __nv_bfloat16>(p, a);
}

}  // namespace dp
