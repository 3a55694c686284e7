// Backward pass (reverse-mode gradients) of the DeltaProduct recurrence on
// CUDA cores, fp32 arithmetic.
//
// DeltaProduct paper, Sec.4 Eq.(2)-(3) and the gated per-token pseudocode:
// every sub-step is H' = H + k u^T with u = beta (v - H^T k); the token's
// gate scales H once before its sub-steps; o_t = H^T q_t. With dH' the
// gradient with respect to the state after a sub-step:
//   du = dH'^T k,  dv = beta du,  dbeta = du . (v - H^T k),
//   dk = dH' u - beta H du,  dH = dH' - beta k du^T;
// readout: dq_t = H do_t, dH += q_t do_t^T;
// gate: dg_t = <dH, H_before_gate>, dH <- g_t dH.
//
// Work split: one CTA owns a 32-column slice of one (batch, head) state:
// lane = value column, warp w (16 warps) = a block of D_k/16 key rows, the
// slice in registers. The recurrence is a chain of dependent matvecs, so
// short per-thread chains and several warps per scheduler set its speed. The value-column quantities (dv,
// dh0) belong to the CTA; the key-row and scalar ones (dq, dk, dbeta, dg)
// are sums over all value columns, so each CTA adds its part with a
// global reduction (the D_v/32 CTAs of a head add in an unspecified order).
//
// Packed variable-length sequences (cu != NULL): CTA row b is sequence b,
// found through seq_range; checkpoints and errors are laid out for the
// longest sequence per (sequence, head).
//
// Time order: the states needed in reverse are rebuilt, not kept. The CTA
// first runs the recurrence forward once, storing its slice of the state at
// the start of every L-th token (checkpoints) and every sub-step's error
// e = v - H^T k into the workspace; both are read back only by the CTA
// that wrote them, after barriers. It then walks the segments of L tokens from the last:
// the segment is replayed from its checkpoint with the stored errors (the
// updates H += k (beta e)^T need no reduction), keeping each token's start
// state in shared memory, and its tokens are differentiated in reverse. A
// sub-step's state is recomputed from the token's gated state with the
// same operations as the forward, so every state the backward uses is
// bit-identical to the forward's.
#include "internal.h"

namespace dp {
namespace {

constexpr int kWarps = 16;
constexpr int kCols = 32;
constexpr int kThreads = kWarps * 32;

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

// Tokens per checkpoint segment: the segment's token-start states fill most
// of the shared memory (L * D_k * 32 floats).
template <int DK>
struct Seg {
    static constexpr int L = 12 * (128 / DK);
    static constexpr size_t kStates = (size_t)L * DK * kCols * 4;
    static constexpr size_t kErr = (size_t)L * 4 * kCols * 4;            // n_h <= 4
    static constexpr size_t kKeys = (size_t)5 * DK * 4;                    // n_h keys + q
    static constexpr size_t kPart = (size_t)2 * kWarps * kCols * 4;
    static constexpr size_t kRed = 16 * 4;
    static constexpr size_t kSmem = kStates + kErr + kKeys + kPart + kRed;
};
static_assert(Seg<32>::kSmem <= 227 * 1024 && Seg<64>::kSmem <= 227 * 1024 && Seg<128>::kSmem <= 227 * 1024,
              "shared memory");

// Sum over the 32 lanes of each of the R per-thread values p[0..R-1]
// (R a power of two, <= 32), by recursive halving: at each exchange a lane
// keeps one half of its values and adds its partner's copy of that half.
// Returns in lane l the full sum of value l * R / 32 (for R < 32, the
// 32 / R consecutive lanes of one value all hold it).
template <int R>
__device__ __forceinline__ float lane_sum_rows(float (&p)[R], int lane)
{
    int n = R;
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) {
        if (n > 1) {
            const bool upper = (lane & m) != 0;
#pragma unroll
            for (int i = 0; i < R / 2; ++i) {
                if (i < n / 2) {
                    const float send = upper ? p[i] : p[i + n / 2];
                    const float keep = upper ? p[i + n / 2] : p[i];
                    p[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
                }
            }
            n >>= 1;
        } else {
            p[0] += __shfl_xor_sync(0xffffffffu, p[0], m);
        }
    }
    return p[0];
}

__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
    return x;
}

struct BwdArgs {
    int T, H, Dv, nh;
    const void *q, *k, *v, *beta, *g;
    const float *h0;
    const void *d_o;
    const float *dh_final;
    float *dq, *dk, *dv, *dbeta, *dg, *dh0;
    float *ckpt;   // [B*H][n_seg of max_T][DK][Dv]
    float *errs;   // [B*H][max_T][nh][Dv] errors v - H^T k of every sub-step
    const int *cu; // packed sequences: token offsets [B+1] (NULL: dense [B,T] layout)
    int max_T;     // longest sequence (T for dense calls)
    uint32_t *status;
};

template <int DK, typename TIn, typename TDo>
__global__ void __launch_bounds__(kThreads, 1) backward_kernel(const BwdArgs a)
{
    constexpr int R = DK / kWarps;   // key rows per warp (and per thread)
    constexpr int L = Seg<DK>::L;
    extern __shared__ float smem[];
    float *spre = smem;                                        // [L][DK][32] token-start states
    float *serr = spre + (size_t)L * DK * kCols;               // [L * nh][32] errors v - H^T k
    float *skey = serr + (size_t)L * 4 * kCols;                // [nh + 1][DK] keys of a token, then q
    float *part = skey + 5 * DK;                               // [2][kWarps][32] matvec partials
    float *red = part + 2 * kWarps * kCols;                    // [kWarps] CTA reductions

    const TIn *q = (const TIn *)a.q, *k = (const TIn *)a.k, *v = (const TIn *)a.v;
    const TIn *beta = (const TIn *)a.beta, *g = (const TIn *)a.g;
    const TDo *d_o = (const TDo *)a.d_o;
    const int Tl = a.T, H = a.H, Dv = a.Dv, nh = a.nh;   // Tl: token rows of the layout
    const int bh = blockIdx.x, b = bh / H, h = bh - b * H;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int col = blockIdx.y * kCols + lane, row0 = w * R;
    const size_t state_base = (size_t)bh * DK * Dv;
    // this sequence's tokens (packed calls: checked against the offsets'
    // contract first; a sequence that breaks it is not touched)
    const SeqRange sq = seq_range(a.cu, b, gridDim.x / H, Tl, a.max_T);
    if (!sq.ok) {
        if (threadIdx.x == 0 && blockIdx.y == 0) report_bad_sequence(a.status);
        return;
    }
    const int T = sq.len;
    const int n_seg = (T + L - 1) / L;
    float *ckpt = a.ckpt + (size_t)bh * ((a.max_T + L - 1) / L) * DK * Dv;
    float *errs = a.errs + (size_t)bh * a.max_T * nh * Dv;
    auto tok_of = [&](int t) { return ((size_t)sq.b_map * Tl + sq.t0 + t) * H + h; };

    // M^T x for the CTA's columns (x: D_k floats in shared memory); one
    // barrier (the partial buffers alternate between calls).
    int pb = 0;
    auto matvec = [&](const float *x, const float (&M)[R]) {
        float acc = 0.f;
#pragma unroll
        for (int r = 0; r < R; ++r) acc = fmaf(M[r], x[row0 + r], acc);
        part[(pb * kWarps + w) * kCols + lane] = acc;
        __syncthreads();
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < kWarps; ++i) s += part[(pb * kWarps + i) * kCols + lane];
        pb ^= 1;
        return s;
    };
    // The inputs of one token, fetched into registers one token ahead of
    // their use so that the global loads overlap the current token's work:
    // this thread's share of the n_h key rows (and q in the backward), and
    // its column's v, the betas, the gate and d_o.
    constexpr int KQ = (5 * DK + kThreads - 1) / kThreads;
    struct TokIn {
        float kq[KQ];
        float v[4], be[4];
        float g, dov;
    };
    // mode: 0 forward (v), 1 replay (stored errors in v[]), 2 backward (q, d_o, stored errors)
    auto fetch = [&](int t, int mode) {
        TokIn in;
        const bool bwd = mode == 2;
        const size_t tok = tok_of(t);
        const float *et = errs + (size_t)t * nh * Dv + col;
        const int nk = nh * DK, n = nk + (bwd ? DK : 0);
#pragma unroll
        for (int m = 0; m < KQ; ++m) {
            const int i = threadIdx.x + m * kThreads;
            in.kq[m] = i < nk ? to_f(k[tok * nk + i]) : (i < n ? to_f(q[tok * DK + i - nk]) : 0.f);
        }
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            in.v[jj] = jj >= nh ? 0.f : mode == 0 ? to_f(v[(tok * nh + jj) * Dv + col]) : mode == 1 ? et[jj * Dv] : 0.f;
            in.be[jj] = jj < nh ? to_f(beta[tok * nh + jj]) : 0.f;
        }
        in.g = g ? to_f(g[tok]) : 1.f;
        in.dov = bwd ? to_f(d_o[tok * Dv + col]) : 0.f;
        return in;
    };
    // The keys (and q) of `in` into skey for the whole CTA.
    auto stage = [&](const TokIn &in, bool bwd) {
        __syncthreads();   // previous users of skey are done
        const int n = nh * DK + (bwd ? DK : 0);
#pragma unroll
        for (int m = 0; m < KQ; ++m) {
            const int i = threadIdx.x + m * kThreads;
            if (i < n) skey[i] = in.kq[m];
        }
        __syncthreads();
    };

    float S[R];
#pragma unroll
    for (int r = 0; r < R; ++r) S[r] = a.h0 ? a.h0[state_base + (size_t)(row0 + r) * Dv + col] : 0.f;

    // one forward token on the state S (keys staged); its errors v - H^T k
    // go to `err` ([nh][Dv] of this token, this CTA's columns)
    auto forward_token = [&](const TokIn &in, float *err) {
        if (g) {
#pragma unroll
            for (int r = 0; r < R; ++r) S[r] *= in.g;
        }
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            if (jj >= nh) break;
            const float *kj = skey + jj * DK;
            const float e = in.v[jj] - matvec(kj, S);
            if (w == 0) err[jj * Dv] = e;
            const float u = in.be[jj] * e;
#pragma unroll
            for (int r = 0; r < R; ++r) S[r] = fmaf(kj[row0 + r], u, S[r]);
        }
    };

    // ---- 1. forward once, checkpoint at every L-th token start
    TokIn cur{};
    if (T > 0) cur = fetch(0, 0);   // every fetch below names a token in [0, T)
    for (int t = 0; t < T; ++t) {
        if (t % L == 0) {
            float *c = ckpt + (size_t)(t / L) * DK * Dv;
#pragma unroll
            for (int r = 0; r < R; ++r) c[(size_t)(row0 + r) * Dv + col] = S[r];
        }
        stage(cur, false);
        const TokIn nxt = t + 1 < T ? fetch(t + 1, 0) : cur;
        forward_token(cur, errs + (size_t)t * nh * Dv + col);
        cur = nxt;
    }
    // the replay starts with the last segment's first token, whose errors
    // must all be written (and visible to the CTA) before they are fetched
    __syncthreads();
    if (T > 0) cur = fetch((n_seg - 1) * L, 1);

    // ---- 2. segments in reverse
    float dS[R];
#pragma unroll
    for (int r = 0; r < R; ++r)
        dS[r] = a.dh_final ? a.dh_final[state_base + (size_t)(row0 + r) * Dv + col] : 0.f;

    for (int sgi = n_seg - 1; sgi >= 0; --sgi) {
        const int t0 = sgi * L, t1 = min(T, t0 + L);
        const float *c = ckpt + (size_t)sgi * DK * Dv;
#pragma unroll
        for (int r = 0; r < R; ++r) S[r] = c[(size_t)(row0 + r) * Dv + col];
        // replay the segment with the stored errors: token-start states and
        // errors into shared memory
        for (int t = t0; t < t1; ++t) {
            float *sp = spre + (size_t)(t - t0) * DK * kCols;
#pragma unroll
            for (int r = 0; r < R; ++r) sp[(row0 + r) * kCols + lane] = S[r];
            stage(cur, false);
            const bool last = t + 1 == t1;
            const TokIn nxt = fetch(last ? t1 - 1 : t + 1, last ? 2 : 1);
            if (g) {
#pragma unroll
                for (int r = 0; r < R; ++r) S[r] *= cur.g;
            }
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                if (jj >= nh) break;
                const float *kj = skey + jj * DK;
                if (w == 0) serr[((t - t0) * nh + jj) * kCols + lane] = cur.v[jj];
                const float u = cur.be[jj] * cur.v[jj];
#pragma unroll
                for (int r = 0; r < R; ++r) S[r] = fmaf(kj[row0 + r], u, S[r]);
            }
            cur = nxt;
        }
        // backward over the segment's tokens
        for (int t = t1 - 1; t >= t0; --t) {
            const size_t tok = tok_of(t);
            stage(cur, true);
            const TokIn in = cur;
            // next: the previous token, or the first token of the previous segment
            cur = fetch(t > t0 ? t - 1 : (sgi > 0 ? (sgi - 1) * L : 0), t > t0 ? 2 : 1);
            const float gt = in.g;
            const float *sp = spre + (size_t)(t - t0) * DK * kCols;
            float Sg[R];
#pragma unroll
            for (int r = 0; r < R; ++r) Sg[r] = g ? sp[(row0 + r) * kCols + lane] * gt : sp[(row0 + r) * kCols + lane];
            float uj[4], ej[4];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                ej[jj] = jj < nh ? serr[((t - t0) * nh + jj) * kCols + lane] : 0.f;
                uj[jj] = in.be[jj] * ej[jj];
            }
            // readout: dq_t = H_nh do_t (sum over this CTA's columns), dH += q do^T
            {
                float p[R];
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    float s = Sg[r];
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj)
                        if (jj < nh) s = fmaf(skey[jj * DK + row0 + r], uj[jj], s);
                    p[r] = s * in.dov;
                }
                const float sum = lane_sum_rows<R>(p, lane);
                if ((lane & (32 / R - 1)) == 0) atomicAdd(&a.dq[tok * DK + row0 + lane * R / 32], sum);
                const float *qv = skey + nh * DK;
#pragma unroll
                for (int r = 0; r < R; ++r) dS[r] = fmaf(qv[row0 + r], in.dov, dS[r]);
            }
            // sub-steps in reverse
#pragma unroll
            for (int jj = 3; jj >= 0; --jj) {
                if (jj >= nh) continue;
                const float *kj = skey + jj * DK;
                float Sj[R];   // state before sub-step jj, as the forward computed it
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    float s = Sg[r];
#pragma unroll
                    for (int i = 0; i < 3; ++i)
                        if (i < jj) s = fmaf(skey[i * DK + row0 + r], uj[i], s);
                    Sj[r] = s;
                }
                const float du = matvec(kj, dS);
                const float de = in.be[jj] * du;
                if (w == 0) {
                    a.dv[(tok * nh + jj) * Dv + col] = de;
                    const float db = warp_sum(du * ej[jj]);
                    if (lane == 0) atomicAdd(&a.dbeta[tok * nh + jj], db);
                }
                float p[R];
#pragma unroll
                for (int r = 0; r < R; ++r) p[r] = fmaf(dS[r], uj[jj], -in.be[jj] * Sj[r] * du);
                const float sum = lane_sum_rows<R>(p, lane);
                if ((lane & (32 / R - 1)) == 0)
                    atomicAdd(&a.dk[(tok * nh + jj) * DK + row0 + lane * R / 32], sum);
#pragma unroll
                for (int r = 0; r < R; ++r) dS[r] = fmaf(-kj[row0 + r], de, dS[r]);
            }
            // gate: dg_t = <dH, H_before_gate>, dH <- g dH
            if (g) {
                float acc = 0.f;
#pragma unroll
                for (int r = 0; r < R; ++r) acc = fmaf(dS[r], sp[(row0 + r) * kCols + lane], acc);
                acc = warp_sum(acc);
                if (lane == 0) red[w] = acc;
                __syncthreads();
                if (threadIdx.x == 0) {
                    float sum = 0.f;
#pragma unroll
                    for (int i = 0; i < kWarps; ++i) sum += red[i];
                    atomicAdd(&a.dg[tok], sum);
                }
#pragma unroll
                for (int r = 0; r < R; ++r) dS[r] *= gt;
            }
        }
    }
    if (a.dh0) {
#pragma unroll
        for (int r = 0; r < R; ++r) a.dh0[state_base + (size_t)(row0 + r) * Dv + col] = dS[r];
    }
}

template <int DK, typename TIn, typename TDo>
cudaError_t launch_dk(const BwdProblem &p, const BwdArgs &a)
{
    auto kernel = backward_kernel<DK, TIn, TDo>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)Seg<DK>::kSmem);
    if (e != cudaSuccess) return e;
    dim3 grid(p.B * p.H, p.Dv / kCols);
    kernel<<<grid, kThreads, Seg<DK>::kSmem, p.stream>>>(a);
    return cudaGetLastError();
}

template <typename TIn, typename TDo>
cudaError_t launch_typed(const BwdProblem &p, const BwdArgs &a)
{
    switch (p.Dk) {
    case 32: return launch_dk<32, TIn, TDo>(p, a);
    case 64: return launch_dk<64, TIn, TDo>(p, a);
    default: return launch_dk<128, TIn, TDo>(p, a);
    }
}

}  // namespace

int backward_segment_tokens(int Dk) { return Dk == 32 ? Seg<32>::L : Dk == 64 ? Seg<64>::L : Seg<128>::L; }

namespace {
size_t backward_ckpt_bytes(const BwdProblem &p)
{
    const int L = backward_segment_tokens(p.Dk);
    const size_t n_seg = p.max_T > 0 ? (size_t)(p.max_T + L - 1) / L : 0;
    return (((size_t)p.B * p.H * n_seg * p.Dk * p.Dv * sizeof(float)) + 255) & ~(size_t)255;
}
}  // namespace

size_t backward_scratch_bytes(const BwdProblem &p)
{
    return backward_ckpt_bytes(p) + (size_t)p.B * p.H * p.max_T * p.nh * p.Dv * sizeof(float);
}

cudaError_t launch_backward(const BwdProblem &p)
{
    const size_t tok = (size_t)(p.cu ? 1 : p.B) * p.T * p.H;   // token-heads of the layout
    cudaError_t e;
    // the key-row and scalar gradients are accumulated by global reductions
    if ((e = cudaMemsetAsync(p.dq, 0, tok * p.Dk * sizeof(float), p.stream)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(p.dk, 0, tok * p.nh * p.Dk * sizeof(float), p.stream)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(p.dbeta, 0, tok * p.nh * sizeof(float), p.stream)) != cudaSuccess) return e;
    if (p.g && (e = cudaMemsetAsync(p.dg, 0, tok * sizeof(float), p.stream)) != cudaSuccess) return e;
    BwdArgs a;
    a.T = p.T; a.H = p.H; a.Dv = p.Dv; a.nh = p.nh;
    a.q = p.q; a.k = p.k; a.v = p.v; a.beta = p.beta; a.g = p.g; a.h0 = p.h0;
    a.d_o = p.d_o; a.dh_final = p.dh_final;
    a.dq = p.dq; a.dk = p.dk; a.dv = p.dv; a.dbeta = p.dbeta; a.dg = p.dg; a.dh0 = p.dh0;
    a.ckpt = (float *)p.scratch;
    a.cu = p.cu;
    a.max_T = p.max_T;
    a.status = p.status;
    a.errs = (float *)((char *)p.scratch + backward_ckpt_bytes(p));
    if (p.dtype == DP_F32) return launch_typed<float, float>(p, a);
    return p.do_dtype == DP_F32 ? launch_typed<__nv_bfloat16, float>(p, a)
                                : launch_typed<__nv_bfloat16, __nv_bfloat16>(p, a);
}

}  // namespace dp
