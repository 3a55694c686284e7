// Tensor-core chunked DeltaProduct forward (tcgen05 / TMEM / TMA), bf16 inputs,
// D_k = D_v = 128, fp32 state and accumulation.
//
// What it computes (DeltaProduct paper, Sec.5.1: the n_h keys of every token
// form an extended T*n_h DeltaNet sequence, the gate is applied once per
// token, only the last step of each token is read out; chunk transform from
// the OSDN paper, App.A.2 / App.C, with write key = read key, state H = S^T).
// Per chunk of ct = floor(64/n_h) whole tokens (R = ct*n_h <= 64 rows of the
// extended sequence, padded with beta = 0 rows, which are exact no-ops), with
// L_r the cumulative log-gate from the chunk start, Gamma_r = exp(L_r),
// E_rs = exp(L_r - L_s):
//   G     = tril(diag(beta) (K K^T * E), -1)          Gram        (tcgen05)
//   T     = (I + G)^{-1}                              UT transform (CUDA cores)
//   W     = T diag(beta*Gamma) K,  U = T diag(beta) V              (tcgen05)
//   U'    = U - W H0                                  state pass   (tcgen05)
//   H     = Gamma_C H0 + K^T diag(Gamma_C/Gamma) U'               (tcgen05)
//   o_t   = Gamma_r H0^T q_t + sum_{s<=r} E_rs (q_t.k_s) u'_s, r = last row of t
// The state stays in TMEM for the whole sequence. Everything is computed in
// the transposed orientation (M = D_v = 128 lanes: lane = value column) so
// that the state and U' feed the next MMA straight from TMEM as the A operand.
#include <string.h>

#include "internal.h"
#include "sm100.cuh"

#include <cudaTypedefs.h>

namespace dp {
namespace {

using namespace sm100;

constexpr int kD = 128;            // D_k = D_v
constexpr int kC = 64;             // extended rows per chunk (padded)
constexpr int kThreads = 128;      // thread i <-> TMEM lane i

// TMEM column map (512 columns allocated)
// The state and U' enter their MMAs as A operands from TMEM in two bf16
// parts, x = hi + lo with hi = bf16(x) and lo = bf16(x - hi), which carries
// about 16 mantissa bits; the B operands are single bf16 tiles.
constexpr uint32_t kColS = 0;      // S^T fp32, lane = dv, 128 cols = dk
constexpr uint32_t kColSB = 128;   // bf16 hi part of S^T, 64 cols
constexpr uint32_t kColUN = 192;   // U'^T fp32, 64 cols = chunk rows; then lo parts of U'
constexpr uint32_t kColUB = 256;   // bf16 hi part of U'^T, 32 cols
constexpr uint32_t kColUBD = 288;  // bf16 hi part of U'^T * Gamma_C/Gamma_s (gated), 32 cols
constexpr uint32_t kColO = 320;    // O^T fp32, up to 64 cols = tokens
constexpr uint32_t kColGW = 384;   // [K;Q] K^T fp32, then W^T fp32 (lane = dk); then lo part of S^T
constexpr uint32_t kColSBL = kColGW;       // bf16 lo part of S^T, 64 cols
constexpr uint32_t kColUBL = kColUN;       // bf16 lo part of U'^T, 32 cols
constexpr uint32_t kColUBDL = kColUN + 32; // bf16 lo part of the decayed U'^T, 32 cols
constexpr uint32_t kTmemCols = 512;

// Shared memory map (bytes from a 1024-aligned base)
constexpr uint32_t kKQBytes = 2 * 128 * 128;       // 2 blocks of 64 dk x 128 rows (K rows 0..63, Q rows 64..127)
constexpr uint32_t kVBytes = 2 * 64 * 128;         // 2 blocks of 64 dv x 64 rows
constexpr uint32_t kStageBytes = kKQBytes + kVBytes;
constexpr uint32_t kOffStage = 0;                  // 2 stages
constexpr uint32_t kOffTb = 2 * kStageBytes;       // T diag(beta), bf16 64 x 64, K-major
constexpr uint32_t kOffTbg = kOffTb + 8192;        // T diag(beta Gamma)
constexpr uint32_t kOffP = kOffTbg + 8192;         // P = tril(Q K^T * E), bf16 hi part, 64 x 64
constexpr uint32_t kOffPL = kOffP + 8192;          // bf16 lo part of P
constexpr uint32_t kOffNW = kOffPL + 8192;         // -W, MN-major (rows dk, 64 i), 16 KB
constexpr uint32_t kOffG = kOffNW + 16384;         // fp32 G [64][65]
constexpr uint32_t kLd = 65;
constexpr uint32_t kOffT = kOffG + 64 * kLd * 4;   // fp32 T [64][65]
constexpr uint32_t kOffX = kOffT + 64 * kLd * 4;   // fp32 scratch [3][16][17]
constexpr uint32_t kOffVec = kOffX + 3 * 16 * 17 * 4;   // beta[64], L[64]
constexpr uint32_t kOffBar = kOffVec + 2 * 64 * 4;      // barriers + misc (64 B)
constexpr uint32_t kSmemBytes = kOffBar + 64 + 1024;    // + alignment slack

constexpr uint32_t kWaitTries = 1u << 22;

struct Params {
    const __nv_bfloat16 *beta, *g;
    const float *h0;
    void *o;
    float *h_final;
    uint32_t *status;
    int T, H, nh, ct, nq, n_chunks;
};

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
        else
            cudaGetLastError();
    }
    return fn;
}

// bf16 tensor map with a 64-element (128-byte) inner box and 128-byte swizzle.
bool encode(CUtensorMap *map, const void *base, int rank, const cuuint64_t *dims,
            const cuuint64_t *strides_bytes, const cuuint32_t *box)
{
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void *>(base),
               dims, strides_bytes, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


__device__ __forceinline__ void flag_error(uint32_t *status, volatile uint32_t *abort_s, uint32_t code)
{
    *abort_s = 1;
    if (status) atomicCAS(status, 0u, code);
}

// Load 64 consecutive fp32 TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld64f(uint32_t taddr, float (&v)[64])
{
    uint32_t r[16];
#pragma unroll
    for (int c0 = 0; c0 < 64; c0 += 16) {
        tmem_ld16(taddr + c0, r);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) v[c0 + j] = __uint_as_float(r[j]);
    }
}

// hi/lo bf16 pairs of (a, b): hi = bf16(x), lo = bf16(x - hi)
__device__ __forceinline__ void split_pack(float a, float b, uint32_t &hi, uint32_t &lo)
{
    hi = pack_bf16x2(a, b);
    const float ah = __uint_as_float(hi << 16), bh = __uint_as_float(hi & 0xFFFF0000u);
    lo = pack_bf16x2(a - ah, b - bh);
}

__device__ __forceinline__ void store_out(float *o, size_t i, float x) { o[i] = x; }
__device__ __forceinline__ void store_out(__nv_bfloat16 *o, size_t i, float x) { o[i] = __float2bfloat16_rn(x); }

template <typename TOut>
__global__ void __launch_bounds__(kThreads, 1)
chunk_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                const __grid_constant__ CUtensorMap tm_q, const Params p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    float *Gs = (float *)(sm + kOffG);
    float *Ts = (float *)(sm + kOffT);
    float *Xs = (float *)(sm + kOffX);
    float *beta_s = (float *)(sm + kOffVec);
    float *L_s = beta_s + 64;
    uint64_t *bar_tma = (uint64_t *)(sm + kOffBar);   // [2], one per stage
    uint64_t *bar_mma = bar_tma + 2;
    uint32_t *tmem_slot = (uint32_t *)(bar_mma + 1);
    volatile uint32_t *abort_s = tmem_slot + 1;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.x, b = bh / p.H, h = bh - b * p.H;
    const int nh = p.nh, ct = p.ct, R = ct * nh, nq = p.nq, T = p.T;
    const bool gated = p.g != nullptr;

    // Zero every tile once: rows TMA never writes (query rows >= ct, the
    // padding row when 64 % n_h != 0) must hold finite zeros.
    for (uint32_t i = tid * 16; i < kOffG; i += kThreads * 16)
        *(uint4 *)(sm + i) = make_uint4(0, 0, 0, 0);
    if (tid == 0) {
        mbar_init(&bar_tma[0], 1);
        mbar_init(&bar_tma[1], 1);
        mbar_init(bar_mma, 1);
        *abort_s = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_q);
    }
    if (warp == 0) tmem_alloc(tmem_slot, kTmemCols);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;
    const uint32_t trow = tbase + ((uint32_t)(warp * 32) << 16);   // this thread's lane, column 0

    auto issue_loads = [&](int chunk) {
        const int st = chunk & 1;
        uint8_t *kq = sm + kOffStage + st * kStageBytes;
        uint8_t *vv = kq + kKQBytes;
        const int t0 = chunk * ct;
        mbar_arrive_expect_tx(&bar_tma[st], (uint32_t)(512 * R + 256 * ct));
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
            tma_load_5d(kq + kb * 16384, &tm_k, &bar_tma[st], kb * 64, 0, h, t0, b);
            tma_load_4d(kq + kb * 16384 + 64 * 128, &tm_q, &bar_tma[st], kb * 64, h, t0, b);
            tma_load_5d(vv + kb * 8192, &tm_v, &bar_tma[st], kb * 64, 0, h, t0, b);
        }
    };

    // S^T <- h0^T (lane = dv, column = dk), or zeros
    {
        uint32_t r[16];
        for (int c0 = 0; c0 < kD; c0 += 16) {
#pragma unroll
            for (int j = 0; j < 16; ++j)
                r[j] = __float_as_uint(p.h0 ? p.h0[((size_t)bh * kD + c0 + j) * kD + tid] : 0.f);
            tmem_st16(trow + kColS + c0, r);
        }
        tmem_wait_st();
    }

    int issued = 0, landed = 0;
    if (tid == 0) issue_loads(0);
    issued = 1;
    if (p.n_chunks > 1) {
        if (tid == 0) issue_loads(1);
        issued = 2;
    }
    uint32_t mma_phase = 0;
    bool mma_pending = false;

    for (int c = 0; c < p.n_chunks; ++c) {
        const int st = c & 1;
        uint8_t *kq = sm + kOffStage + st * kStageBytes;
        uint8_t *vv = kq + kKQBytes;
        const int t0 = c * ct;

        // (1) betas and cumulative log-gates of the chunk's rows
        if (tid < kC) {
            const int r = tid, tl = r / nh, j = r - tl * nh, t = t0 + tl;
            const bool valid = (r < R) && (t < T);
            const size_t tok = ((size_t)b * T + t) * p.H + h;
            beta_s[r] = valid ? __bfloat162float(p.beta[tok * nh + j]) : 0.f;
            float lg = 0.f;
            if (gated && valid && j == 0) lg = fmaxf(logf(__bfloat162float(p.g[tok])), -80.f);
            Xs[r] = lg;
        }
        __syncthreads();
        if (tid < kC) {
            float acc = 0.f;
            for (int s = 0; s <= tid; ++s) acc += Xs[s];
            L_s[tid] = acc;
        }
        // (2) this chunk's K, Q, V tiles
        if (!mbar_wait(&bar_tma[st], (c >> 1) & 1, kWaitTries, abort_s)) flag_error(p.status, abort_s, kDevTimeout);
        __syncthreads();
        if (*abort_s) break;
        landed = c + 1;

        // (3) [K;Q] K^T -> TMEM (lanes 0..63 Gram rows, 64..127 query rows)
        if (tid == 0) {
            tc_fence_after();
            const uint32_t id = idesc_bf16(128, 64, false, false);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t a = smem_addr(kq) + (kk >> 2) * 16384 + (kk & 3) * 32;
                mma_ss(tbase + kColGW, sdesc_sw128(a, 16, 1024), sdesc_sw128(a, 16, 1024), id, kk > 0);
            }
            mma_commit(bar_mma);
        }
        mma_pending = true;
        if (!mbar_wait(bar_mma, mma_phase, kWaitTries, abort_s)) flag_error(p.status, abort_s, kDevTimeout);
        mma_phase ^= 1;
        __syncthreads();
        if (*abort_s) break;
        mma_pending = false;
        tc_fence_after();

        // (4) Gram rows -> G (fp32), query rows -> P (bf16 hi + lo parts)
        {
            float gq[64];
            tmem_ld64f(trow + kColGW, gq);
            if (tid < kC) {
                const int r = tid;
                const float br = beta_s[r], Lr = L_s[r];
#pragma unroll
                for (int s = 0; s < kC; ++s) {
                    float v = 0.f;
                    if (s < r) {
                        v = br * gq[s];
                        if (gated) v *= __expf(Lr - L_s[s]);
                    }
                    Gs[r * kLd + s] = v;
                }
            } else {
                const int i = tid - kC;
                const int r = i * nh + nh - 1;
                const bool valid = i < ct;
                const float Lr = valid ? L_s[r] : 0.f;
                uint8_t *P = sm + kOffP, *PL = sm + kOffPL;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    uint32_t w[4], wl[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int s0 = ch * 8 + 2 * e;
                        float v0 = 0.f, v1 = 0.f;
                        if (valid && s0 <= r) v0 = gated ? gq[s0] * __expf(Lr - L_s[s0]) : gq[s0];
                        if (valid && s0 + 1 <= r) v1 = gated ? gq[s0 + 1] * __expf(Lr - L_s[s0 + 1]) : gq[s0 + 1];
                        split_pack(v0, v1, w[e], wl[e]);
                    }
                    *(uint4 *)(P + sw128_offset(i, ch)) = make_uint4(w[0], w[1], w[2], w[3]);
                    *(uint4 *)(PL + sw128_offset(i, ch)) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
                }
            }
        }
        tc_fence_before();
        __syncthreads();

        // (5) T = (I + G)^{-1}: 16x16 diagonal blocks by forward substitution
        // (one warp per block, one column per lane), then the off-diagonal
        // blocks level by level: T_ab = -T_aa sum_{m=b}^{a-1} G_am T_mb.
        if (lane < 16) {
            const int base = warp * 16, col = base + lane;
            float x[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                float acc = (i == lane) ? 1.f : 0.f;
#pragma unroll
                for (int s2 = 0; s2 < i; ++s2) acc = fmaf(-Gs[(base + i) * kLd + base + s2], x[s2], acc);
                x[i] = acc;
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) Ts[(base + i) * kLd + col] = x[i];
        }
        __syncthreads();
        for (int d = 1; d < 4; ++d) {
            const int nblk = 4 - d;
            for (int e = tid; e < nblk * 256; e += kThreads) {
                const int bb = e >> 8, i = (e >> 4) & 15, j = e & 15, a = bb + d;
                float acc = 0.f;
                for (int m = 16 * bb; m < 16 * a; ++m)
                    acc = fmaf(Gs[(16 * a + i) * kLd + m], Ts[m * kLd + 16 * bb + j], acc);
                Xs[(bb * 16 + i) * 17 + j] = acc;
            }
            __syncthreads();
            for (int e = tid; e < nblk * 256; e += kThreads) {
                const int bb = e >> 8, i = (e >> 4) & 15, j = e & 15, a = bb + d;
                float acc = 0.f;
                for (int u = 0; u <= i; ++u)
                    acc = fmaf(Ts[(16 * a + i) * kLd + 16 * a + u], Xs[(bb * 16 + u) * 17 + j], acc);
                Ts[(16 * a + i) * kLd + 16 * bb + j] = -acc;
            }
            __syncthreads();
        }
        // T diag(beta) -> Tb (threads 0..63), T diag(beta Gamma) -> Tbg (64..127, gated)
        {
            const int i = tid & 63;
            const bool second = tid >= 64;
            if (!second || gated) {
                uint8_t *dst = sm + (second ? kOffTbg : kOffTb);
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int s0 = ch * 8 + 2 * e;
                        float v0 = s0 <= i ? Ts[i * kLd + s0] * beta_s[s0] : 0.f;
                        float v1 = s0 + 1 <= i ? Ts[i * kLd + s0 + 1] * beta_s[s0 + 1] : 0.f;
                        if (second) {
                            v0 *= __expf(L_s[s0]);
                            v1 *= __expf(L_s[s0 + 1]);
                        }
                        w[e] = pack_bf16x2(v0, v1);
                    }
                    *(uint4 *)(dst + sw128_offset(i, ch)) = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
        }
        fence_proxy_async_smem();
        __syncthreads();

        // (6) U^T = V^T Tb^T -> UN (lane = dv);  W^T = K^T Tbg^T -> GW (lane = dk)
        if (tid == 0) {
            tc_fence_after();
            const uint32_t id = idesc_bf16(128, 64, true, false);
            const uint32_t tb = smem_addr(sm + kOffTb), tbg = smem_addr(sm + (gated ? kOffTbg : kOffTb));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_ss(tbase + kColUN, sdesc_sw128(smem_addr(vv) + kk * 2048, 8192, 1024),
                       sdesc_sw128(tb + kk * 32, 16, 1024), id, kk > 0);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_ss(tbase + kColGW, sdesc_sw128(smem_addr(kq) + kk * 2048, 16384, 1024),
                       sdesc_sw128(tbg + kk * 32, 16, 1024), id, kk > 0);
            mma_commit(bar_mma);
        }
        mma_pending = true;
        if (!mbar_wait(bar_mma, mma_phase, kWaitTries, abort_s)) flag_error(p.status, abort_s, kDevTimeout);
        mma_phase ^= 1;
        __syncthreads();
        if (*abort_s) break;
        mma_pending = false;
        tc_fence_after();

        // (7) -W as the MN-major B tile (row dk = this lane); S^T -> bf16 copy
        // (and S <- Gamma_C S when gated)
        const float Lend = L_s[kC - 1];
        {
            float wv[64];
            tmem_ld64f(trow + kColGW, wv);
            uint8_t *NW = sm + kOffNW;
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) w[e] = pack_bf16x2(-wv[ch * 8 + 2 * e], -wv[ch * 8 + 2 * e + 1]);
                *(uint4 *)(NW + sw128_offset(tid, ch)) = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
        {
            const float gC = gated ? __expf(Lend) : 1.f;
            uint32_t r[16], r2[16], pk[16], pl[16];
            for (int c0 = 0; c0 < kD; c0 += 32) {
                tmem_ld16(trow + kColS + c0, r);
                tmem_ld16(trow + kColS + c0 + 16, r2);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    split_pack(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]), pk[j], pl[j]);
                    split_pack(__uint_as_float(r2[2 * j]), __uint_as_float(r2[2 * j + 1]), pk[8 + j], pl[8 + j]);
                }
                tmem_st16(trow + kColSB + c0 / 2, pk);
                tmem_st16(trow + kColSBL + c0 / 2, pl);
                if (gated) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        r[j] = __float_as_uint(__uint_as_float(r[j]) * gC);
                        r2[j] = __float_as_uint(__uint_as_float(r2[j]) * gC);
                    }
                    tmem_st16(trow + kColS + c0, r);
                    tmem_st16(trow + kColS + c0 + 16, r2);
                }
            }
            tmem_wait_st();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        // (8) U'^T = U^T - S^T W^T;  O^T = S^T Q^T
        if (tid == 0) {
            tc_fence_after();
            const uint32_t idU = idesc_bf16(128, 64, false, true);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint64_t bd = sdesc_sw128(smem_addr(sm + kOffNW) + kk * 2048, 8192, 1024);
                mma_ts(tbase + kColUN, tbase + kColSB + kk * 8, bd, idU, 1);
                mma_ts(tbase + kColUN, tbase + kColSBL + kk * 8, bd, idU, 1);
            }
            const uint32_t idO = idesc_bf16(128, nq, false, false);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t a = smem_addr(kq) + (kk >> 2) * 16384 + 64 * 128 + (kk & 3) * 32;
                const uint64_t bd = sdesc_sw128(a, 16, 1024);
                mma_ts(tbase + kColO, tbase + kColSB + kk * 8, bd, idO, kk > 0);
                mma_ts(tbase + kColO, tbase + kColSBL + kk * 8, bd, idO, 1);
            }
            mma_commit(bar_mma);
        }
        mma_pending = true;
        if (!mbar_wait(bar_mma, mma_phase, kWaitTries, abort_s)) flag_error(p.status, abort_s, kDevTimeout);
        mma_phase ^= 1;
        __syncthreads();
        if (*abort_s) break;
        mma_pending = false;
        tc_fence_after();

        // (9) U'^T -> bf16 hi/lo copies (readout; decayed for the state update when
        // gated); gated: O^T columns scaled by Gamma of their readout rows
        {
            // all 64 fp32 columns are read before any lo part overwrites them
            float un[64];
            tmem_ld64f(trow + kColUN, un);
            uint32_t pk[16], pl[16];
            for (int c0 = 0; c0 < kC; c0 += 32) {
#pragma unroll
                for (int j = 0; j < 16; ++j) split_pack(un[c0 + 2 * j], un[c0 + 2 * j + 1], pk[j], pl[j]);
                tmem_st16(trow + kColUB + c0 / 2, pk);
                tmem_st16(trow + kColUBL + c0 / 2, pl);
                if (gated) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int s0 = c0 + 2 * j;
                        split_pack(un[s0] * __expf(Lend - L_s[s0]), un[s0 + 1] * __expf(Lend - L_s[s0 + 1]),
                                   pk[j], pl[j]);
                    }
                    tmem_st16(trow + kColUBD + c0 / 2, pk);
                    tmem_st16(trow + kColUBDL + c0 / 2, pl);
                }
            }
            if (gated) {
                // O^T column i holds S0^T q_i: scale it by Gamma at token i's readout row
                uint32_t r[16];
                for (int c0 = 0; c0 < nq; c0 += 16) {
                    tmem_ld16(trow + kColO + c0, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int i = c0 + j;
                        const float gr = i < ct ? __expf(L_s[i * nh + nh - 1]) : 0.f;
                        r[j] = __float_as_uint(__uint_as_float(r[j]) * gr);
                    }
                    tmem_st16(trow + kColO + c0, r);
                }
            }
            tmem_wait_st();
        }
        tc_fence_before();
        __syncthreads();

        // (10) S^T += U'^T(decayed) K;  O^T += U'^T P^T
        if (tid == 0) {
            tc_fence_after();
            const uint32_t idS = idesc_bf16(128, 128, false, true);
            const uint32_t ubd = gated ? kColUBD : kColUB, ubdl = gated ? kColUBDL : kColUBL;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint64_t bd = sdesc_sw128(smem_addr(kq) + kk * 2048, 16384, 1024);
                mma_ts(tbase + kColS, tbase + ubd + kk * 8, bd, idS, 1);
                mma_ts(tbase + kColS, tbase + ubdl + kk * 8, bd, idS, 1);
            }
            const uint32_t idO = idesc_bf16(128, nq, false, false);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint64_t bd = sdesc_sw128(smem_addr(sm + kOffP) + kk * 32, 16, 1024);
                const uint64_t bdl = sdesc_sw128(smem_addr(sm + kOffPL) + kk * 32, 16, 1024);
                mma_ts(tbase + kColO, tbase + kColUB + kk * 8, bd, idO, 1);
                mma_ts(tbase + kColO, tbase + kColUBL + kk * 8, bd, idO, 1);
                mma_ts(tbase + kColO, tbase + kColUB + kk * 8, bdl, idO, 1);
            }
            mma_commit(bar_mma);
        }
        mma_pending = true;
        if (!mbar_wait(bar_mma, mma_phase, kWaitTries, abort_s)) flag_error(p.status, abort_s, kDevTimeout);
        mma_phase ^= 1;
        __syncthreads();
        if (*abort_s) break;
        mma_pending = false;
        tc_fence_after();
        // stage st is free: prefetch chunk c + 2 into it
        if (c + 2 < p.n_chunks) {
            if (tid == 0) issue_loads(c + 2);
            issued = c + 3;
        }

        // (11) outputs of the chunk's tokens (lane = dv)
        {
            uint32_t r[16];
            for (int c0 = 0; c0 < nq; c0 += 16) {
                tmem_ld16(trow + kColO + c0, r);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int i = c0 + j, t = t0 + i;
                    if (i < ct && t < T)
                        store_out((TOut *)p.o, (((size_t)b * T + t) * p.H + h) * kD + tid, __uint_as_float(r[j]));
                }
            }
        }
        tc_fence_before();
    }

    if (*abort_s) {
        // drain what is still in flight before releasing TMEM and shared memory
        uint32_t no_abort = 0;   // these waits must not be cut short by the flag
        if (mma_pending) mbar_wait(bar_mma, mma_phase ^ 1, kWaitTries, &no_abort);
        for (int cc = landed; cc < issued; ++cc)
            mbar_wait(&bar_tma[cc & 1], (cc >> 1) & 1, kWaitTries, &no_abort);
    } else if (p.h_final) {
        uint32_t r[16];
        for (int c0 = 0; c0 < kD; c0 += 16) {
            tmem_ld16(trow + kColS + c0, r);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j)
                p.h_final[((size_t)bh * kD + c0 + j) * kD + tid] = __uint_as_float(r[j]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, kTmemCols);
}

}  // namespace

bool chunk_tc_supported(const Problem &p)
{
    return p.dtype == DP_BF16 && p.Dk == kD && p.Dv == kD && p.nh >= 1 && p.nh <= 4 && p.T > 0 &&
           tensor_map_encoder() != nullptr;
}

size_t chunk_tc_scratch_bytes(const Problem &) { return 0; }

cudaError_t launch_chunk_tc(const Problem &p)
{
    const int nh = p.nh, ct = kC / nh;
    const cuuint64_t B = p.B, T = p.T, H = p.H;
    CUtensorMap tk, tv, tq;
    const cuuint64_t dk[5] = {kD, (cuuint64_t)nh, H, T, B};
    const cuuint64_t sk[4] = {kD * 2, (cuuint64_t)nh * kD * 2, H * nh * kD * 2, T * H * nh * kD * 2};
    const cuuint32_t bk[5] = {64, (cuuint32_t)nh, 1, (cuuint32_t)ct, 1};
    const cuuint64_t dq[4] = {kD, H, T, B};
    const cuuint64_t sq[3] = {kD * 2, H * kD * 2, T * H * kD * 2};
    const cuuint32_t bq[4] = {64, 1, (cuuint32_t)ct, 1};
    if (!encode(&tk, p.k, 5, dk, sk, bk) || !encode(&tv, p.v, 5, dk, sk, bk) ||
        !encode(&tq, p.q, 4, dq, sq, bq))
        return cudaErrorInvalidValue;
    auto kernel = p.out_dtype == DP_F32 ? chunk_tc_kernel<float> : chunk_tc_kernel<__nv_bfloat16>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    Params pr;
    pr.beta = (const __nv_bfloat16 *)p.beta;
    pr.g = (const __nv_bfloat16 *)p.g;
    pr.h0 = p.h0;
    pr.o = p.o;
    pr.h_final = p.h_final;
    pr.status = p.status;
    pr.T = p.T;
    pr.H = p.H;
    pr.nh = nh;
    pr.ct = ct;
    pr.nq = (ct + 15) & ~15;
    pr.n_chunks = (p.T + ct - 1) / ct;
    kernel<<<p.B * p.H, kThreads, kSmemBytes, p.stream>>>(tk, tv, tq, pr);
    return cudaGetLastError();
}

}  // namespace dp
