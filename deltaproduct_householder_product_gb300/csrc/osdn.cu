// OSDN write keys, phase 1: the online preconditioner scan (OSDN paper,
// Alg.1 and Eq.(3); APF retention, Sec.4.4).
//
// Per (batch, head), over the extended rows in order (T tokens x n_h keys):
//   emit k~ = d (.) k with the current d;
//   s = k (.) k, nbar = max(||k||^2, eps), a = beta <d, s>;
//   d <- clamp(r d + eta beta (1 - a) / nbar * s, d_lo, d_hi)
// with r the token's retention on its first row (1 without APF). The scan
// reads only keys, betas and retentions, never the state, so it runs apart
// from (and before) the recurrence.
//
// One warp per (batch, head): lane = D_k/32 consecutive coordinates of d,
// kept in registers; both dot products come from one 5-step butterfly. The
// next row's key and beta are fetched while the current row is processed.
#include "internal.h"

namespace dp {
namespace {

__device__ __forceinline__ float ld(const float *p, size_t i) { return p[i]; }
__device__ __forceinline__ float ld(const __nv_bfloat16 *p, size_t i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ void st(float *p, size_t i, float x) { p[i] = x; }
__device__ __forceinline__ void st(__nv_bfloat16 *p, size_t i, float x) { p[i] = __float2bfloat16_rn(x); }

template <typename T, int DK>
__global__ void __launch_bounds__(128) dscan_kernel(int n_heads, int Tn, int H, int nh, const T *k,
                                                    const T *beta, const T *r, const float *d0, float eta,
                                                    float d_lo, float d_hi, float eps, T *kw,
                                                    float *d_final)
{
    constexpr int E = DK / 32;
    const int bh = blockIdx.x * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (bh >= n_heads) return;
    const int b = bh / H, h = bh - b * H;
    float d[E];
#pragma unroll
    for (int e = 0; e < E; ++e) d[e] = d0 ? d0[(size_t)bh * DK + lane * E + e] : 1.f;

    const int rows = Tn * nh;
    // extended row x -> (token t, key j); element offset of its key
    auto key_at = [&](int x) { return ((((size_t)b * Tn + x / nh) * H + h) * nh + x % nh) * DK + lane * E; };
    auto beta_at = [&](int x) { return (((size_t)b * Tn + x / nh) * H + h) * nh + x % nh; };
    float kn[E], bn = 0.f;
    if (rows > 0) {
#pragma unroll
        for (int e = 0; e < E; ++e) kn[e] = ld(k, key_at(0) + e);
        bn = ld(beta, beta_at(0));
    }
    for (int x = 0; x < rows; ++x) {
        float kk[E];
#pragma unroll
        for (int e = 0; e < E; ++e) kk[e] = kn[e];
        const float bt = bn;
        if (x + 1 < rows) {   // the next row, in flight while this one is scanned
#pragma unroll
            for (int e = 0; e < E; ++e) kn[e] = ld(k, key_at(x + 1) + e);
            bn = ld(beta, beta_at(x + 1));
        }
        const size_t ko = key_at(x);
        float n = 0.f, ds = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            st(kw, ko + e, d[e] * kk[e]);   // the write key, with the current d
            const float s = kk[e] * kk[e];
            n += s;
            ds = fmaf(d[e], s, ds);
        }
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) {
            n += __shfl_xor_sync(0xffffffffu, n, m);
            ds += __shfl_xor_sync(0xffffffffu, ds, m);
        }
        const float coef = eta * bt * (1.f - bt * ds) / fmaxf(n, eps);
        const float keep = (r && x % nh == 0) ? ld(r, beta_at(x) / nh) : 1.f;
#pragma unroll
        for (int e = 0; e < E; ++e) d[e] = fminf(fmaxf(fmaf(coef, kk[e] * kk[e], keep * d[e]), d_lo), d_hi);
    }
    if (d_final) {
#pragma unroll
        for (int e = 0; e < E; ++e) d_final[(size_t)bh * DK + lane * E + e] = d[e];
    }
}

template <typename T>
cudaError_t launch_typed(const Problem &p, const void *r, const float *d0, const OsdnScan &sc, void *kw,
                         float *d_final)
{
    const int n_heads = p.B * p.H;
    const unsigned blocks = (unsigned)((n_heads + 3) / 4);
    const T *k = (const T *)p.k, *be = (const T *)p.beta, *rr = (const T *)r;
    switch (p.Dk) {
    case 32:
        dscan_kernel<T, 32><<<blocks, 128, 0, p.stream>>>(n_heads, p.T, p.H, p.nh, k, be, rr, d0, sc.eta, sc.d_lo,
                                                          sc.d_hi, sc.eps, (T *)kw, d_final);
        break;
    case 64:
        dscan_kernel<T, 64><<<blocks, 128, 0, p.stream>>>(n_heads, p.T, p.H, p.nh, k, be, rr, d0, sc.eta, sc.d_lo,
                                                          sc.d_hi, sc.eps, (T *)kw, d_final);
        break;
    default:
        dscan_kernel<T, 128><<<blocks, 128, 0, p.stream>>>(n_heads, p.T, p.H, p.nh, k, be, rr, d0, sc.eta,
                                                           sc.d_lo, sc.d_hi, sc.eps, (T *)kw, d_final);
        break;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_osdn_dscan(const Problem &p, const void *r, const float *d0, const OsdnScan &sc, void *kw,
                              float *d_final)
{
    return p.dtype == DP_F32 ? launch_typed<float>(p, r, d0, sc, kw, d_final)
                             : launch_typed<__nv_bfloat16>(p, r, d0, sc, kw, d_final);
}

}  // namespace dp
