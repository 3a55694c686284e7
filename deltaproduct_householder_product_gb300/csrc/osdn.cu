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
// scan is a chain of dependent rows, so the loads are kept far ahead of it:
// keys 32 rows ahead through cp.async, betas a 32-row block ahead.
#include "internal.h"

namespace dp {
namespace {

__device__ __forceinline__ float ld(const float *p, size_t i) { return p[i]; }
__device__ __forceinline__ float ld(const __nv_bfloat16 *p, size_t i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ void st(float *p, size_t i, float x) { p[i] = x; }
__device__ __forceinline__ void st(__nv_bfloat16 *p, size_t i, float x) { p[i] = __float2bfloat16_rn(x); }

// Asynchronous copy of `bytes` (4, 8 or 16) from global to shared memory,
// tracked per thread by commit groups.
// (2 bytes, below cp.async's minimum: an ordinary load and store.)
template <int kBytes>
__device__ __forceinline__ void cp_async(void *smem, const void *gmem)
{
    const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    if constexpr (kBytes == 16)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
    else if constexpr (kBytes >= 4)
        asm volatile("cp.async.ca.shared.global [%0], [%1], %2;" ::"r"(s), "l"(gmem), "n"(kBytes) : "memory");
    else
        *(uint16_t *)smem = *(const uint16_t *)gmem;
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <typename T, int E>
__device__ __forceinline__ void unpack(const uint8_t *src, float (&x)[E])
{
#pragma unroll
    for (int e = 0; e < E; ++e) x[e] = ld((const T *)src, e);
}
template <typename T, int E>
__device__ __forceinline__ void store_row(T *dst, const float (&x)[E])
{
    if constexpr (sizeof(T) == 2 && E == 4) {   // one 8-byte store
        __nv_bfloat162 a = __floats2bfloat162_rn(x[0], x[1]), b = __floats2bfloat162_rn(x[2], x[3]);
        uint2 u;
        u.x = *reinterpret_cast<uint32_t *>(&a);
        u.y = *reinterpret_cast<uint32_t *>(&b);
        *(uint2 *)dst = u;
    } else {
#pragma unroll
        for (int e = 0; e < E; ++e) st(dst, e, x[e]);
    }
}

// The scan of one (batch, head) per warp. Keys stream through a per-lane
// ring of kRing rows in shared memory filled by cp.async, kRing - 1 rows
// ahead (each lane copies and later reads only its own E elements, so no
// barrier is needed, and a slot is refilled a row after its read); the
// betas (and retentions) of the next 32 rows are loaded one per lane a
// block ahead and broadcast by shuffle.
constexpr int kRing = 32;

template <typename T, int DK>
__global__ void __launch_bounds__(128) dscan_kernel(int n_heads, int Tn, int H, int nh, const T *k,
                                                    const T *beta, const T *r, const float *d0, float eta,
                                                    float d_lo, float d_hi, float eps, T *kw,
                                                    float *d_final)
{
    constexpr int E = DK / 32, kB = E * (int)sizeof(T);   // bytes per lane per row
    static_assert(kB == 2 || kB == 4 || kB == 8 || kB == 16, "row piece per lane");
    __shared__ __align__(16) uint8_t ring[4][kRing][32][kB];
    const int w = threadIdx.x >> 5, bh = blockIdx.x * 4 + w, lane = threadIdx.x & 31;
    if (bh >= n_heads) return;
    const int b = bh / H, h = bh - b * H;
    float d[E];
#pragma unroll
    for (int e = 0; e < E; ++e) d[e] = d0 ? d0[(size_t)bh * DK + lane * E + e] : 1.f;

    const int rows = Tn * nh;
    // extended row x -> (token t, key j): offsets of its key and beta
    auto beta_at = [&](int x) { return (((size_t)b * Tn + x / nh) * H + h) * nh + x % nh; };
    auto key_at = [&](int x) { return beta_at(x) * DK + lane * E; };
    // walking a row cursor instead: +1 key within a token, else on to the
    // next token's first key (H n_h rows further, less the n_h - 1 passed)
    struct Cursor {
        size_t off;
        int j;
    };
    const size_t tok_step = ((size_t)H * nh - (nh - 1)) * DK;
    auto advance = [&](Cursor &cu) {
        if (++cu.j < nh) {
            cu.off += DK;
        } else {
            cu.j = 0;
            cu.off += tok_step;
        }
    };
    // per-row scalars of rows x0 .. x0 + 31 (lane l: row x0 + l)
    auto scalars = [&](int x0, float &bt, float &rt) {
        const int x = x0 + lane;
        bt = x < rows ? ld(beta, beta_at(x)) : 0.f;
        rt = (r && x < rows && x % nh == 0) ? ld(r, beta_at(x) / nh) : 1.f;
    };
    // prime the ring: rows 0 .. kRing-2, one commit group per row
    Cursor cx{key_at(0), 0}, cy = cx;   // row x (being scanned) and row x + kRing - 1 (being fetched)
#pragma unroll 1
    for (int x = 0; x < kRing - 1; ++x) {
        if (x < rows) cp_async<kB>(ring[w][x][lane], k + cy.off);
        cp_commit();
        advance(cy);
    }
    float b_cur, r_cur, b_nxt = 0.f, r_nxt = 1.f;
    scalars(0, b_cur, r_cur);
    for (int x0 = 0; x0 < rows; x0 += 32) {
        if (x0 + 32 < rows) scalars(x0 + 32, b_nxt, r_nxt);   // next block, in flight
        const int n = min(32, rows - x0);
        for (int i = 0; i < n; ++i) {
            const int x = x0 + i;
            // row x + kRing - 1 into the slot row x - 1 used (read a row ago;
            // an empty group past the end keeps the count), then wait for row x
            const int y = x + kRing - 1;
            if (y < rows) cp_async<kB>(ring[w][y % kRing][lane], k + cy.off);
            cp_commit();
            advance(cy);
            cp_wait<kRing - 1>();   // groups complete in order: row x has landed
            float kk[E];
            unpack<T, E>(ring[w][x % kRing][lane], kk);
            const float bt = __shfl_sync(0xffffffffu, b_cur, i), keep = __shfl_sync(0xffffffffu, r_cur, i);
            float kt[E], n2 = 0.f, ds = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                kt[e] = d[e] * kk[e];   // the write key, with the current d
                const float s2 = kk[e] * kk[e];
                n2 += s2;
                ds = fmaf(d[e], s2, ds);
            }
            store_row<T, E>(kw + cx.off, kt);
            advance(cx);
#pragma unroll
            for (int m = 16; m >= 1; m >>= 1) {
                n2 += __shfl_xor_sync(0xffffffffu, n2, m);
                ds += __shfl_xor_sync(0xffffffffu, ds, m);
            }
            const float coef = eta * bt * (1.f - bt * ds) / fmaxf(n2, eps);
#pragma unroll
            for (int e = 0; e < E; ++e) d[e] = fminf(fmaxf(fmaf(coef, kk[e] * kk[e], keep * d[e]), d_lo), d_hi);
        }
        b_cur = b_nxt;
        r_cur = r_nxt;
    }
    cp_wait<0>();
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
