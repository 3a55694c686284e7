// Standalone input prologue (dp_prologue): the element-wise maps of the
// DeltaProduct paper's Sec.4 inputs applied to raw projections, written back
// in the input dtype. One warp per key or query row (lane = D/32 consecutive
// elements; the row's sum of squares by a warp reduction), a grid-stride
// loop for betas and gates. The fused kernels apply the same maps (the
// pro_* functions) while loading their inputs.
#include "internal.h"

namespace dp {
namespace {

__device__ __forceinline__ float ld(const float *p, size_t i) { return p[i]; }
__device__ __forceinline__ float ld(const __nv_bfloat16 *p, size_t i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ void st(float *p, size_t i, float x) { p[i] = x; }
__device__ __forceinline__ void st(__nv_bfloat16 *p, size_t i, float x) { p[i] = __float2bfloat16_rn(x); }

// rows [0, n_k) are key rows of k, [n_k, n_k + n_q) query rows of q
template <typename T, int D>
__global__ void __launch_bounds__(256) prologue_rows_kernel(size_t n_k, size_t n_q, const T *k, T *k_out,
                                                             const T *q, T *q_out)
{
    constexpr int E = D / 32;
    const int lane = threadIdx.x & 31;
    const size_t warps = (size_t)gridDim.x * (blockDim.x >> 5);
    for (size_t row = (size_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < n_k + n_q;
         row += warps) {
        const bool key = row < n_k;
        const T *src = key ? k + row * D : q + (row - n_k) * D;
        T *dst = key ? k_out + row * D : q_out + (row - n_k) * D;
        float x[E], ss = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            x[e] = ld(src, lane * E + e);
            if (key) x[e] = pro_silu(x[e]);
            ss = fmaf(x[e], x[e], ss);
        }
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
        const float inv = pro_inv_norm(ss);
#pragma unroll
        for (int e = 0; e < E; ++e) st(dst, lane * E + e, x[e] * inv);
    }
}

template <typename T>
__global__ void prologue_scalars_kernel(size_t n_beta, size_t n_g, int flags, const T *beta, T *beta_out,
                                        const T *g, T *g_out)
{
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_beta + n_g;
         i += (size_t)gridDim.x * blockDim.x) {
        if (i < n_beta) st(beta_out, i, pro_beta(ld(beta, i), flags));
        else st(g_out, i - n_beta, pro_gate(ld(g, i - n_beta), flags));
    }
}

template <typename T, int D>
cudaError_t launch_rows(size_t n_k, size_t n_q, const Problem &p, void *k_out, void *q_out)
{
    const size_t rows = n_k + n_q;
    const unsigned blocks = (unsigned)((rows + 7) / 8 < 152 * 16 ? (rows + 7) / 8 : 152 * 16);
    prologue_rows_kernel<T, D><<<blocks, 256, 0, p.stream>>>(n_k, n_q, (const T *)p.k, (T *)k_out,
                                                             (const T *)p.q, (T *)q_out);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_typed(const Problem &p, void *q_out, void *k_out, void *beta_out, void *g_out)
{
    const int f = p.prologue;
    const size_t tok = (size_t)p.B * p.T * p.H;
    const size_t n_k = (f & DP_PRO_KEY_SILU_L2) ? tok * p.nh : 0, n_q = (f & DP_PRO_QUERY_L2) ? tok : 0;
    cudaError_t e = cudaSuccess;
    if (n_k + n_q > 0) {
        // keys and queries share D = D_k
        e = p.Dk == 32   ? launch_rows<T, 32>(n_k, n_q, p, k_out, q_out)
            : p.Dk == 64 ? launch_rows<T, 64>(n_k, n_q, p, k_out, q_out)
                         : launch_rows<T, 128>(n_k, n_q, p, k_out, q_out);
        if (e != cudaSuccess) return e;
    }
    const size_t n_beta = (f & (DP_PRO_BETA_SIGMOID | DP_PRO_BETA_2SIGMOID)) ? tok * p.nh : 0;
    const size_t n_g = g_out ? tok : 0;
    if (n_beta + n_g > 0) {
        const size_t n = n_beta + n_g;
        const unsigned blocks = (unsigned)((n + 255) / 256 < 152 * 8 ? (n + 255) / 256 : 152 * 8);
        prologue_scalars_kernel<T><<<blocks, 256, 0, p.stream>>>(n_beta, n_g, f, (const T *)p.beta,
                                                                 (T *)beta_out, (const T *)p.g, (T *)g_out);
        e = cudaGetLastError();
    }
    return e;
}

}  // namespace

cudaError_t launch_prologue(const Problem &p, void *q_out, void *k_out, void *beta_out, void *g_out)
{
    return p.dtype == DP_F32 ? launch_typed<float>(p, q_out, k_out, beta_out, g_out)
                             : launch_typed<__nv_bfloat16>(p, q_out, k_out, beta_out, g_out);
}

}  // namespace dp
