// Token-by-token DeltaProduct recurrence on CUDA cores, fp32 arithmetic.
//
// DeltaProduct paper, Sec.4 Eq.(3) and the gated per-token pseudocode
// (Sec.4, Appendix B.1): H <- g H; for each of the n_h steps
// e = v - H^T k, H <- H + beta k e^T; then o = H^T q.
//
// Serves four calls: the fp32 path of dp_forward (and any head size the
// tensor-core kernel does not take), dp_decode_step (T = 1 with the state
// updated in place), dp_forward_write_keys (the OSDN variant: the state is
// written along the write key k~ while the error still reads with k), and
// the state import/export of dp_state_io.
//
// Packed variable-length calls (cu != NULL): CTA row b is sequence b, whose
// tokens are found through seq_range.
//
// Work split: one CTA owns a 32-column slice of one (batch, head) state and
// keeps it in registers for the whole sequence: 4 warps x 32 lanes, lane =
// value column, warp w = a contiguous block of D_k/4 key rows. A matvec
// H^T x is a per-thread partial dot over its rows followed by a 4-way
// shared-memory reduction across the warps.
#include "internal.h"

namespace dp {
namespace {

constexpr int kWarps = 4;
constexpr int kCols = 32;

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void from_f(float *p, float x) { *p = x; }
// x rounded to T's precision (the identity for float)
template <typename T> __device__ __forceinline__ float round_to(float x) { return x; }
template <> __device__ __forceinline__ float round_to<__nv_bfloat16>(float x)
{
    return __bfloat162float(__float2bfloat16_rn(x));
}
__device__ __forceinline__ void from_f(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

// kExtra: the input prologue or write keys are in use (the plain
// instantiation carries neither, for the decode step's latency).
template <int DK, typename TIn, typename TOut, bool kExtra>
__global__ void __launch_bounds__(kWarps * 32)
recurrent_kernel(int T, int H, int Dv, int nh, const int *cu, int N, int max_T, int pro, uint32_t *status,
                 const TIn *__restrict__ q, const TIn *__restrict__ k,
                 const TIn *__restrict__ v, const TIn *__restrict__ beta,
                 const TIn *__restrict__ g, const float *h0, TOut *__restrict__ o,
                 float *h_final, const TIn *__restrict__ kw)
{
    constexpr int R = DK / kWarps;            // key rows per warp
    __shared__ float kbuf[2][DK];
    __shared__ float xrows[5][DK];      // plain instantiation: the token's n_h keys and its query
    __shared__ float kwbuf[2][DK];      // OSDN write keys (kw != NULL)
    __shared__ float part[2][kWarps][kCols];
    __shared__ float nred[2][kWarps];   // prologue: partial sums of squares

    // Launched with programmatic stream serialization (the decode step), a
    // kernel may start while the one before it on the stream finishes: it
    // waits for that grid's completion and memory before touching anything,
    // and lets the next launch get resident right away. Without the launch
    // attribute both instructions do nothing.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int bh = blockIdx.x;                // b * H + h
    const int b = bh / H, h = bh - b * H;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int col = blockIdx.y * kCols + lane;
    const int row0 = w * R;
    const size_t state_base = (size_t)bh * DK * Dv;
    const SeqRange sq = seq_range(cu, b, N, T, max_T);
    if (!sq.ok) {   // nothing of this sequence is touched
        if (threadIdx.x == 0 && blockIdx.y == 0) report_bad_sequence(status);
        return;
    }

    float S[R];
#pragma unroll
    for (int r = 0; r < R; ++r)
        S[r] = h0 ? h0[state_base + (size_t)(row0 + r) * Dv + col] : 0.f;

    int buf = 0;   // alternating buffers: one barrier per matvec
    for (int t = 0; t < sq.len; ++t) {
        const size_t tok = ((size_t)sq.b_map * T + sq.t0 + t) * H + h;
        if (!kExtra) {
            // every row of the token (n_h keys, the query) and this thread's
            // values and betas in one round of loads, so that the n_h + 1
            // matvecs wait on no global load (the decode step's latency)
            if (threadIdx.x < DK) {
                for (int j = 0; j < nh; ++j) xrows[j][threadIdx.x] = to_f(k[(tok * nh + j) * DK + threadIdx.x]);
                xrows[nh][threadIdx.x] = to_f(q[tok * DK + threadIdx.x]);
            }
            float vj[4], bj[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (j < nh) {
                    vj[j] = to_f(v[(tok * nh + j) * Dv + col]);
                    bj[j] = to_f(beta[tok * nh + j]);
                }
            const float gt = g ? to_f(g[tok]) : 1.f;
            __syncthreads();
            if (g) {
#pragma unroll
                for (int r = 0; r < R; ++r) S[r] *= gt;
            }
#pragma unroll
            for (int j = 0; j <= 4; ++j) {
                if (j > nh) break;
                const float *x = xrows[j];
                float a4[4] = {0.f, 0.f, 0.f, 0.f};   // four independent chains
#pragma unroll
                for (int r = 0; r < R; ++r) a4[r & 3] = fmaf(S[r], x[row0 + r], a4[r & 3]);
                part[buf][w][lane] = (a4[0] + a4[1]) + (a4[2] + a4[3]);
                __syncthreads();
                float hx = 0.f;
#pragma unroll
                for (int i = 0; i < kWarps; ++i) hx += part[buf][i][lane];
                if (j < nh) {
                    const float e = bj[j] * (vj[j] - hx);
#pragma unroll
                    for (int r = 0; r < R; ++r) S[r] = fmaf(x[row0 + r], e, S[r]);
                } else if (w == 0) {
                    from_f(o + tok * Dv + col, hx);
                }
                buf ^= 1;
            }
            continue;
        }
        if (g) {
            const float gt = kExtra ? pro_gate(to_f(g[tok]), pro) : to_f(g[tok]);
#pragma unroll
            for (int r = 0; r < R; ++r) S[r] *= gt;
        }
        for (int j = 0; j <= nh; ++j) {
            // j < nh: one Householder step with key k_{t,j}; j == nh: readout with q_t
            const TIn *x = (j < nh) ? k + (tok * nh + j) * DK : q + tok * DK;
            // prologue: SiLU + L2 normalisation of keys, L2 of queries, each
            // rounded to the input dtype like a given input (DK <= threads)
            const bool silu = kExtra && j < nh && (pro & DP_PRO_KEY_SILU_L2);
            const bool norm = kExtra && (silu || (j == nh && (pro & DP_PRO_QUERY_L2)));
            float xv = 0.f;
            if (threadIdx.x < DK) {
                xv = to_f(x[threadIdx.x]);
                if (silu) xv = pro_silu(xv);
            }
            if (norm) {
                float ss = xv * xv;
#pragma unroll
                for (int m = 16; m >= 1; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
                if (lane == 0) nred[buf][w] = ss;
                __syncthreads();
                float tot = 0.f;
#pragma unroll
                for (int i = 0; i < kWarps; ++i) tot += nred[buf][i];
                xv = round_to<TIn>(xv * pro_inv_norm(tot));
            }
            if (threadIdx.x < DK) {
                kbuf[buf][threadIdx.x] = xv;
                if (kExtra && kw && j < nh) kwbuf[buf][threadIdx.x] = to_f(kw[(tok * nh + j) * DK + threadIdx.x]);
            }
            __syncthreads();
            float a4[4] = {0.f, 0.f, 0.f, 0.f};   // the plain instantiation's summation order
#pragma unroll
            for (int r = 0; r < R; ++r) a4[r & 3] = fmaf(S[r], kbuf[buf][row0 + r], a4[r & 3]);
            part[buf][w][lane] = (a4[0] + a4[1]) + (a4[2] + a4[3]);
            __syncthreads();
            float hx = 0.f;
#pragma unroll
            for (int i = 0; i < kWarps; ++i) hx += part[buf][i][lane];
            if (j < nh) {
                const float vj = to_f(v[(tok * nh + j) * Dv + col]);
                const float bj = kExtra ? pro_beta(to_f(beta[tok * nh + j]), pro) : to_f(beta[tok * nh + j]);
                const float e = bj * (vj - hx);
                const float *wk = (kExtra && kw) ? kwbuf[buf] : kbuf[buf];   // the write direction
#pragma unroll
                for (int r = 0; r < R; ++r) S[r] = fmaf(wk[row0 + r], e, S[r]);
            } else if (w == 0) {
                from_f(o + tok * Dv + col, hx);
            }
            buf ^= 1;
        }
    }
    if (h_final) {
#pragma unroll
        for (int r = 0; r < R; ++r)
            h_final[state_base + (size_t)(row0 + r) * Dv + col] = S[r];
    }
}

template <int DK, typename TIn, typename TOut>
void launch_dk(const Problem &p, dim3 grid, dim3 block)
{
    const TIn *q = (const TIn *)p.q, *k = (const TIn *)p.k, *v = (const TIn *)p.v;
    const TIn *be = (const TIn *)p.beta, *g = (const TIn *)p.g, *kw = (const TIn *)p.kw;
    TOut *o = (TOut *)p.o;
    auto kernel = (p.prologue != 0 || p.kw != nullptr) ? recurrent_kernel<DK, TIn, TOut, true>
                                                       : recurrent_kernel<DK, TIn, TOut, false>;
    if (!p.decode) {
        kernel<<<grid, block, 0, p.stream>>>(p.T, p.H, p.Dv, p.nh, p.cu, p.B, p.max_T, p.prologue, p.status, q, k, v,
                                             be, g, p.h0, o, p.h_final, kw);
        return;
    }
    // decode step: programmatic dependent launch, so that consecutive steps
    // (one launch each, in a loop or a captured graph) overlap their launch
    // latency with the step before (see griddepcontrol in the kernel)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = p.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaLaunchKernelEx(&cfg, kernel, p.T, p.H, p.Dv, p.nh, p.cu, p.B, p.max_T, p.prologue, p.status, q, k, v, be, g,
                       p.h0, o, p.h_final, kw);
}

template <typename TIn, typename TOut>
cudaError_t launch_typed(const Problem &p)
{
    dim3 grid(p.B * p.H, p.Dv / kCols), block(kWarps * 32);
    switch (p.Dk) {
    case 32: launch_dk<32, TIn, TOut>(p, grid, block); break;
    case 64: launch_dk<64, TIn, TOut>(p, grid, block); break;
    default: launch_dk<128, TIn, TOut>(p, grid, block); break;
    }
    return cudaGetLastError();
}

// ---------------------------------------------------------------- state I/O
template <typename TExt>
__global__ void state_io_kernel(int op, size_t n, int Dk, int Dv, float *state, TExt *ext,
                                int transposed)
{
    const size_t per = (size_t)Dk * Dv;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
         i += (size_t)gridDim.x * blockDim.x) {
        const size_t head = i / per, rem = i - head * per;
        const int r = (int)(rem / Dv), c = (int)(rem - (size_t)r * Dv);
        const size_t e = transposed ? head * per + (size_t)c * Dk + r : i;
        if (op == DP_STATE_IMPORT) state[i] = to_f(ext[e]);
        else from_f(ext + e, state[i]);
    }
}

}  // namespace

cudaError_t launch_recurrent(const Problem &p)
{
    if (p.B * p.H == 0) return cudaSuccess;
    if (p.dtype == DP_F32) return launch_typed<float, float>(p);
    if (p.out_dtype == DP_F32) return launch_typed<__nv_bfloat16, float>(p);
    return launch_typed<__nv_bfloat16, __nv_bfloat16>(p);
}

cudaError_t launch_state_io(int op, int B, int H, int Dk, int Dv, float *state, void *ext,
                            int ext_dtype, int ext_transposed, cudaStream_t stream)
{
    const size_t n = (size_t)B * H * Dk * Dv;
    if (n == 0) return cudaSuccess;
    if (op == DP_STATE_ZERO) return cudaMemsetAsync(state, 0, n * sizeof(float), stream);
    const int threads = 256;
    const int blocks = (int)((n + threads - 1) / threads < 4096 ? (n + threads - 1) / threads : 4096);
    if (ext_dtype == DP_F32)
        state_io_kernel<float><<<blocks, threads, 0, stream>>>(op, n, Dk, Dv, state, (float *)ext, ext_transposed);
    else
        state_io_kernel<__nv_bfloat16><<<blocks, threads, 0, stream>>>(op, n, Dk, Dv, state, (__nv_bfloat16 *)ext, ext_transposed);
    return cudaGetLastError();
}

}  // namespace dp
