// C ABI of libdp.so: argument validation, workspace layout and dispatch.
// See include/dp.h for the contract of every entry point.
#include <string.h>

#include "internal.h"

namespace {

constexpr size_t kStatusBlock = 256;   // status word + padding, start of the workspace

bool supported_dim(int d) { return d == 32 || d == 64 || d == 128; }
bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// The pointer must be usable by a kernel on the current device.
bool device_pointer(const void *p)
{
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

dp_status check_dims(const dp_dims *d, bool decode)
{
    if (!d) return DP_ERR_INVALID_ARG;
    if (d->B < 0 || d->H < 0 || (!decode && d->T < 0)) return DP_ERR_INVALID_ARG;
    if (d->max_seqlen < 0 || (!decode && d->max_seqlen > d->T)) return DP_ERR_INVALID_ARG;
    if (d->dtype != DP_F32 && d->dtype != DP_BF16) return DP_ERR_INVALID_ARG;
    if (d->impl < DP_IMPL_AUTO || d->impl > DP_IMPL_CHUNK_TC) return DP_ERR_INVALID_ARG;
    if (d->out_dtype != d->dtype && d->out_dtype != DP_F32) return DP_ERR_INVALID_ARG;
    if (!supported_dim(d->Dk) || !supported_dim(d->Dv)) return DP_ERR_UNSUPPORTED;
    if (d->nh < 1 || d->nh > 4) return DP_ERR_UNSUPPORTED;
    if ((d->prologue & ~31) != 0 ||
        ((d->prologue & DP_PRO_BETA_SIGMOID) && (d->prologue & DP_PRO_BETA_2SIGMOID)))
        return DP_ERR_INVALID_ARG;
    // indices are formed in 64-bit, but keep every extent within int range
    const long long tok = (long long)d->B * (decode ? 1 : d->T) * d->H;
    if (tok * d->nh * (d->Dk > d->Dv ? d->Dk : d->Dv) > (1ll << 40)) return DP_ERR_UNSUPPORTED;
    return DP_OK;
}

// Required pointer: non-NULL, device-accessible, aligned to `align` bytes.
dp_status check_ptr(const void *p, size_t align)
{
    if (!p) return DP_ERR_INVALID_ARG;
    if (((uintptr_t)p & (align - 1)) != 0) return DP_ERR_ALIGNMENT;
    if (!device_pointer(p)) return DP_ERR_INVALID_ARG;
    return DP_OK;
}

#define DP_TRY(expr)                         \
    do {                                     \
        dp_status s_ = (expr);               \
        if (s_ != DP_OK) return s_;          \
    } while (0)

dp::Problem make_problem(const dp_dims *d, int T)
{
    dp::Problem p;
    memset(&p, 0, sizeof(p));
    p.B = d->B; p.T = T; p.H = d->H; p.Dk = d->Dk; p.Dv = d->Dv; p.nh = d->nh;
    p.dtype = d->dtype;
    p.out_dtype = d->out_dtype;
    p.max_T = d->max_seqlen > 0 ? d->max_seqlen : T;
    p.prologue = d->prologue;
    return p;
}

dp_status check_io(const dp::Problem &p, bool has_g)
{
    const size_t el = p.dtype == DP_F32 ? 4 : 2;
    const bool any = (size_t)p.B * p.H * p.T > 0;
    if (any) {
        DP_TRY(check_ptr(p.q, 16));
        DP_TRY(check_ptr(p.k, 16));
        DP_TRY(check_ptr(p.v, 16));
        DP_TRY(check_ptr(p.o, 16));
        DP_TRY(check_ptr(p.beta, el));
        if (has_g) DP_TRY(check_ptr(p.g, el));
    }
    return DP_OK;
}

dp_status from_cuda(cudaError_t e) { return e == cudaSuccess ? DP_OK : DP_ERR_CUDA; }

bool use_chunk_tc(const dp_dims *d, const dp::Problem &p)
{
    if (d->impl == DP_IMPL_RECURRENT) return false;
    return dp::chunk_tc_supported(p);
}

}  // namespace

extern "C" {

int dp_abi_version(void) { return DP_ABI_VERSION; }

const char *dp_status_string(dp_status s)
{
    switch (s) {
    case DP_OK: return "ok";
    case DP_ERR_INVALID_ARG: return "invalid argument";
    case DP_ERR_UNSUPPORTED: return "unsupported shape or option";
    case DP_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case DP_ERR_WORKSPACE: return "workspace missing or too small";
    case DP_ERR_CUDA: return "CUDA runtime error";
    case DP_ERR_TIMEOUT: return "device-side wait timed out";
    case DP_ERR_DEVICE: return "device reported an inconsistency";
    }
    return "unknown status";
}

dp_status dp_forward_workspace_size(const dp_dims *dims, size_t *bytes)
{
    if (!bytes) return DP_ERR_INVALID_ARG;
    DP_TRY(check_dims(dims, false));
    if (dims->impl == DP_IMPL_CHUNK_TC) {
        dp::Problem p = make_problem(dims, dims->T);
        if (!dp::chunk_tc_supported(p)) return DP_ERR_UNSUPPORTED;
    }
    *bytes = kStatusBlock;
    return DP_OK;
}

dp_status dp_forward_workspace_size_fast(const dp_dims *dims, size_t *bytes)
{
    DP_TRY(dp_forward_workspace_size(dims, bytes));
    dp::Problem p = make_problem(dims, dims->T);
    if (use_chunk_tc(dims, p)) *bytes += (dp::chunk_tc_fast_bytes(p) + 255) & ~(size_t)255;
    return DP_OK;
}

dp_status dp_forward_path(const dp_dims *dims, size_t workspace_bytes, int *path)
{
    if (!path) return DP_ERR_INVALID_ARG;
    DP_TRY(check_dims(dims, false));
    size_t need = 0;
    DP_TRY(dp_forward_workspace_size(dims, &need));
    if (workspace_bytes < need) return DP_ERR_WORKSPACE;
    dp::Problem p = make_problem(dims, dims->T);
    if (!use_chunk_tc(dims, p)) {
        *path = DP_PATH_RECURRENT;
        return DP_OK;
    }
    p.scratch_bytes = workspace_bytes - kStatusBlock;
    return from_cuda(dp::chunk_tc_path(p, path));
}

}  // extern "C"

namespace {
dp_status forward_impl(const dp_dims *dims, const int *cu, const void *q, const void *k, const void *v,
                       const void *beta, const void *g, const float *h0, void *o, float *h_final,
                       void *workspace, size_t workspace_bytes, dp_stream_t stream)
{
    DP_TRY(check_dims(dims, false));
    dp::Problem p = make_problem(dims, dims->T);
    p.cu = cu;
    p.q = q; p.k = k; p.v = v; p.beta = beta; p.g = g; p.h0 = h0; p.o = o;
    p.h_final = h_final;
    p.stream = (cudaStream_t)stream;
    const bool tc = use_chunk_tc(dims, p);
    if (dims->impl == DP_IMPL_CHUNK_TC && !tc) return DP_ERR_UNSUPPORTED;
    DP_TRY(check_io(p, g != nullptr));
    if (h0) DP_TRY(check_ptr(h0, 16));
    if (h_final) DP_TRY(check_ptr(h_final, 16));
    size_t need = 0;
    DP_TRY(dp_forward_workspace_size(dims, &need));
    if (!workspace || workspace_bytes < need) return DP_ERR_WORKSPACE;
    if (!aligned16(workspace)) return DP_ERR_ALIGNMENT;
    if (!device_pointer(workspace)) return DP_ERR_INVALID_ARG;
    p.status = (uint32_t *)workspace;
    p.scratch = (char *)workspace + kStatusBlock;
    p.scratch_bytes = workspace_bytes - kStatusBlock;

    if ((size_t)p.B * p.H == 0) return DP_OK;
    return from_cuda(tc ? dp::launch_chunk_tc(p) : dp::launch_recurrent(p));
}
}  // namespace

extern "C" {

dp_status dp_forward(const dp_dims *dims, const void *q, const void *k, const void *v,
                     const void *beta, const void *g, const float *h0, void *o,
                     float *h_final, void *workspace, size_t workspace_bytes,
                     dp_stream_t stream)
{
    if (dims && dims->max_seqlen != 0) return DP_ERR_INVALID_ARG;   // dense calls: every sequence is T long
    return forward_impl(dims, nullptr, q, k, v, beta, g, h0, o, h_final, workspace, workspace_bytes, stream);
}

dp_status dp_forward_varlen(const dp_dims *dims, const int *cu_seqlens, const void *q, const void *k,
                            const void *v, const void *beta, const void *g, const float *h0, void *o,
                            float *h_final, void *workspace, size_t workspace_bytes, dp_stream_t stream)
{
    DP_TRY(check_dims(dims, false));
    if ((size_t)dims->B * dims->H == 0) return DP_OK;
    if (dims->T > 0 && dims->max_seqlen < 1) return DP_ERR_INVALID_ARG;
    DP_TRY(check_ptr(cu_seqlens, 4));
    // the packed layouts are the dense ones with one batch row of T tokens
    dp_dims flat = *dims;
    return forward_impl(&flat, cu_seqlens, q, k, v, beta, g, h0, o, h_final, workspace, workspace_bytes, stream);
}

dp_status dp_decode_step(const dp_dims *dims, const void *q, const void *k, const void *v,
                         const void *beta, const void *g, float *state, void *o,
                         dp_stream_t stream)
{
    DP_TRY(check_dims(dims, true));
    dp::Problem p = make_problem(dims, 1);
    p.q = q; p.k = k; p.v = v; p.beta = beta; p.g = g; p.o = o;
    p.h0 = state;
    p.h_final = state;
    p.stream = (cudaStream_t)stream;
    p.decode = true;
    if ((size_t)p.B * p.H == 0) return DP_OK;
    DP_TRY(check_io(p, g != nullptr));
    DP_TRY(check_ptr(state, 16));
    return from_cuda(dp::launch_recurrent(p));
}

dp_status dp_state_io(int op, int B, int H, int Dk, int Dv, float *state, void *ext,
                      int ext_dtype, int ext_transposed, dp_stream_t stream)
{
    if (op < DP_STATE_ZERO || op > DP_STATE_EXPORT) return DP_ERR_INVALID_ARG;
    if (B < 0 || H < 0) return DP_ERR_INVALID_ARG;
    if (!supported_dim(Dk) || !supported_dim(Dv)) return DP_ERR_UNSUPPORTED;
    if (ext_dtype != DP_F32 && ext_dtype != DP_BF16) return DP_ERR_INVALID_ARG;
    if ((size_t)B * H == 0) return DP_OK;
    DP_TRY(check_ptr(state, 16));
    if (op != DP_STATE_ZERO) DP_TRY(check_ptr(ext, ext_dtype == DP_F32 ? 4 : 2));
    return from_cuda(dp::launch_state_io(op, B, H, Dk, Dv, state, ext, ext_dtype,
                                         ext_transposed, (cudaStream_t)stream));
}

dp_status dp_test_set_wait_fault(int withhold_first_record, unsigned int flag_wait_polls)
{
    if (withhold_first_record != 0 && withhold_first_record != 1) return DP_ERR_INVALID_ARG;
    dp::set_coop_fault({flag_wait_polls, withhold_first_record});
    return DP_OK;
}

dp_status dp_check_status(const void *workspace, dp_stream_t stream)
{
    if (!workspace) return DP_ERR_INVALID_ARG;
    if (!aligned16(workspace)) return DP_ERR_ALIGNMENT;
    if (!device_pointer(workspace)) return DP_ERR_INVALID_ARG;
    uint32_t word = 0;
    if (cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost,
                        (cudaStream_t)stream) != cudaSuccess)
        return DP_ERR_CUDA;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return DP_ERR_CUDA;
    if (word == dp::kDevOk) return DP_OK;
    // read-and-clear: the next calls start from a clean word
    if (cudaMemsetAsync((void *)workspace, 0, sizeof(word), (cudaStream_t)stream) != cudaSuccess ||
        cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess)
        return DP_ERR_CUDA;
    if (word == dp::kDevTimeout) return DP_ERR_TIMEOUT;
    return DP_ERR_DEVICE;
}

}  // extern "C"

namespace {
dp::BwdProblem make_bwd(const dp_dims *d)
{
    dp::BwdProblem p;
    memset(&p, 0, sizeof(p));
    p.B = d->B; p.T = d->T; p.H = d->H; p.Dk = d->Dk; p.Dv = d->Dv; p.nh = d->nh;
    p.dtype = d->dtype;
    p.do_dtype = d->out_dtype;
    p.max_T = d->max_seqlen > 0 ? d->max_seqlen : d->T;
    return p;
}

// varlen: dims->max_seqlen bounds the packed sequences (checked by check_dims);
// dense calls leave it 0
dp_status check_bwd_dims(const dp_dims *d, bool varlen)
{
    DP_TRY(check_dims(d, false));
    if (d->prologue != 0) return DP_ERR_INVALID_ARG;
    if (d->impl != DP_IMPL_AUTO && d->impl != DP_IMPL_RECURRENT && d->impl != DP_IMPL_CHUNK_TC)
        return DP_ERR_INVALID_ARG;
    if (!varlen && d->max_seqlen != 0) return DP_ERR_INVALID_ARG;
    if (varlen && d->T > 0 && d->max_seqlen < 1) return DP_ERR_INVALID_ARG;
    return DP_OK;
}

size_t bwd_recurrent_need(const dp::BwdProblem &p)
{
    return kStatusBlock + ((dp::backward_scratch_bytes(p) + 255) & ~(size_t)255);
}
size_t bwd_chunk_need(const dp::BwdProblem &p)
{
    return kStatusBlock + ((dp::backward_chunk_scratch_bytes(p) + 255) & ~(size_t)255);
}
// workspace the dims ask for: the recurrent form's, and the chunked form's
// where the shape allows it (AUTO, CHUNK_TC)
size_t bwd_workspace_bytes(const dp_dims *d, const dp::BwdProblem &p)
{
    size_t n = d->impl == DP_IMPL_CHUNK_TC ? 0 : bwd_recurrent_need(p);
    if (d->impl != DP_IMPL_RECURRENT && dp::backward_chunk_shape_ok(p)) {
        const size_t c = bwd_chunk_need(p);
        n = c > n ? c : n;
    }
    return n;
}

dp_status backward_impl(const dp_dims *dims, const int *cu, const void *q, const void *k, const void *v,
                        const void *beta, const void *g, const float *h0, const void *d_o, const float *dh_final,
                        float *dq, float *dk, float *dv, float *dbeta, float *dg, float *dh0, void *workspace,
                        size_t workspace_bytes, dp_stream_t stream)
{
    DP_TRY(check_bwd_dims(dims, cu != nullptr));
    dp::BwdProblem p = make_bwd(dims);
    const size_t el = p.dtype == DP_F32 ? 4 : 2;
    if ((size_t)p.B * p.H * p.T > 0) {
        DP_TRY(check_ptr(q, 16));
        DP_TRY(check_ptr(k, 16));
        DP_TRY(check_ptr(v, 16));
        DP_TRY(check_ptr(beta, el));
        if (g) DP_TRY(check_ptr(g, el));
        DP_TRY(check_ptr(d_o, 16));
        DP_TRY(check_ptr(dq, 16));
        DP_TRY(check_ptr(dk, 16));
        DP_TRY(check_ptr(dv, 16));
        DP_TRY(check_ptr(dbeta, 4));
        if (g) DP_TRY(check_ptr(dg, 4));
    }
    if (cu) DP_TRY(check_ptr(cu, 4));
    if (h0) DP_TRY(check_ptr(h0, 16));
    if (dh_final) DP_TRY(check_ptr(dh_final, 16));
    if (dh0) DP_TRY(check_ptr(dh0, 16));
    p.g = g;
    p.cu = cu;
    // AUTO takes the chunked form for ungated problems with D = 128 (dense
    // or packed) when the workspace holds its records, else the recurrent
    // form; CHUNK_TC also takes gated problems with D = 128
    bool chunked = dims->impl != DP_IMPL_RECURRENT && dp::backward_chunk_supported(p) &&
                   (g == nullptr || dims->impl == DP_IMPL_CHUNK_TC);
    if (dims->impl == DP_IMPL_CHUNK_TC && !chunked) return DP_ERR_UNSUPPORTED;
    if (chunked && dims->impl == DP_IMPL_AUTO && workspace_bytes < bwd_chunk_need(p)) chunked = false;
    const size_t need = chunked ? bwd_chunk_need(p) : bwd_recurrent_need(p);
    if (!workspace || workspace_bytes < need) return DP_ERR_WORKSPACE;
    if (!aligned16(workspace)) return DP_ERR_ALIGNMENT;
    if (!device_pointer(workspace)) return DP_ERR_INVALID_ARG;
    p.q = q; p.k = k; p.v = v; p.beta = beta; p.g = g; p.h0 = h0;
    p.d_o = d_o; p.dh_final = dh_final;
    p.dq = dq; p.dk = dk; p.dv = dv; p.dbeta = dbeta; p.dg = g ? dg : nullptr; p.dh0 = dh0;
    p.cu = cu;
    p.status = (uint32_t *)workspace;
    p.scratch = (char *)workspace + kStatusBlock;
    p.stream = (cudaStream_t)stream;
    if ((size_t)p.B * p.H == 0) return DP_OK;
    return from_cuda(chunked ? dp::launch_backward_chunk(p) : dp::launch_backward(p));
}
}  // namespace

extern "C" {

dp_status dp_backward_workspace_size(const dp_dims *dims, size_t *bytes)
{
    if (!bytes) return DP_ERR_INVALID_ARG;
    DP_TRY(check_bwd_dims(dims, dims && dims->max_seqlen != 0));
    *bytes = bwd_workspace_bytes(dims, make_bwd(dims));
    return DP_OK;
}

dp_status dp_backward(const dp_dims *dims, const void *q, const void *k, const void *v, const void *beta,
                      const void *g, const float *h0, const void *d_o, const float *dh_final, float *dq,
                      float *dk, float *dv, float *dbeta, float *dg, float *dh0, void *workspace,
                      size_t workspace_bytes, dp_stream_t stream)
{
    return backward_impl(dims, nullptr, q, k, v, beta, g, h0, d_o, dh_final, dq, dk, dv, dbeta, dg, dh0,
                         workspace, workspace_bytes, stream);
}

dp_status dp_backward_varlen(const dp_dims *dims, const int *cu_seqlens, const void *q, const void *k,
                             const void *v, const void *beta, const void *g, const float *h0, const void *d_o,
                             const float *dh_final, float *dq, float *dk, float *dv, float *dbeta, float *dg,
                             float *dh0, void *workspace, size_t workspace_bytes, dp_stream_t stream)
{
    if (!dims) return DP_ERR_INVALID_ARG;
    if ((size_t)dims->B * dims->H == 0) return check_bwd_dims(dims, true);
    if (!cu_seqlens) return DP_ERR_INVALID_ARG;
    return backward_impl(dims, cu_seqlens, q, k, v, beta, g, h0, d_o, dh_final, dq, dk, dv, dbeta, dg, dh0,
                         workspace, workspace_bytes, stream);
}

}  // extern "C"

extern "C" dp_status dp_prologue(const dp_dims *dims, const void *q, const void *k, const void *beta, const void *g,
                                 void *q_out, void *k_out, void *beta_out, void *g_out, dp_stream_t stream)
{
    DP_TRY(check_dims(dims, false));
    if (dims->max_seqlen != 0) return DP_ERR_INVALID_ARG;
    dp::Problem p = make_problem(dims, dims->T);
    const int f = dims->prologue;
    const size_t el = p.dtype == DP_F32 ? 4 : 2;
    if ((size_t)p.B * p.T * p.H > 0) {
        if (f & DP_PRO_KEY_SILU_L2) {
            DP_TRY(check_ptr(k, 16));
            DP_TRY(check_ptr(k_out, 16));
        }
        if (f & DP_PRO_QUERY_L2) {
            DP_TRY(check_ptr(q, 16));
            DP_TRY(check_ptr(q_out, 16));
        }
        if (f & (DP_PRO_BETA_SIGMOID | DP_PRO_BETA_2SIGMOID)) {
            DP_TRY(check_ptr(beta, el));
            DP_TRY(check_ptr(beta_out, el));
        }
        if ((f & DP_PRO_GATE_SIGMOID) && g) DP_TRY(check_ptr(g_out, el));
        if ((f & DP_PRO_GATE_SIGMOID) && g) DP_TRY(check_ptr(g, el));
    }
    p.q = q; p.k = k; p.beta = beta; p.g = (f & DP_PRO_GATE_SIGMOID) ? g : nullptr;
    p.stream = (cudaStream_t)stream;
    if ((size_t)p.B * p.T * p.H == 0 || f == 0) return DP_OK;
    return from_cuda(dp::launch_prologue(p, q_out, k_out, beta_out, p.g ? g_out : nullptr));
}

extern "C" dp_status dp_osdn_write_keys(const dp_dims *dims, const void *k, const void *beta, const void *r,
                                        const float *d0, float eta, float d_lo, float d_hi, float eps, void *kw,
                                        float *d_final, dp_stream_t stream)
{
    DP_TRY(check_dims(dims, false));
    if (dims->max_seqlen != 0 || dims->prologue != 0) return DP_ERR_INVALID_ARG;
    if (!(d_lo > 0.f) || !(d_hi >= d_lo) || !(eps > 0.f) || !(eta >= 0.f)) return DP_ERR_INVALID_ARG;
    dp::Problem p = make_problem(dims, dims->T);
    const size_t el = p.dtype == DP_F32 ? 4 : 2;
    if ((size_t)p.B * p.T * p.H > 0) {
        DP_TRY(check_ptr(k, 16));
        DP_TRY(check_ptr(beta, el));
        DP_TRY(check_ptr(kw, 16));
        if (r) DP_TRY(check_ptr(r, el));
    }
    if (d0) DP_TRY(check_ptr(d0, 16));
    if (d_final) DP_TRY(check_ptr(d_final, 16));
    p.k = k;
    p.beta = beta;
    p.stream = (cudaStream_t)stream;
    if ((size_t)p.B * p.H == 0) return DP_OK;
    const dp::OsdnScan sc{eta, d_lo, d_hi, eps};
    return from_cuda(dp::launch_osdn_dscan(p, r, d0, sc, kw, d_final));
}

extern "C" dp_status dp_forward_write_keys(const dp_dims *dims, const void *q, const void *k, const void *kw,
                                           const void *v, const void *beta, const void *g, const float *h0,
                                           void *o, float *h_final, void *workspace, size_t workspace_bytes,
                                           dp_stream_t stream)
{
    DP_TRY(check_dims(dims, false));
    if (dims->max_seqlen != 0 || (dims->prologue & DP_PRO_KEY_SILU_L2)) return DP_ERR_INVALID_ARG;
    dp::Problem p = make_problem(dims, dims->T);
    p.q = q; p.k = k; p.v = v; p.beta = beta; p.g = g; p.h0 = h0; p.o = o; p.h_final = h_final;
    p.kw = kw;
    p.stream = (cudaStream_t)stream;
    DP_TRY(check_io(p, g != nullptr));
    if ((size_t)p.B * p.H * p.T > 0) DP_TRY(check_ptr(kw, 16));
    if (h0) DP_TRY(check_ptr(h0, 16));
    if (h_final) DP_TRY(check_ptr(h_final, 16));
    size_t need = 0;
    DP_TRY(dp_forward_workspace_size(dims, &need));
    if (!workspace || workspace_bytes < need) return DP_ERR_WORKSPACE;
    if (!aligned16(workspace)) return DP_ERR_ALIGNMENT;
    if (!device_pointer(workspace)) return DP_ERR_INVALID_ARG;
    p.status = (uint32_t *)workspace;
    p.scratch = (char *)workspace + kStatusBlock;
    p.scratch_bytes = workspace_bytes - kStatusBlock;
    // the chunk path takes write keys in its split modes (per-chunk records
    // in the workspace), without a prologue; otherwise the recurrent kernel
    bool tc = dims->impl != DP_IMPL_RECURRENT && dp::chunk_tc_supported(p) && p.prologue == 0 && p.T > 0;
    if (tc) {
        int path = DP_PATH_CHUNK_FUSED;
        if (dp::chunk_tc_path(p, &path) != cudaSuccess) return DP_ERR_CUDA;
        tc = path != DP_PATH_CHUNK_FUSED;
    }
    if (dims->impl == DP_IMPL_CHUNK_TC && !tc) return DP_ERR_UNSUPPORTED;
    if ((size_t)p.B * p.H == 0) return DP_OK;
    return from_cuda(tc ? dp::launch_chunk_tc(p) : dp::launch_recurrent(p));
}
