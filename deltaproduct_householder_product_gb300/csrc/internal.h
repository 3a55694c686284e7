// Internal declarations shared by the translation units of libdp.so.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dp.h"

namespace dp {

// One validated forward / decode problem (device pointers, row-major layouts
// as documented in dp.h).
struct Problem {
    int B, T, H, Dk, Dv, nh;
    int dtype;                 // dp_dtype of the inputs
    int out_dtype;             // dp_dtype of o
    const void *q, *k, *v, *beta, *g;
    const float *h0;
    void *o;
    float *h_final;
    uint32_t *status;          // device status word (may be NULL for decode)
    const int *cu;             // packed sequences: int32 [B+1] token offsets (NULL: dense [B,T] layout)
    int max_T;                 // longest sequence (T for dense calls)
    int prologue;              // dp_prologue_flags applied to the inputs on load
    const void *kw;            // OSDN write keys (layout of k), or NULL: write with k
    void *scratch;             // workspace bytes after the status block
    size_t scratch_bytes;
    cudaStream_t stream;
    bool decode;               // dp_decode_step: launched as a programmatic dependent launch
};

// Sequential (token by token) SIMT kernel: any supported D_k, D_v, n_h and
// dtype. Also serves dp_decode_step (T = 1, state in place).
cudaError_t launch_recurrent(const Problem &p);

// Tensor-core chunked kernel (tcgen05 / TMEM / TMA): bf16, D_k = D_v = 128.
bool chunk_tc_supported(const Problem &p);
// Workspace bytes (after the status block) of the per-chunk records that
// let launch_chunk_tc split into a parallel prep kernel and the state-pass
// kernel; with less scratch it runs the fused single kernel.
size_t chunk_tc_records_bytes(const Problem &p);
// Workspace bytes (after the status block) of the fastest way to run this
// problem on the current device: the records, or the segmented mode's
// larger workspace where that mode applies.
size_t chunk_tc_fast_bytes(const Problem &p);
// Which way launch_chunk_tc runs this problem with p.scratch_bytes of scratch
// (a dp_path value).
cudaError_t chunk_tc_path(const Problem &p, int *path);
cudaError_t launch_chunk_tc(const Problem &p);
// Fault-injection setting of the cooperative mode (dp_test_set_wait_fault):
// flag_tries = polls of a record flag before the wait expires (0: the
// default, seconds); withhold_first = the prep CTAs never publish the first
// record, so the state pass's wait for it expires. Process-wide.
struct CoopFault {
    uint32_t flag_tries;
    int withhold_first;
};
CoopFault coop_fault();
void set_coop_fault(CoopFault f);

// One validated backward problem (dp_backward; layouts in dp.h).
struct BwdProblem {
    int B, T, H, Dk, Dv, nh;
    int dtype;                 // dp_dtype of q, k, v, beta, g
    int do_dtype;              // dp_dtype of d_o
    const void *q, *k, *v, *beta, *g;
    const float *h0;
    const void *d_o;
    const float *dh_final;
    float *dq, *dk, *dv, *dbeta, *dg, *dh0;
    const int *cu;             // packed sequences: int32 [B+1] token offsets (NULL: dense)
    int max_T;                 // longest sequence (T for dense calls)
    uint32_t *status;          // device status word
    void *scratch;             // checkpoint area (backward_scratch_bytes)
    cudaStream_t stream;
};

// Recurrent backward on CUDA cores: checkpoints every
// backward_segment_tokens(Dk) tokens in the scratch area.
int backward_segment_tokens(int Dk);
size_t backward_scratch_bytes(const BwdProblem &p);
cudaError_t launch_backward(const BwdProblem &p);
// Chunked backward (ungated, dense, D_k = D_v = 128): per-chunk records and
// the chunk-boundary states and gradients in the scratch area.
bool backward_chunk_shape_ok(const BwdProblem &p);   // dims only (g not known)
bool backward_chunk_supported(const BwdProblem &p);  // gated or not (AUTO takes it ungated only)
size_t backward_chunk_scratch_bytes(const BwdProblem &p);
cudaError_t launch_backward_chunk(const BwdProblem &p);

cudaError_t launch_state_io(int op, int B, int H, int Dk, int Dv, float *state,
                            void *ext, int ext_dtype, int ext_transposed,
                            cudaStream_t stream);

// OSDN phase 1 (dp_osdn_write_keys): the preconditioner scan over the
// extended rows, emitting the write keys k~ = d (.) k.
struct OsdnScan {
    float eta, d_lo, d_hi, eps;
};
cudaError_t launch_osdn_dscan(const Problem &p, const void *r, const float *d0, const OsdnScan &sc, void *kw,
                              float *d_final);

// Standalone input prologue (dp_prologue), dense layouts.
cudaError_t launch_prologue(const Problem &p, void *q_out, void *k_out, void *beta_out, void *g_out);

// ---- input prologue maps (dp_prologue_flags), fp32, shared by every kernel
__device__ __forceinline__ float pro_sigmoid(float x) { return 1.f / (1.f + expf(-x)); }
// Key rows: SiLU and the reciprocal norm with the hardware approximations
// (relative error ~1e-6, far below the bf16 rounding the mapped rows get as
// tensor-core operands); the maps sit next to the chunk kernel's MMA chain.
__device__ __forceinline__ float pro_silu(float x) { return __fdividef(x, 1.f + __expf(-x)); }
__device__ __forceinline__ float pro_inv_norm(float ss) { return ss > 0.f ? rsqrtf(ss) : 0.f; }
__device__ __forceinline__ float pro_beta(float x, int flags)
{
    if (flags & DP_PRO_BETA_SIGMOID) return pro_sigmoid(x);
    if (flags & DP_PRO_BETA_2SIGMOID) return 2.f * pro_sigmoid(x);
    return x;
}
__device__ __forceinline__ float pro_gate(float x, int flags)
{
    return (flags & DP_PRO_GATE_SIGMOID) ? pro_sigmoid(x) : x;
}
// log of the gate, clamped at -80 (e^-80 stands in for a gate of 0); with
// the sigmoid map, log sigmoid(x) = -softplus(-x) without forming sigmoid(x)
__device__ __forceinline__ float pro_log_gate(float x, int flags)
{
    if (flags & DP_PRO_GATE_SIGMOID) return fmaxf(-(fmaxf(-x, 0.f) + log1pf(expf(-fabsf(x)))), -80.f);
    return fmaxf(logf(x), -80.f);
}

// Device status codes written into the status word (first one wins).
enum : uint32_t { kDevOk = 0, kDevTimeout = 1, kDevBadState = 2 };

// The token range of sequence b: token t (0 <= t < len) sits at row
// (b_map * T + t0 + t) of the [.., T, H, ..] layouts. Dense calls: b_map =
// b, t0 = 0, len = T. Packed calls: b_map = 0, t0 = cu[b], len = cu[b+1] -
// cu[b], after checking cu[b] <= cu[b+1] <= T, len <= max_len, cu[0] = 0
// and cu[N] = T; a sequence that fails the check gets ok = false and len = 0
// (nothing of it is read or written).
struct SeqRange {
    int b_map, t0, len;
    bool ok;
};

__device__ __forceinline__ SeqRange seq_range(const int *cu, int b, int N, int T, int max_len)
{
    if (!cu) return {b, 0, T, true};
    const int a = cu[b], e = cu[b + 1];
    const bool ok = 0 <= a && a <= e && e <= T && e - a <= max_len && (b > 0 || a == 0) &&
                    (b < N - 1 || e == T);
    return ok ? SeqRange{0, a, e - a, true} : SeqRange{0, 0, 0, false};
}

__device__ __forceinline__ void report_bad_sequence(uint32_t *status)
{
    if (status) atomicCAS(status, 0u, kDevBadState);
}

}  // namespace dp
