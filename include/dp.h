/*
 * dp.h -- C ABI of the GB300 DeltaProduct forward library (libdp.so).
 *
 * The operation (DeltaProduct: Improving State-Tracking in Linear RNNs via
 * Householder Products, Sec.4 Eq.(2)-(3), the gated variant of Sec.4 and the
 * per-token pseudocode of Sec.4 / Appendix B.1): for every batch b, head h
 * and token t, with the D_k x D_v matrix state H,
 *
 *     H <- g_t H                                   (optional gate, once per token)
 *     for j = 1..n_h:  H <- H + beta_{t,j} k_{t,j} (v_{t,j} - H^T k_{t,j})^T
 *                    (= (I - beta k k^T) H + beta k v^T, a generalised Householder step)
 *     o_t = H^T q_t                                (readout of the post-update state)
 *
 * Keys are expected unit-norm and beta in [0,1] or [0,2]; the library does
 * not renormalise or clamp (those are properties of the caller's inputs).
 *
 * Memory: every pointer is a DEVICE pointer on the current CUDA device,
 * owned by the caller. The library allocates no device memory and keeps no
 * state between calls; all work is enqueued asynchronously on `stream`.
 * Layouts are contiguous row-major:
 *     q    [B, T, H, D_k]          k    [B, T, H, n_h, D_k]
 *     v    [B, T, H, n_h, D_v]     beta [B, T, H, n_h]
 *     g    [B, T, H]  (NULL: ungated)
 *     o    [B, T, H, D_v]
 *     state (h0, h_final, decode state) [B, H, D_k, D_v], always fp32.
 * q, k, v, beta and g share the element type `dims->dtype`; o has type
 * `dims->out_dtype` (the input type, or fp32 with bf16 inputs: an fp32 o
 * carries the kernel's fp32 accumulation without a final bf16 rounding).
 *
 * Errors: every entry point validates its arguments on the host first and
 * returns a non-zero dp_status without enqueuing anything when a check
 * fails (outputs untouched). A failed launch returns DP_ERR_CUDA. Conditions
 * found on the device (a bounded wait that expired) are recorded in the
 * first word of the caller's workspace and read back (and cleared) by
 * dp_check_status. Zero a workspace once after allocating it; the library
 * never sets that word except on a device-side error.
 * No entry point aborts, traps or throws.
 */
#ifndef DP_H_
#define DP_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *dp_stream_t;   /* same type as cudaStream_t */

typedef enum {
    DP_OK = 0,
    DP_ERR_INVALID_ARG = 1,   /* NULL / host pointer, negative size, bad enum */
    DP_ERR_UNSUPPORTED = 2,   /* D_k, D_v not in {32,64,128}; n_h not in 1..4 */
    DP_ERR_ALIGNMENT = 3,     /* q, k, v, o, state, workspace not 16-byte aligned */
    DP_ERR_WORKSPACE = 4,     /* workspace NULL or smaller than required */
    DP_ERR_CUDA = 5,          /* a CUDA runtime call or launch failed */
    DP_ERR_TIMEOUT = 6,       /* a device-side bounded wait expired */
    DP_ERR_DEVICE = 7         /* the device reported another inconsistency */
} dp_status;

typedef enum { DP_F32 = 0, DP_BF16 = 1 } dp_dtype;

/* Kernel family for dp_forward. AUTO picks the tensor-core chunked kernel
 * where it applies (bf16, D_k = D_v = 128) and the recurrent kernel
 * otherwise; the others force one family (CHUNK_TC returns
 * DP_ERR_UNSUPPORTED where it does not apply). */
typedef enum { DP_IMPL_AUTO = 0, DP_IMPL_RECURRENT = 1, DP_IMPL_CHUNK_TC = 2 } dp_impl;

typedef struct {
    int B, T, H;     /* batch, tokens, heads (T may be 0) */
    int Dk, Dv;      /* key and value head dims: 32, 64 or 128 */
    int nh;          /* Householder steps per token (n_h), 1..4 */
    int dtype;       /* dp_dtype of q, k, v, beta, g */
    int impl;        /* dp_impl */
    int out_dtype;   /* dp_dtype of o: equal to dtype, or DP_F32 with bf16 inputs */
    int max_seqlen;  /* dp_forward_varlen: the longest packed sequence (bounds the
                        workspace); 0 for every other call */
    int prologue;    /* dp_prologue_flags applied to the inputs as they are loaded
                        (dp_forward, dp_forward_varlen, dp_decode_step,
                        dp_forward_noalloc); 0 = inputs used as given */
} dp_dims;

/* Input prologue (DeltaProduct paper, Sec.4: keys are psi(W x) / ||psi(W x)||
 * with psi = SiLU, betas phi(U x) with phi = sigmoid or 2 sigmoid; the gated
 * variant's gate is a sigmoid). With a flag set, the corresponding input
 * holds the raw projection and the kernels apply the map while loading it,
 * in fp32: the normalised keys and queries are then rounded to the input
 * dtype (they are tensor-core operands), betas and gates stay fp32.
 * BETA_SIGMOID and BETA_2SIGMOID are exclusive. */
typedef enum {
    DP_PRO_KEY_SILU_L2 = 1,    /* k <- SiLU(k) / ||SiLU(k)||_2 (a zero row stays zero) */
    DP_PRO_QUERY_L2 = 2,       /* q <- q / ||q||_2 */
    DP_PRO_BETA_SIGMOID = 4,   /* beta <- sigmoid(beta) */
    DP_PRO_BETA_2SIGMOID = 8,  /* beta <- 2 sigmoid(beta) */
    DP_PRO_GATE_SIGMOID = 16   /* g <- sigmoid(g) */
} dp_prologue_flags;

/* ABI version of this header (bumped on any signature change). */
#define DP_ABI_VERSION 10
int dp_abi_version(void);

/* Human-readable name of a status code (static string, never NULL). */
const char *dp_status_string(dp_status s);

/* Bytes of device workspace dp_forward needs for `dims` (>= 256). The first
 * 4 bytes hold the device status word. */
dp_status dp_forward_workspace_size(const dp_dims *dims, size_t *bytes);

/* Bytes of device workspace with which dp_forward runs its fastest path
 * (>= dp_forward_workspace_size; it depends on the current device's SM
 * count). For the tensor-core chunk path this adds, per (batch, head,
 * chunk) of ceil(T / ct) chunks, ct = min(16, 32 / n_h) tokens, an
 * 18688-byte record and a 4-byte flag (each area rounded up to 256 bytes):
 * every chunk's UT transform is then prepared in parallel (by the other
 * CTAs of one cooperative launch when B*H leaves at least half the SMs
 * free, else by a first kernel) and the state pass streams the records in.
 * In the cooperative mode the prep runs at most 16 chunks ahead of each
 * head's state pass and the state pass drops each record from L2 once it
 * has read it, so records live in L2 only and do not reach DRAM.
 * Dense problems without prologue or write keys whose B*H is small enough
 * that each sequence can be cut into P >= 2 segments of at least 16 chunks
 * with B*H*(2P - 1) <= the SM count take the segmented mode instead
 * (DP_PATH_CHUNK_SEG; the recurrence is affine in the state, so each segment
 * runs from a zero state and from the identity at once and a short combine
 * chains them); its workspace adds, after the records, 3 B*H*P fp32 D x D
 * matrices and two fp32 arrays of o's size. With at least
 * dp_forward_workspace_size bytes but less than the records, dp_forward
 * runs one fused kernel instead. The split, cooperative and fused modes
 * agree with each other up to rounding (split and cooperative bit for bit);
 * the segmented mode adds the rounding of its combine and correction. Both
 * sizes are equal for the recurrent path. The library clears the flags on
 * the stream before every cooperative launch, so a workspace may be reused
 * by calls of any shapes, in any order; calls sharing a workspace must be
 * ordered (one stream). */
dp_status dp_forward_workspace_size_fast(const dp_dims *dims, size_t *bytes);

/* How dp_forward runs a problem given `workspace_bytes` of workspace
 * (library facility, no counterpart in the paper): the kernel family and,
 * for the chunk path, its mode, which fixes the number of kernels one call
 * enqueues (1, or 2 for DP_PATH_CHUNK_SPLIT). Queries the current device;
 * enqueues nothing. */
typedef enum {
    DP_PATH_RECURRENT = 0,    /* token-by-token SIMT kernel */
    DP_PATH_CHUNK_FUSED = 1,  /* one tensor-core kernel, prep inside */
    DP_PATH_CHUNK_SPLIT = 2,  /* prep kernel, then the state-pass kernel */
    DP_PATH_CHUNK_COOP = 3,   /* one cooperative launch: prep CTAs beside the state pass */
    DP_PATH_CHUNK_SEG = 4     /* segmented: each sequence cut into segments run at once (four launches) */
} dp_path;
dp_status dp_forward_path(const dp_dims *dims, size_t workspace_bytes, int *path);

/* Whole-sequence forward (the extended T*n_h sequence of the paper's Sec.5.1,
 * processed in chunks by the tensor-core kernel):
 *   h0       initial state, NULL = zeros;
 *   h_final  final state, NULL = not written; may alias h0;
 *   o        outputs for every token.
 * T = 0 copies h0 (or zeros) to h_final. */
dp_status dp_forward(const dp_dims *dims,
                     const void *q, const void *k, const void *v,
                     const void *beta, const void *g,
                     const float *h0, void *o, float *h_final,
                     void *workspace, size_t workspace_bytes,
                     dp_stream_t stream);

/* Variable-length sequences packed back to back (a library facility for
 * training batches; the paper's Sec.4 recurrence runs on each sequence
 * independently: every sequence starts from its own initial state and no
 * state crosses a boundary, as with a gate of 0 at each sequence start).
 * dims->B = N sequences, dims->T = total tokens, dims->max_seqlen >= the
 * longest sequence (sizes the workspace, see dp_forward_workspace_size*).
 * cu_seqlens: int32 [N+1] in device memory, 0 = cu[0] <= cu[1] <= ... <=
 * cu[N] = T; sequence s holds tokens cu[s] .. cu[s+1]-1.
 * Layouts drop the batch axis: q [T,H,D_k], k [T,H,n_h,D_k],
 * v [T,H,n_h,D_v], beta [T,H,n_h], g [T,H] or NULL, o [T,H,D_v];
 * h0 / h_final [N,H,D_k,D_v] fp32 (NULL as in dp_forward).
 * The host cannot read cu_seqlens: each CTA checks its sequence's bounds
 * before touching any token and, if they break the rules above or exceed
 * max_seqlen, records DP_ERR_DEVICE (dp_check_status) and computes nothing
 * for that sequence. */
dp_status dp_forward_varlen(const dp_dims *dims, const int *cu_seqlens,
                            const void *q, const void *k, const void *v,
                            const void *beta, const void *g,
                            const float *h0, void *o, float *h_final,
                            void *workspace, size_t workspace_bytes,
                            dp_stream_t stream);

/* One decode step (dims->T is ignored and taken as 1) on a carried state,
 * updated in place. Shapes drop the T axis: q [B,H,D_k], k [B,H,n_h,D_k],
 * v [B,H,n_h,D_v], beta [B,H,n_h], g [B,H] or NULL, o [B,H,D_v],
 * state [B,H,D_k,D_v] fp32. Same recurrence as dp_forward with T = 1. */
dp_status dp_decode_step(const dp_dims *dims,
                         const void *q, const void *k, const void *v,
                         const void *beta, const void *g,
                         float *state, void *o, dp_stream_t stream);

/* State import / export / reset between the library's canonical fp32
 * [B,H,D_k,D_v] state and a caller buffer `ext` of type ext_dtype, laid out
 * [B,H,D_k,D_v] or, when ext_transposed != 0, [B,H,D_v,D_k] (the S = H^T
 * convention). ZERO ignores ext. */
typedef enum { DP_STATE_ZERO = 0, DP_STATE_IMPORT = 1, DP_STATE_EXPORT = 2 } dp_state_op;
dp_status dp_state_io(int op, int B, int H, int Dk, int Dv, float *state,
                      void *ext, int ext_dtype, int ext_transposed,
                      dp_stream_t stream);

/* Backward pass: gradients of L = <d_o, o> + <dh_final, h_final> through
 * the recurrence dp_forward computes (DeltaProduct paper, Sec.4 Eq.(2)-(3),
 * gated variant), for training. Same dims and input layouts as dp_forward
 * (dims->prologue and dims->max_seqlen must be 0; dims->out_dtype is the
 * type of d_o). dims->impl picks the form:
 *   DP_IMPL_AUTO       the chunked form for ungated problems with
 *                      D_k = D_v = 128 when the workspace holds its records,
 *                      else the recurrent form;
 *   DP_IMPL_RECURRENT  the recurrent form (any shape, gated or not);
 *   DP_IMPL_CHUNK_TC   the chunked form (WY representation of each chunk of
 *                      tokens, OSDN paper App.A.2, differentiated per chunk;
 *                      fp32 on CUDA cores), gated or not; DP_ERR_UNSUPPORTED
 *                      when D_k, D_v != 128. Gated: gates g >= 0 (a gate
 *                      below 1.8e-35, zero included, is taken as 1.8e-35, as
 *                      the forward's chunk path does); a negative or NaN
 *                      gate records DP_ERR_DEVICE (dp_check_status).
 *   d_o      [B,T,H,D_v] gradient of the outputs;
 *   dh_final [B,H,D_k,D_v] fp32 gradient of the final state, NULL = zeros;
 * outputs, fp32, written in full:
 *   dq [B,T,H,D_k], dk [B,T,H,n_h,D_k], dv [B,T,H,n_h,D_v],
 *   dbeta [B,T,H,n_h], dg [B,T,H] (required iff g != NULL, else ignored),
 *   dh0 [B,H,D_k,D_v] (NULL = not written; the gradient with respect to
 *   h0, or to the zero initial state when h0 is NULL).
 * In the recurrent form the gradients with respect to the key rows and the
 * scalars (dq, dk, dbeta, dg) are sums over the value columns that the
 * kernel accumulates with fp32 atomic additions, so their last bits may
 * vary between calls; the chunked form has no atomics and is deterministic.
 * workspace: at least dp_backward_workspace_size bytes for the same dims
 * (and impl): the status block, then for the recurrent form the state
 * checkpoints (fp32 D_k x D_v per (b,h) every few tokens) and every
 * sub-step's error v - H^T k (fp32 B T H n_h D_v); for the chunked form, per
 * chunk of min(16, 32 / n_h) tokens, its WY record and the fp32 state at its
 * start and state gradient at its end (about 200 KB per chunk). AUTO's size
 * covers both forms. */
dp_status dp_backward_workspace_size(const dp_dims *dims, size_t *bytes);
/* dp_backward over packed variable-length sequences: layouts, cu_seqlens
 * and dims->max_seqlen as in dp_forward_varlen (the gradients take the
 * layouts of their inputs: dq [T,H,D_k], ..., dh0 [N,H,D_k,D_v]); forms as
 * in dp_backward (dims->impl); the workspace (dp_backward_workspace_size
 * with the same dims) holds the recurrent form's checkpoints and errors or
 * the chunked form's records for max_seqlen per (sequence, head); each
 * sequence is cut into its own chunks. Sequences whose offsets break the
 * contract record DP_ERR_DEVICE and are skipped. */
dp_status dp_backward_varlen(const dp_dims *dims, const int *cu_seqlens,
                             const void *q, const void *k, const void *v,
                             const void *beta, const void *g, const float *h0,
                             const void *d_o, const float *dh_final,
                             float *dq, float *dk, float *dv, float *dbeta, float *dg,
                             float *dh0, void *workspace, size_t workspace_bytes,
                             dp_stream_t stream);
dp_status dp_backward(const dp_dims *dims,
                      const void *q, const void *k, const void *v,
                      const void *beta, const void *g, const float *h0,
                      const void *d_o, const float *dh_final,
                      float *dq, float *dk, float *dv, float *dbeta, float *dg,
                      float *dh0, void *workspace, size_t workspace_bytes,
                      dp_stream_t stream);

/* The prologue on its own (the unfused form): reads the raw q, k, beta, g
 * of a dense problem (dims->prologue selects the maps; layouts as in
 * dp_forward) and writes the mapped tensors to q_out, k_out, beta_out,
 * g_out in the input dtype. Outputs whose flag is clear are not written
 * (their pointer may be NULL); g and g_out are ignored without
 * DP_PRO_GATE_SIGMOID. dp_forward with dims->prologue = 0 on the outputs
 * computes what dp_forward with the flags computes on the raw inputs, up to
 * rounding (here betas and gates are rounded to the input dtype). */
dp_status dp_prologue(const dp_dims *dims, const void *q, const void *k, const void *beta,
                      const void *g, void *q_out, void *k_out, void *beta_out, void *g_out,
                      dp_stream_t stream);

/* OSDN write keys (the OSDN paper's online preconditioning applied to this
 * recurrence). Phase 1, dp_osdn_write_keys: per (b,h), over the extended
 * rows in order (token t, then its n_h keys), emit the write key
 * k~ = d (.) k with the current d, then update
 *   d <- clamp(r d + eta beta (1 - beta <d, k (.) k>) / max(||k||^2, eps) * (k (.) k),
 *              d_lo, d_hi)
 * (OSDN paper, Alg.1 / Eq.(3); APF retention r, Sec.4.4, applied once per
 * token on its first row; r = 1 without APF). The paper's configuration:
 * eta = 0.003, [d_lo, d_hi] = [0.5, 2], eps = 1e-6, d0 = 1.
 *   k [B,T,H,n_h,D_k], beta [B,T,H,n_h] (dims->dtype; used as given:
 *   dims->prologue must not map keys or betas), r [B,T,H] or NULL;
 *   d0 [B,H,D_k] fp32 or NULL (ones); kw [B,T,H,n_h,D_k] output in
 *   dims->dtype; d_final [B,H,D_k] fp32 or NULL. fp32 arithmetic.
 * Phase 2, dp_forward_write_keys: dp_forward with the state written along
 * the write key, H <- H + beta k~ (v - H^T k)^T, the error still read with
 * k (OSDN paper, Sec.4.1, Eq.(5)); kw has the layout of k. The chunk
 * (tensor-core) path takes it in its split modes, i.e. with a workspace of
 * at least dp_forward_workspace_size_fast and dims->prologue = 0 (the Gram
 * becomes K K~^T, the readout scores Q K~^T, the state update runs along
 * K~, W keeps K); otherwise, or with dims->impl RECURRENT, the recurrent
 * kernel; CHUNK_TC where the chunk path cannot take it returns
 * DP_ERR_UNSUPPORTED. dims->prologue must not map keys. */
dp_status dp_osdn_write_keys(const dp_dims *dims, const void *k, const void *beta, const void *r,
                             const float *d0, float eta, float d_lo, float d_hi, float eps,
                             void *kw, float *d_final, dp_stream_t stream);
dp_status dp_forward_write_keys(const dp_dims *dims, const void *q, const void *k, const void *kw,
                                const void *v, const void *beta, const void *g, const float *h0,
                                void *o, float *h_final, void *workspace, size_t workspace_bytes,
                                dp_stream_t stream);

/* Synchronises `stream`, returns the status the device recorded in the
 * workspace since it was last cleared, and clears it. */
dp_status dp_check_status(const void *workspace, dp_stream_t stream);

/* Fault injection for tests of the device-side bounded waits (a library
 * facility; the paper has no counterpart). Applies to the cooperative mode
 * of the chunk path (DP_PATH_CHUNK_COOP), process-wide, to every launch
 * made after the call until it is called again with (0, 0):
 *   withhold_first_record  1: the prep CTAs never publish the record of the
 *                          first chunk (batch 0, head 0, chunk 0), so the
 *                          state pass's wait for it must expire; 0: normal.
 *   flag_wait_polls        polls of a record flag (about 64 ns or more
 *                          each) before that wait gives up; 0 restores the
 *                          default (2^24 polls, about a second or more).
 * An expired wait makes the waiting CTA record DP_ERR_TIMEOUT in the
 * workspace's status word, drain what it has in flight, release its tensor
 * memory and return; the other CTAs finish normally, so the launch ends and
 * the context stays usable (a head stuck at chunk c holds the prep of its
 * chunks >= c + 16 back, and prep work queued behind them then times out
 * too: every wait is bounded). Nothing faults, traps or hangs. Returns
 * DP_ERR_INVALID_ARG unless withhold_first_record is 0 or 1. */
dp_status dp_test_set_wait_fault(int withhold_first_record, unsigned int flag_wait_polls);

/* dp_forward for callers that cannot allocate device memory (their HBM is
 * owned by a framework allocator or a fixed memory budget, or cudaMalloc's
 * implicit synchronisation is not acceptable on their path). This entry
 * point is a library facility; the DeltaProduct paper has no counterpart.
 * Same arguments, layouts and results as dp_forward, without the workspace:
 * the scratch lives in a fixed 64 KiB device array inside libdp.so that
 * every GPU loading the library holds until the process exits, and the call
 * allocates nothing. Problems whose dp_forward_workspace_size exceeds 64 KiB
 * return DP_ERR_WORKSPACE. Each call made outside stream capture looks up
 * the array's device address on the current device (cudaGetSymbolAddress);
 * a call made while `stream` is capturing reuses the address the last
 * uncaptured call on that device found, so make one call before any stream
 * capture. All calls on a device share the array and it keeps what the
 * last call left: calls whose kernels overlap on the GPU (unordered
 * streams) race on it; calls ordered on one stream are safe, whatever their
 * shapes. Device-side wait timeouts are not reported by this entry point
 * (each call clears the array's status word behind its kernel); host-side
 * validation and launch errors are. */
dp_status dp_forward_noalloc(const dp_dims *dims,
                             const void *q, const void *k, const void *v,
                             const void *beta, const void *g,
                             const float *h0, void *o, float *h_final,
                             dp_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* DP_H_ */
