// Tensor-core chunked DeltaProduct forward (tcgen05 / TMEM / TMA), bf16 inputs,
// D_k = D_v = 128, fp32 state and accumulation.
//
// What it computes (DeltaProduct paper, Sec.5.1: the n_h keys of every token
// form an extended T*n_h DeltaNet sequence, the gate is applied once per
// token, only the last step of each token is read out; chunk transform from
// the OSDN paper, App.A.2 / App.C, with write key = read key, state H = S^T).
// Per chunk of ct whole tokens (R = ct*n_h <= 32 rows of the extended
// sequence, padded with beta = 0 rows, which are exact no-ops), with L_r the
// cumulative log-gate from the chunk start, Gamma_r = exp(L_r) and
// E_rs = exp(L_r - L_s):
//   G   = tril(diag(beta) (K K^T * E), -1)               Gram
//   T   = (I + G)^{-1}                                   UT transform
//   W   = T diag(beta*Gamma) K,  U = T diag(beta) V
//   U'  = U - W S0                                       state pass, part 1
//   S   = Gamma_C S0 + K^T diag(Gamma_C/Gamma) U'        state pass, part 2
//   o_t = Gamma_r S0^T q_t + sum_{s<=r} E_rs (q_t.k_s) u'_s,  r = last row of t
//
// Four ways to run it (split and cooperative bit-identical; fused and
// segmented equal to them up to rounding):
//  * split (two kernels): the warp-per-chunk prep kernel (chunk_wprep_kernel;
//    chunk_prep_kernel with a prologue or write keys) does "phase A" (G, P,
//    T: the work that needs only one chunk's inputs) for every chunk of every
//    head at once and writes a record per chunk into the workspace; the
//    state-pass kernel then streams the records in with the inputs. The
//    sequential kernel keeps only the work that has to follow the state.
//  * cooperative (one launch, chunk_coop_kernel): state-pass CTAs and prep
//    CTAs side by side, each record published through a flag; the prep
//    stays at most kPaceLead chunks ahead of each head's state pass.
//  * fused (one kernel, no workspace beyond the status word): the state-pass
//    kernel's prep groups do phase A themselves, one chunk ahead.
//  * segmented (chunk_seg_kernel, seg_combine_kernel, seg_correct_kernel):
//    long sequences cut into segments that run at once, chained by their
//    affine transitions (see seg_combine_kernel).
// Compile-time variants (the Job type's flags), so that the plain
// instantiation carries none of their code:
//  * packed sequences (kPacked): each CTA reads its sequence's range from
//    cu_seqlens; chunk c of sequence s starts at token cu[s] + c*ct.
//  * input prologue (kPro): SiLU + L2 keys, L2 queries, sigmoid betas and
//    gates mapped on load; in the split modes the prep maps K and Q and
//    passes them in the record, in the fused mode the prep groups map the
//    stage in place.
//  * OSDN write keys (kWK, split modes): the Gram takes the write keys K~ as
//    its B operand (G = tril(diag(beta)(K K~^T * E), -1), P from Q K~^T) and
//    the state update runs along K~ (decayed K~^T tile); W keeps K.
//
// State-pass kernel organisation (one CTA per (batch, head), the state S^T
// resident in TMEM for the whole sequence, lanes = value columns):
//  * warp 20   TMA producer: K, Q, V tiles of each chunk (and its record in
//              split mode), 3-stage ring.
//  * warp 21   state-pass MMA issuer (one thread, tf32):
//              [U' | O_b] += S [-W; Gamma q]^T and [S | O_a] += U'^T [K^T; P].
//              These MMAs read S and U' straight from their fp32 TMEM
//              accumulators as the A operand; each hand-off (S -> U' -> S)
//              waits for the producing group's commit (see chain_role_plain).
//              The readout rides along in the same instructions (stacked B
//              operands), since each MMA instruction costs about the same
//              issue time whatever its N.
//  * warp 22   prep MMA issuer (bf16: [K;Q] K^T in fused mode, U, W), one
//              chunk ahead, on its own thread so its issue latency overlaps
//              the state pass.
//  * warps 4-11 and 12-19: two prep groups, taking even and odd chunks.
//              Phase A (fused mode only): turn the Gram MMA into G and P,
//              solve T on CUDA cores (16x16 diagonal blocks by forward
//              substitution, one lane per column, then the off-diagonal
//              block), write T as bf16 hi/lo tiles for the U/W MMAs.
//              Phase B (once the state pass has released the group's
//              buffers): write the fp32 B tiles of the state pass (P, Gamma q,
//              decayed K^T, and -W once the W MMA is done).
//  * warps 0-3 epilogue: initial state in, outputs and final state out; for
//              gated inputs the stored state is S / sigma (sigma: the chunk
//              decays since the last rescale, folded into the B tiles), and
//              on the few chunks that rescale it the epilogue multiplies it
//              by sigma Gamma_C between the two halves.
// Every wait on an mbarrier is bounded; on expiry the CTA records a timeout
// in the caller's status word, drains what it has in flight and exits.
#include <string.h>

#include <atomic>

#include "internal.h"
#include "sm100.cuh"

#include <cudaTypedefs.h>

namespace dp {
namespace {

using namespace sm100;

constexpr int kD = 128;        // D_k = D_v
constexpr int kC = 32;         // extended rows per chunk (padded)
constexpr int kNQ = 16;        // readout columns per chunk (tokens, padded)
constexpr int kNS = 3;         // TMA stages

constexpr int kPrepWarp = 4;   // warps 0-3 epilogue; 4-11 prep group 0, 12-19 prep group 1
constexpr int kPrepThreads = 256;
constexpr int kTmaWarp = 20;   // warp 21: state-pass MMA issuer; warp 22: prep MMA issuer
constexpr int kChainWarp = 21;
constexpr int kThreads = 23 * 32;

// ---- TMEM columns (512 allocated)
// The readout accumulates in two parts per chunk buffer g: O_b next to
// U'[g] (filled by the first state-pass MMA, B = [-W; Gamma q]) and O_a next
// to S (filled by the second, B = [K^T; P] or [P; K^T]); o = O_a + O_b.
constexpr uint32_t kColOa0 = 0;    // O_a[0]: 16 columns, left of S
constexpr uint32_t kColS = 16;     // S^T fp32: 128 columns (dk), lane = dv
constexpr uint32_t kColOa1 = 144;  // O_a[1]: 16 columns, right of S
constexpr uint32_t kColUN = 160;   // U'^T[g] at 160 + 48 g (32 columns), O_b[g] right after (16)
constexpr uint32_t kColGQ = 256;   // [K;Q] K^T fp32 (M = 64 layout): 2 x 32 columns (fused mode)
constexpr uint32_t kColW = 320;    // W^T fp32: 2 x 32 columns (chunk rows), lane = dk
constexpr uint32_t kTmemCols = 512;
__host__ __device__ constexpr uint32_t col_un(int g) { return kColUN + 48 * g; }
__host__ __device__ constexpr uint32_t col_ob(int g) { return kColUN + 48 * g + 32; }
__host__ __device__ constexpr uint32_t col_oa(int g) { return g ? kColOa1 : kColOa0; }

// ---- shared memory (offsets from a 1024-aligned base)
// TMA stage: KQ = 2 blocks (dk 0-63, 64-127) x 64 rows x 128 B (rows 0-31 K,
// rows 32-47 Q), V = 2 blocks (dv halves) x 32 rows x 128 B; bf16, 128-B swizzle.
constexpr uint32_t kKQBlock = 64 * 128;
constexpr uint32_t kVBlock = 32 * 128;
constexpr uint32_t kStageIn = 2 * kKQBlock + 2 * kVBlock;             // 24 KB of inputs
// Per prep group: fp32 B tiles of the state pass (K-major, 128-B swizzle,
// 32 fp32 per 128-B row) and, in fused mode, the bf16 T tiles.
// X = [-W (rows 0-31); Gamma q (rows 32-47)]: 4 K-blocks (dk) x 48 rows.
// Y = decayed K^T (128 rows, dk) and P (16 rows, token) over K = 32 chunk
// rows: group 0 stores [P; K^T], group 1 [K^T; P], matching O_a's side of S.
constexpr uint32_t kXRows = kC + kNQ;                 // 48
constexpr uint32_t kXBlock = kXRows * 128;            // 6 KB
constexpr uint32_t kYRows = kD + kNQ;                 // 144
constexpr uint32_t kGX = 0;
constexpr uint32_t kGY = kGX + 4 * kXBlock;           // 24 KB
constexpr uint32_t kGTb = kGY + kYRows * 128;         // + 18 KB; T tiles: 4 x (32 rows x 128 B)
constexpr uint32_t kTTile = 32 * 128;
constexpr uint32_t kLd = 33;                          // fp32 scratch row stride
constexpr uint32_t kGGs = 0;                          // G [32][33]
constexpr uint32_t kGTs = kGGs + 32 * kLd * 4;        // T [32][33]
constexpr uint32_t kGXs = kGTs + 32 * kLd * 4;        // X [16][17]
constexpr uint32_t kGPs = kGXs + 16 * 17 * 4;         // P staging [16][33]
constexpr uint32_t kGBeta = kGPs + 16 * kLd * 4;      // beta[32]
constexpr uint32_t kGL = kGBeta + 32 * 4;             // L[32]
constexpr uint32_t kPrepScratch = ((kGL + 32 * 4) + 15) & ~15u;

// ---- per-chunk record (split mode), written by chunk_prep_kernel into the
// workspace and copied verbatim into the chunk's stage:
//   T diag(beta) hi, lo | T diag(beta Gamma) hi, lo  (bf16, 32 rows x 128 B,
//   128-B swizzled as in shared memory; the Gamma pair only for gated input)
//   P [16][32] fp32 | beta [32] fp32 | L [32] fp32 (cumulative log-gate)
constexpr uint32_t kRecT = 0;
constexpr uint32_t kRecP = 4 * kTTile;                // 16 KB
constexpr uint32_t kRecBeta = kRecP + kNQ * kC * 4;   // + 2 KB
constexpr uint32_t kRecL = kRecBeta + kC * 4;
constexpr uint32_t kRecBytes = kRecL + kC * 4;        // 18688
static_assert(kRecBytes % 16 == 0, "bulk copies move 16-byte multiples");
// Write keys without a gate: the two T-tile slots the Gamma pair would use
// carry the chunk's K~ tile instead (two 64-column blocks of 32 rows x
// 128 B, swizzled as in shared memory), so the state pass finds it in its
// stage with the record.
constexpr uint32_t kRecKW = kRecT + 2 * kTTile;
// With a key or query prologue the record also carries the chunk's mapped
// K and Q rows (the 48 rows of each 64-column KQ block, swizzled as in
// shared memory), so the state pass copies them instead of mapping them.
constexpr uint32_t kRecKQBlock = (kC + kNQ) * 128;    // 6144
constexpr uint32_t kRecKQ = kRecBytes;
constexpr uint32_t kRecKQBytes = 2 * kRecKQBlock;
__host__ __device__ constexpr bool kq_in_record(int prologue)
{
    return (prologue & (DP_PRO_KEY_SILU_L2 | DP_PRO_QUERY_L2)) != 0;
}
__host__ __device__ constexpr uint32_t record_stride(int prologue)
{
    return kq_in_record(prologue) ? kRecBytes + kRecKQBytes : kRecBytes;
}
static_assert(record_stride(DP_PRO_KEY_SILU_L2) % 16 == 0, "bulk copies move 16-byte multiples");

// Output staging of one epilogue warp: a chunk's kNQ token rows of its 32
// value columns (fp32 rows of 128 B, bf16 rows of 64 B).
constexpr uint32_t kOutTile = kNQ * 128;

// Shared-memory layout of the state-pass kernel in each mode.
template <bool kSplit>
struct Layout {
    // split: the record follows the inputs in the stage (T tiles 1024-aligned)
    static constexpr uint32_t kStage = kSplit ? ((kStageIn + kRecBytes + 1023) & ~1023u) : kStageIn;
    static constexpr uint32_t kGroup = kSplit ? kGTb : kGTb + 4 * kTTile;
    static constexpr uint32_t kScratch = kSplit ? 0 : kPrepScratch;
    static constexpr uint32_t kOffGroup = kNS * kStage;
    static constexpr uint32_t kOffScratch = kOffGroup + 2 * kGroup;
    static constexpr uint32_t kOffOut = kOffScratch + 2 * kScratch;
    static constexpr uint32_t kOffBar = kOffOut + 4 * kOutTile;
};

constexpr uint32_t kNumBars = 2 * kNS + 2 * 7 + 8;
template <bool kSplit>
constexpr uint32_t smem_bytes() { return Layout<kSplit>::kOffBar + kNumBars * 8 + 16 + 1024; }
static_assert(smem_bytes<true>() <= 227 * 1024 && smem_bytes<false>() <= 227 * 1024, "shared memory");

constexpr uint32_t kWaitTries = 1u << 22;

struct Params {
    const __nv_bfloat16 *beta, *g;
    const float *h0;
    void *o;
    float *h_final;
    uint32_t *status;
    uint8_t *rec;              // per-chunk records (split mode), [B*H][n_chunks][rec_stride]
    uint32_t *flags;           // cooperative mode: record published, [B*H][n_chunks]
    uint32_t flag_tries;       // cooperative mode: polls of a flag before the wait gives up
    int withhold_first;        // cooperative mode, fault-injection hook: the first record is never published
    int T, H, nh, ct;
    int n_chunks;              // chunks of the longest sequence: records per (sequence, head)
    int bh_count;
    const int *cu;             // packed sequences: token offsets [B+1] (NULL: dense [B,T] layout)
    int B;
    int max_T;                 // longest sequence (T for dense calls)
    int prologue;              // dp_prologue_flags applied on load
    uint32_t rec_stride;       // bytes per record: record_stride(prologue)
    const __nv_bfloat16 *kw;   // OSDN write keys (layout of k), split modes only; NULL: write with k
    // segmented mode (see launch_chunk_tc): P segments of seg_chunks chunks per sequence
    int seg_count, seg_chunks;
    float *seg_h;              // [B*H][P][2][D][D]: end state of each segment's part 0 and part 1
    float *seg_o0;             // [B,T,H,D_v]: readout of part 0 (segments >= 1)
    float *seg_qt;             // [B,T,H,D_k]: readout of part 1 (segments >= 1)
};

// The (sequence, head) pair one state-pass CTA, or one prep step, works on.
// Dense calls (kPacked = false): sequence b is batch row b, T tokens, and
// every extent comes straight from the kernel parameters. Packed calls: the
// extent is read from cu (and checked) once.
template <bool kPk, bool kPr, bool kW = false, bool kSg = false>
struct Job {
    static constexpr bool kPacked = kPk;   // offsets from cu (else the dense layout)
    static constexpr bool kPro = kPr;      // input prologue (Params::prologue) applied on load
    static constexpr bool kWK = kW;        // OSDN write keys (Params::kw)
    static constexpr bool kSeg = kSg;      // one segment of a dense sequence (segmented mode)
    int b, h;          // sequence and head
    int b_map, t0;     // packed / segment: token t sits at row (row_b() * T + t0 + t) of the token layouts
    int len, nc;       // packed / segment: its tokens and chunks
    int c0;            // segment: its first chunk in the sequence's chunk grid (records)
    int seg, part;     // segment: index, and 0 = the state from the segment's start state, 1 = its transition
    bool valid;        // packed: false when the offsets broke their contract for this sequence
    __device__ __forceinline__ int row_b() const { return kPacked ? b_map : b; }
    __device__ __forceinline__ int first() const { return (kPacked || kSeg) ? t0 : 0; }
    __device__ __forceinline__ int tokens(const Params &p) const { return (kPacked || kSeg) ? len : p.T; }
    __device__ __forceinline__ int chunks(const Params &p) const { return (kPacked || kSeg) ? nc : p.n_chunks; }
    __device__ __forceinline__ bool ok() const { return kPacked ? valid : true; }
};

template <bool kPacked, bool kPro, bool kWK = false, bool kSeg = false>
__device__ __forceinline__ Job<kPacked, kPro, kWK, kSeg> make_job(const Params &p, int bh)
{
    Job<kPacked, kPro, kWK, kSeg> j;
    if (kSeg) {
        // segmented mode: CTA bh < B*H runs segment 0 of sequence bh from its
        // initial state; the others run, for segments 1 .. P-1 of every
        // sequence, the state from zero (part 0) and the transition (part 1)
        const int nbh = p.bh_count;
        int q = bh, seg = 0, part = 0;
        if (bh >= nbh) {
            const int r = bh - nbh, per = 2 * (p.seg_count - 1);
            q = r / per;
            seg = 1 + (r - q * per) / 2;
            part = (r - q * per) & 1;
        }
        j.b = q / p.H;
        j.h = q - j.b * p.H;
        j.b_map = j.b;
        j.seg = seg;
        j.part = part;
        j.c0 = seg * p.seg_chunks;
        j.t0 = j.c0 * p.ct;
        const int rest = p.T - j.t0, cap = p.seg_chunks * p.ct;
        j.len = rest < cap ? (rest > 0 ? rest : 0) : cap;
        j.nc = (j.len + p.ct - 1) / p.ct;
        j.valid = true;
        return j;
    }
    j.b = bh / p.H;
    j.h = bh - j.b * p.H;
    j.b_map = j.t0 = j.len = j.nc = 0;
    j.c0 = j.seg = j.part = 0;
    j.valid = true;
    if (kPacked) {
        const SeqRange r = seq_range(p.cu, j.b, p.B, p.T, p.max_T);
        j.b_map = r.b_map;
        j.t0 = r.t0;
        j.len = r.len;
        j.valid = r.ok;
        j.nc = (r.len + p.ct - 1) / p.ct;
    }
    return j;
}

// (token, head) index of token t of the job: rows of q, g, o (x n_h for k, v, beta)
template <class J>
__device__ __forceinline__ size_t tok_row(const Params &p, const J &j, int t)
{
    return ((size_t)j.row_b() * p.T + j.first() + t) * p.H + j.h;
}

// Cooperative mode: a record is published by storing 1 into its flag
// (release); the state pass acquires it before loading the record. The
// host clears every flag on the stream before each cooperative launch, so
// no value left in the workspace by an earlier call (of any shape) can
// pass for a published record.
__device__ __forceinline__ void flag_publish(uint32_t *flag, uint32_t v)
{
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(flag), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t flag_read(const uint32_t *flag)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
    return v;
}

// Once the state pass has issued the loads of a chunk it stores 2 into the
// chunk's flag. The warp prep paces itself on these marks: it loads chunk c
// of a head only once that head's state pass has taken chunk c - kPaceLead,
// so the records it writes (and the K and Q rows it reads, which the state
// pass reads again) are still in L2 when the state pass gets to them. The
// marks order nothing (relaxed): they only hold the prep back.
constexpr int kPaceLead = 16;
__device__ __forceinline__ void flag_mark_taken(uint32_t *flag)
{
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(flag), "r"(2u) : "memory");
}

__device__ __forceinline__ uint32_t flag_peek(const uint32_t *flag)
{
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
    return v;
}

template <class J>
__device__ __forceinline__ size_t rec_index(const Params &p, const J &j, int c)
{
    return ((size_t)j.b * p.H + j.h) * (size_t)p.n_chunks + (J::kSeg ? j.c0 + c : c);
}

// Cooperative mode: a chunk's record is read once, by the state pass's
// bulk copy, and is dead once that copy has landed. Its L2 lines are then
// dropped without a write-back (only lines wholly inside the record), so
// that records, which the prep writes only a few chunks ahead of the state
// pass, never travel to DRAM and back. Thread lt of nthreads drops every
// nthreads-th line.
template <class J>
__device__ __forceinline__ void discard_record(const Params &p, const J &j, int c, int lt, int nthreads)
{
    const uintptr_t r0 = (uintptr_t)(p.rec + rec_index(p, j, c) * p.rec_stride);
    const uintptr_t a = (r0 + 127) & ~(uintptr_t)127, e = (r0 + p.rec_stride) & ~(uintptr_t)127;
    for (uintptr_t l = a + (uintptr_t)lt * 128; l < e; l += (uintptr_t)nthreads * 128)
        asm volatile("discard.global.L2 [%0], 128;" ::"l"(l) : "memory");
}

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

// Tensor map with a 128-byte inner box and 128-byte swizzle (64 bf16, or
// 32 fp32 elements).
bool encode(CUtensorMap *map, const void *base, int rank, const cuuint64_t *dims,
            const cuuint64_t *strides_bytes, const cuuint32_t *box,
            CUtensorMapDataType type = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16)
{
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return enc(map, type, (cuuint32_t)rank, const_cast<void *>(base),
               dims, strides_bytes, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

enum : int {
    kBarFull = 0,                 // [kNS] TMA stage loaded (transaction bytes)
    kBarEmpty = kBarFull + kNS,   // [kNS] stage consumed by its prep group
    kBarGQ = kBarEmpty + kNS,     // [2] Gram MMA of the group's chunk done (fused)
    kBarTb = kBarGQ + 2,          // [2] T tiles written (fused)
    kBarUW = kBarTb + 2,          // [2] U and W MMAs done
    kBarReady = kBarUW + 2,       // [2] X = [-W; Gamma q] written
    kBarReadyY = kBarReady + 2,   // [2] Y = decayed K^T and P written, stage read
    kBarM2 = kBarReadyY + 2,      // [2] chunk's state pass and readout done
    kBarOFree = kBarM2 + 2,       // [2] O buffers drained by the epilogue (one arrival per warp)
    kBarM1 = kBarOFree + 2,       // first half (U', S^T q) done (gated, rescaling chunks only)
    kBarScaled,                   // stored state rescaled (gated; one arrival per epilogue warp)
    kBarInit,                     // initial state in TMEM
    kBarFinal,                    // [2] every MMA of an issuer retired (teardown)
    kBarNorm = kBarFinal + 2,     // [2] prologue applied to the group's stage (fused mode with a prologue)
    kBarXD = kBarNorm + 2,        // chain: a chunk's first-half MMAs retired (U' complete)
    kBarCount
};
static_assert(kBarCount == (int)kNumBars, "barrier count");

struct Smem {
    uint8_t *base;
    uint64_t *bar;
    uint32_t *tmem_slot;
    volatile uint32_t *abort;
    volatile uint32_t *renorm;   // [2] gated: the group's chunk rescales the stored state (see epi_role)
    uint32_t stage_bytes, group_off, group_bytes, scratch_off, out_off;
    __device__ uint8_t *stage(int st) const { return base + st * stage_bytes; }
    __device__ uint8_t *out_tile(int warp) const { return base + out_off + warp * kOutTile; }
    __device__ uint8_t *group(int g) const { return base + group_off + g * group_bytes; }
    __device__ uint8_t *scratch(int g) const { return base + scratch_off + g * kPrepScratch; }
};

__device__ __forceinline__ void flag_error(uint32_t *status, volatile uint32_t *abort, uint32_t code)
{
    *abort = 1;
    if (status) atomicCAS(status, 0u, code);
}

__device__ __forceinline__ bool wait_bar(const Smem &s, int idx, uint32_t parity, uint32_t *status)
{
    if (mbar_wait(&s.bar[idx], parity, kWaitTries, s.abort)) return true;
    flag_error(status, s.abort, kDevTimeout);
    return false;
}

// OR of `v` over the `count` threads of named barrier `id` (also a barrier).
__device__ __forceinline__ bool group_any(uint32_t id, uint32_t count, bool v)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\t"
        "bar.red.or.pred po, %2, %3, pi;\n\tselp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// Lane 0 waits (bounded); the warp agrees on the outcome, which is false
// when the wait expired or another role aborted.
__device__ __forceinline__ bool warp_wait(const Smem &s, int idx, uint32_t parity, uint32_t *status)
{
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = wait_bar(s, idx, parity, status) && !*s.abort;
    return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

__device__ __forceinline__ void split_pack(float a, float b, uint32_t &hi, uint32_t &lo)
{
    hi = pack_bf16x2(a, b);
    const float ah = __uint_as_float(hi << 16), bh = __uint_as_float(hi & 0xFFFF0000u);
    lo = pack_bf16x2(a - ah, b - bh);
}

__device__ __forceinline__ void store_out(float *o, size_t i, float x) { o[i] = x; }
__device__ __forceinline__ void store_out(__nv_bfloat16 *o, size_t i, float x) { o[i] = __float2bfloat16_rn(x); }

// One chunk's outputs from one epilogue warp: lane = value column (32 of
// them, from o0 on), v[i] = token i's value, rows 0 .. n_rows-1 stored, row
// i at o0 + i * tok_stride. The block turns around in the warp's staging
// tile so that each lane stores 16 contiguous bytes (4 lanes per bf16 row, 8
// per fp32 row): a few wide stores instead of one 2- or 4-byte store per
// token. o0 is 16-byte aligned (o is, and the column block starts at a
// multiple of 32 elements).
template <typename T>
__device__ __forceinline__ void store_rows(T *o0, size_t tok_stride, const uint32_t (&v)[kNQ], int n_rows,
                                           uint8_t *stg, int lane)
{
    constexpr int kRowB = 32 * (int)sizeof(T);   // bytes of a row
    constexpr int kLanesRow = kRowB / 16;
    constexpr int kRowsPer = 32 / kLanesRow;      // rows per store instruction
    __syncwarp();   // the previous chunk's reads of the tile are done
#pragma unroll
    for (int i = 0; i < kNQ; ++i)
        if (i < n_rows) store_out((T *)(stg + i * kRowB), lane, __uint_as_float(v[i]));
    __syncwarp();
    const int r0 = lane / kLanesRow, piece = lane % kLanesRow;
#pragma unroll
    for (int k = 0; k < kNQ / kRowsPer; ++k) {
        const int r = r0 + k * kRowsPer;
        if (r < n_rows)
            *(uint4 *)((uint8_t *)(o0 + (size_t)r * tok_stride) + piece * 16) =
                *(const uint4 *)(stg + r * kRowB + piece * 16);
    }
}

// Gram MMA [K;Q] K^T of the chunk in the KQ tiles at `kq` (A = 64 rows: K
// rows 0-31, Q rows 32-47, zero rows; B = the K rows), into 32 TMEM columns.
__device__ __forceinline__ void issue_gram(uint32_t d_tmem, uint32_t kq)
{
    const uint32_t id_gq = idesc_bf16(64, kC, false, false);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint64_t d = sdesc_sw128(kq + (kk >> 2) * kKQBlock + (kk & 3) * 32, 16, 1024);
        mma_ss(d_tmem, d, d, id_gq, kk > 0);
    }
}

// The Gram MMA with write keys (OSDN): [K;Q] K~^T, B = the K~ tile (rows
// 0..31 of two 64-column blocks of kKWBlock bytes), so G and P come out
// asymmetric as the write-key chunk form needs.
constexpr uint32_t kKWBlock = kC * 128;   // 4 KB: 32 rows x 128 B
__device__ __forceinline__ void issue_gram_wk(uint32_t d_tmem, uint32_t kq, uint32_t kwt)
{
    const uint32_t id_gq = idesc_bf16(64, kC, false, false);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint64_t a = sdesc_sw128(kq + (kk >> 2) * kKQBlock + (kk & 3) * 32, 16, 1024);
        const uint64_t b = sdesc_sw128(kwt + (kk >> 2) * kKWBlock + (kk & 3) * 32, 16, 1024);
        mma_ss(d_tmem, a, b, id_gq, kk > 0);
    }
}

// ------------------------------------------------------------------ TMA producer
constexpr uint32_t kFlagTries = 1u << 24;   // default flag polls: x >= 64 ns each, seconds, then a timeout

template <bool kSplit, bool kCoop, class J>
__device__ void tma_role(const Smem &s, const Params &p, const CUtensorMap *tk,
                         const CUtensorMap *tv, const CUtensorMap *tq, const J &jb)
{
    const int h = jb.h;
    const int ct = p.ct, R = ct * p.nh;
    const bool gated = p.g != nullptr;
    // K and V: 2 x R rows x 128 B each; Q: 2 x ct rows. Record: the T tiles
    // it uses (2 or 4) and P, beta, L.
    const uint32_t rec_t = ((gated || J::kWK) ? 4 : 2) * kTTile, rec_tail = kRecBytes - kRecP;
    // mapped K and Q from the record (split modes with a key/query prologue)
    const bool kq_rec = kSplit && J::kPro && kq_in_record(p.prologue);
    // segmented mode, transition part: no values (the V tiles stay zero, so U = 0)
    const bool no_v = J::kSeg && jb.part == 1;
    const uint32_t bytes = (kq_rec ? 256u * R + kRecKQBytes : (no_v ? 256u : 512u) * R + 256u * ct) +
                           (kSplit ? rec_t + rec_tail : 0u);
    int last_use[kNS];
    for (int i = 0; i < kNS; ++i) last_use[i] = -1;
    for (int c = 0; c < jb.chunks(p); ++c) {
        const int st = c % kNS, u = c / kNS;
        if (u >= 1 && !wait_bar(s, kBarEmpty + st, (u - 1) & 1, p.status)) break;
        if (kCoop) {
            // the prep CTAs of this launch publish the chunk's record: acquire
            // it, then order the bulk copy (async proxy) after that read
            const uint32_t *flag = p.flags + rec_index(p, jb, c);
            uint32_t tries = 0;
            while (flag_read(flag) != 1u && ++tries < p.flag_tries && !*s.abort) __nanosleep(64);
            if (tries >= p.flag_tries || *s.abort) {
                flag_error(p.status, s.abort, kDevTimeout);
                break;
            }
            asm volatile("fence.proxy.async.global;" ::: "memory");
        }
        uint8_t *kq = s.stage(st), *vv = kq + 2 * kKQBlock;
        uint64_t *bar = &s.bar[kBarFull + st];
        mbar_arrive_expect_tx(bar, bytes);
        const int t0 = jb.first() + c * ct, b = jb.row_b();
        const uint8_t *rec = kSplit ? p.rec + rec_index(p, jb, c) * p.rec_stride : nullptr;
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
            if (kq_rec) {
                bulk_load(kq + kb * kKQBlock, rec + kRecKQ + kb * kRecKQBlock, kRecKQBlock, bar);
            } else {
                tma_load_5d(kq + kb * kKQBlock, tk, bar, kb * 64, 0, h, t0, b);
                tma_load_4d(kq + kb * kKQBlock + kC * 128, tq, bar, kb * 64, h, t0, b);
            }
            if (!no_v) tma_load_5d(vv + kb * kVBlock, tv, bar, kb * 64, 0, h, t0, b);
        }
        if (kSplit) {
            uint8_t *dst = kq + kStageIn;
            bulk_load(dst + kRecT, rec + kRecT, rec_t, bar);
            bulk_load(dst + kRecP, rec + kRecP, rec_tail, bar);
        }
        if (kCoop) flag_mark_taken(p.flags + rec_index(p, jb, c));
        last_use[st] = u;
    }
    // every issued load must have landed before shared memory is released
    uint32_t no_abort = 0;
    for (int st = 0; st < kNS; ++st)
        if (last_use[st] >= 0) mbar_wait(&s.bar[kBarFull + st], last_use[st] & 1, kWaitTries, &no_abort);
}

// ------------------------------------------------------------------ MMA issuers
// Prep MMAs (bf16): [K;Q] K^T (fused mode), U^T = V^T (T diag beta)^T,
// W^T = K^T (T diag(beta Gamma))^T. They run one chunk ahead of the state
// pass and are issued by their own thread so that their issue latency
// overlaps the state pass's.
template <bool kSplit, bool kPro>
__device__ void prep_mma_role(const Smem &s, const Params &p, uint32_t tbase, int n)
{
    const bool gated = p.g != nullptr;
    const uint32_t id_uw = idesc_bf16(128, kC, true, false);

    // T enters as hi + lo bf16 tiles (in the group's tiles, or in the stage's record)
    auto issue_uw = [&](int c) {
        const int g = c & 1;
        const uint32_t kq = smem_addr(s.stage(c % kNS)), vv = kq + 2 * kKQBlock;
        const uint32_t tt = kSplit ? kq + kStageIn + kRecT : smem_addr(s.group(g)) + kGTb;
        const uint32_t tg = tt + (gated ? 2 * kTTile : 0);
#pragma unroll
        for (int part = 0; part < 2; ++part)
#pragma unroll
            for (int kk = 0; kk < 2; ++kk)
                mma_ss(tbase + col_un(g), sdesc_sw128(vv + kk * 2048, kVBlock, 1024),
                       sdesc_sw128(tt + part * kTTile + kk * 32, 16, 1024), id_uw, part | kk);
#pragma unroll
        for (int part = 0; part < 2; ++part)
#pragma unroll
            for (int kk = 0; kk < 2; ++kk)
                mma_ss(tbase + kColW + g * 32, sdesc_sw128(kq + kk * 2048, kKQBlock, 1024),
                       sdesc_sw128(tg + part * kTTile + kk * 32, 16, 1024), id_uw, part | kk);
        mma_commit(&s.bar[kBarUW + g]);
    };
    // U/W of chunk u: its T tiles are in place, and the state pass of chunk
    // u - 2 (which read U'[g]; W[g] was drained before it started) has finished
    auto uw_ready = [&](int u) {
        if (kSplit) {
            if (!wait_bar(s, kBarFull + u % kNS, (u / kNS) & 1, p.status)) return false;
        } else {
            if (!wait_bar(s, kBarTb + (u & 1), (u >> 1) & 1, p.status)) return false;
        }
        if (u >= 2 && !wait_bar(s, kBarM2 + (u & 1), ((u - 2) >> 1) & 1, p.status)) return false;
        tc_fence_after();
        return true;
    };

    bool ok = true;
    if (kSplit) {
        for (int c = 0; c < n && ok; ++c)
            if ((ok = uw_ready(c))) issue_uw(c);
    } else {
        for (int c = 0; c < n && ok; ++c) {
            ok = kPro ? wait_bar(s, kBarNorm + (c & 1), (c >> 1) & 1, p.status)
                      : wait_bar(s, kBarFull + c % kNS, (c / kNS) & 1, p.status);
            if (!ok) break;
            tc_fence_after();
            issue_gram(tbase + kColGQ + (c & 1) * 32, smem_addr(s.stage(c % kNS)));
            mma_commit(&s.bar[kBarGQ + (c & 1)]);
            if (c >= 1) {
                if (!(ok = uw_ready(c - 1))) break;
                issue_uw(c - 1);
            }
        }
        if (ok && n > 0 && uw_ready(n - 1)) issue_uw(n - 1);   // an empty sequence has no chunk
    }
    mma_commit(&s.bar[kBarFinal + 1]);
    uint32_t no_abort = 0;
    mbar_wait(&s.bar[kBarFinal + 1], 0, kWaitTries, &no_abort);
}

// State-pass MMAs (tf32, A = the fp32 accumulators in TMEM):
//   [U'^T | O_b] += S^T [-W; Gamma q]^T          (16 instructions, N = 48)
//   [S^T | O_a] or [O_a | S^T] += U'^T [K^T; P]   (4 instructions, N = 144)
// The second group reads as its A operand what the first wrote (U'), and the
// next chunk's first group reads what the second wrote (S). The tcgen05
// memory model runs one thread's MMAs in issue order only when they share
// the accumulator and the shape, which these do not: each such hand-off
// waits for the producing MMAs' commit (the first group's on kBarXD, the
// second group's on the chunk's M2 barrier) and fences before the consuming
// MMAs. (Issued back to back, the second group read a partly written U' in
// a few chunks per 10^5 under a full CTA's load.) Any other instruction
// of the issuing thread between two of its MMAs costs the tensor pipe about
// as much as several MMAs, so the waits of a chunk sit at these two points.
__device__ void chain_role_plain(const Smem &s, const Params &p, uint32_t tbase, int n)
{
    const uint32_t id_x = idesc_tf32(128, kXRows);
    const uint32_t id_y = idesc_tf32(128, kYRows);
    bool ok = wait_bar(s, kBarInit, 0, p.status);
    for (int c = 0; c < n && ok; ++c) {
        const int g = c & 1;
        const uint32_t gb = smem_addr(s.group(g));
        const uint32_t d_x = tbase + col_un(g);
        const uint32_t d_y = g ? tbase + kColS : tbase + kColOa0;   // O_a[0] | S  or  S | O_a[1]
        if (!(ok = wait_bar(s, kBarReady + g, (c >> 1) & 1, p.status))) break;
        if (!(ok = wait_bar(s, kBarReadyY + g, (c >> 1) & 1, p.status))) break;
        if (c >= 2 && !(ok = wait_bar(s, kBarOFree + g, ((c - 2) >> 1) & 1, p.status))) break;
        // S as the previous chunk's second group left it
        if (c >= 1 && !(ok = wait_bar(s, kBarM2 + (g ^ 1), ((c - 1) >> 1) & 1, p.status))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 16; ++kk)
            mma_ts_tf32(d_x, tbase + kColS + kk * 8,
                        sdesc_sw128(gb + kGX + (kk >> 2) * kXBlock + (kk & 3) * 32, 16, 1024), id_x, 1);
        mma_commit(&s.bar[kBarXD]);
        if (!(ok = wait_bar(s, kBarXD, c & 1, p.status))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            mma_ts_tf32(d_y, d_x + kk * 8, sdesc_sw128(gb + kGY + kk * 32, 16, 1024), id_y, 1);
        mma_commit(&s.bar[kBarM2 + g]);
    }
    mma_commit(&s.bar[kBarFinal]);
    uint32_t no_abort = 0;
    mbar_wait(&s.bar[kBarFinal], 0, kWaitTries, &no_abort);
}

// With a gate: the chain starts a chunk on the X tile while phase B writes
// the Y tile (the chain waits for the first group's commit anyway, and the
// Y tile is mostly ready by then), and a chunk that rescales the stored
// state hands it to the epilogue between the halves. The hand-offs between
// the MMA groups wait for commits as in chain_role_plain.
__device__ void chain_role_gated(const Smem &s, const Params &p, uint32_t tbase, int n)
{
    const uint32_t id_x = idesc_tf32(128, kXRows);
    const uint32_t id_y = idesc_tf32(128, kYRows);
    bool ok = wait_bar(s, kBarInit, 0, p.status);
    uint32_t n_renorm = 0;
    for (int c = 0; c < n && ok; ++c) {
        const int g = c & 1;
        const uint32_t gb = smem_addr(s.group(g));
        if (!(ok = wait_bar(s, kBarReady + g, (c >> 1) & 1, p.status))) break;
        if (c >= 2 && !(ok = wait_bar(s, kBarOFree + g, ((c - 2) >> 1) & 1, p.status))) break;
        if (c >= 1 && !(ok = wait_bar(s, kBarM2 + (g ^ 1), ((c - 1) >> 1) & 1, p.status))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 16; ++kk)
            mma_ts_tf32(tbase + col_un(g), tbase + kColS + kk * 8,
                        sdesc_sw128(gb + kGX + (kk >> 2) * kXBlock + (kk & 3) * 32, 16, 1024), id_x, 1);
        mma_commit(&s.bar[kBarXD]);
        const bool rescale = s.renorm[g] != 0u;   // this chunk rescales the stored state
        if (rescale) mma_commit(&s.bar[kBarM1]);
        if (!(ok = wait_bar(s, kBarXD, c & 1, p.status))) break;
        if (rescale) {
            if (!(ok = wait_bar(s, kBarScaled, n_renorm & 1, p.status))) break;
            ++n_renorm;
        }
        if (!(ok = wait_bar(s, kBarReadyY + g, (c >> 1) & 1, p.status))) break;
        tc_fence_after();
        const uint32_t d_y = g ? tbase + kColS : tbase + kColOa0;   // O_a[0] | S  or  S | O_a[1]
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            mma_ts_tf32(d_y, tbase + col_un(g) + kk * 8, sdesc_sw128(gb + kGY + kk * 32, 16, 1024), id_y, 1);
        mma_commit(&s.bar[kBarM2 + g]);
    }
    mma_commit(&s.bar[kBarFinal]);
    uint32_t no_abort = 0;
    mbar_wait(&s.bar[kBarFinal], 0, kWaitTries, &no_abort);
}

// ------------------------------------------------------------------ prep work
// Input prologue on a landed KQ stage (bf16; two 64-column blocks of 64
// rows x 128 B, 128-byte swizzle): SiLU + L2 normalisation of key rows
// 0..R-1 and L2 normalisation of query rows kC..kC+ct-1, as the flags
// select, in place, one warp per row, rounded back to bf16. The swizzle
// only permutes 16-byte pieces within a row, and the maps are per element
// plus a row norm, so each lane takes its 8 bytes where they lie (lane l:
// block l/16, byte 8(l%16) of the row).
__device__ void normalise_rows(uint8_t *kq, int R, int ct, int flags, int lt, int nthreads)
{
    const int lane = lt & 31, nw = nthreads >> 5;
    const int nk = (flags & DP_PRO_KEY_SILU_L2) ? R : 0, nq = (flags & DP_PRO_QUERY_L2) ? ct : 0;
    for (int i = lt >> 5; i < nk + nq; i += nw) {
        const bool key = i < nk;
        const int row = key ? i : kC + (i - nk);
        uint2 *ptr = (uint2 *)(kq + (lane >> 4) * kKQBlock + row * 128 + (lane & 15) * 8);
        uint2 raw = *ptr;
        const float2 a = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&raw.x));
        const float2 b = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&raw.y));
        float x[4] = {a.x, a.y, b.x, b.y}, ss = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (key) x[e] = pro_silu(x[e]);
            ss = fmaf(x[e], x[e], ss);
        }
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
        const float inv = pro_inv_norm(ss);
        __nv_bfloat162 lo = __floats2bfloat162_rn(x[0] * inv, x[1] * inv);
        __nv_bfloat162 hi = __floats2bfloat162_rn(x[2] * inv, x[3] * inv);
        raw.x = *reinterpret_cast<uint32_t *>(&lo);
        raw.y = *reinterpret_cast<uint32_t *>(&hi);
        *ptr = raw;
    }
}

// Per-row betas and log-gates of one chunk (lane = extended row).
struct RowVals {
    float beta, lg;
};

template <class J>
__device__ __forceinline__ RowVals load_rows(const Params &p, const J &jb, int c, int lane)
{
    RowVals v{0.f, 0.f};
    if (c >= jb.chunks(p)) return v;
    const int nh = p.nh, R = p.ct * nh, tl = lane / nh, j = lane - tl * nh, t = c * p.ct + tl;
    if (lane < R && t < jb.tokens(p)) {   // rows past the sequence's end: beta = 0, exact no-ops
        const size_t tok = tok_row(p, jb, t);
        v.beta = __bfloat162float(p.beta[tok * nh + j]);
        if (J::kPro) v.beta = pro_beta(v.beta, p.prologue);
        if (p.g != nullptr && j == 0)
            v.lg = J::kPro ? pro_log_gate(__bfloat162float(p.g[tok]), p.prologue)
                           : fmaxf(logf(__bfloat162float(p.g[tok])), -80.f);
    }
    return v;
}

// beta and the cumulative log-gate L (inclusive scan over the chunk's rows;
// the token gate sits on its first row) into shared memory. One warp.
__device__ __forceinline__ void scan_rows(RowVals rv, int lane, float *beta_s, float *L_s)
{
    float lg = rv.lg;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, lg, d);
        if (lane >= d) lg += y;
    }
    beta_s[lane] = rv.beta;
    L_s[lane] = lg;
}

// Gated inputs: the state kept in TMEM is S^ with S = sigma S^, sigma the
// product of the chunk decays Gamma_C since the last rescale, so that most
// chunks need no pass over the state: sigma folds into the state pass's B
// tiles (-W and Gamma q rows times sigma_c, decayed K rows over sigma_{c+1}).
// A chunk whose decay would take log sigma below kRenormLog rescales S^ by
// sigma_c Gamma_C instead (the epilogue, between the two halves of the
// state pass) and restarts sigma at 1; so sigma >= e^-27 and the B-tile
// factors stay below e^27. Every role evaluates this sequence from the same
// fp32 values with the same operations, so all agree bit for bit.
constexpr float kRenormLog = -27.f;

__device__ __forceinline__ bool renorm_at(float ls, float lgc) { return ls + lgc < kRenormLog; }
__device__ __forceinline__ float ls_after(float ls, float lgc)
{
    const float x = ls + lgc;
    return x < kRenormLog ? 0.f : x;
}

// log Gamma_C of a chunk (its cumulative log-gate at its last row) in two
// steps, so that the load runs ahead of its use: gate_raw fetches row
// `lane`'s raw bf16 gate (its token's gate on the token's first row, by the
// read-only path so that the load may be issued before the stores that
// precede its use), or kNoGate; gate_lgc makes the same per-row values and
// the same scan as load_rows and scan_rows (so the result equals the L[kC-1]
// the prep side computes for that chunk, bit for bit). Whole warp.
constexpr uint32_t kNoGate = 0xFFFFFFFFu;
template <class J>
__device__ __forceinline__ uint32_t gate_raw(const Params &p, const J &jb, int c, int lane)
{
    const int nh = p.nh, R = p.ct * nh, tl = lane / nh, j = lane - tl * nh, t = c * p.ct + tl;
    if (c < jb.chunks(p) && lane < R && j == 0 && t < jb.tokens(p))
        return (uint32_t)__ldg((const unsigned short *)p.g + tok_row(p, jb, t));
    return kNoGate;
}

template <class J>
__device__ __forceinline__ float gate_lgc(const Params &p, uint32_t raw, int lane)
{
    float lg = 0.f;
    if (raw != kNoGate) {
        const float x = __uint_as_float(raw << 16);   // the bf16 value, exactly
        lg = J::kPro ? pro_log_gate(x, p.prologue) : fmaxf(logf(x), -80.f);
    }
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, lg, d);
        if (lane >= d) lg += y;
    }
    return __shfl_sync(0xffffffffu, lg, 31);
}

struct PrepScratch {
    float *Gs, *Ts, *Xs, *Ps, *beta_s, *L_s;
};

__device__ __forceinline__ PrepScratch prep_scratch(uint8_t *sc)
{
    return {(float *)(sc + kGGs), (float *)(sc + kGTs), (float *)(sc + kGXs),
            (float *)(sc + kGPs), (float *)(sc + kGBeta), (float *)(sc + kGL)};
}

// Phase A of one chunk, by the 256 threads `lt` of named barrier `bar_id`
// (warps whose index mod 4 is lt / 32 mod 4, for TMEM lane access): G and P
// from the finished Gram accumulator at TMEM columns `gq_col`, T by blocked
// forward substitution, then T diag(beta) and (gated) T diag(beta Gamma) as
// hi + lo bf16 tiles at `tdst` (shared or global memory, 128-B swizzled
// rows). Needs beta_s / L_s in place. Leaves P in w.Ps.
__device__ void phase_a(const PrepScratch &w, uint32_t tbase, uint32_t gq_col, uint8_t *tdst,
                        int lt, int nh, int ct, bool gated, uint32_t bar_id)
{
    const int lw = lt >> 5, lane = lt & 31, lq = lw & 3, hf = lw >> 2;   // TMEM lane quarter, column half
    float *Gs = w.Gs, *Ts = w.Ts, *Xs = w.Xs, *Ps = w.Ps;
    const float *beta_s = w.beta_s, *L_s = w.L_s;

    // Gram MMA (M = 64 layout): quarter lq's lanes 0..15 hold rows
    // 16*lq .. 16*lq + 15; half hf takes columns 16*hf .. 16*hf + 15.
    {
        uint32_t r[16];
        tmem_ld16(tbase + ((uint32_t)(lq * 32) << 16) + gq_col + 16 * hf, r);
        tmem_wait_ld();
        const int m = 16 * lq + lane;
        if (lane < 16 && m < kC) {
            const float br = beta_s[m], Lr = L_s[m];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int s2 = 16 * hf + j;
                float v = 0.f;
                if (s2 < m) {
                    v = br * __uint_as_float(r[j]);
                    if (gated) v *= __expf(Lr - L_s[s2]);
                }
                Gs[m * kLd + s2] = v;
            }
        } else if (lane < 16 && m < kC + kNQ) {
            const int i = m - kC, rr = i * nh + nh - 1;
            const bool valid = i < ct;
            const float Lr = valid ? L_s[rr] : 0.f;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int s2 = 16 * hf + j;
                float x = 0.f;
                if (valid && s2 <= rr) {
                    x = __uint_as_float(r[j]);
                    if (gated) x *= __expf(Lr - L_s[s2]);
                }
                Ps[i * kLd + s2] = x;
            }
        }
    }
    tc_fence_before();
    named_sync(bar_id, kPrepThreads);

    // T = (I + G)^{-1}: diagonal 16x16 blocks (one lane per column,
    // forward substitution), then T_10 = -T_11 (G_10 T_00)
    if (lw < 2 && lane < 16) {
        const int base = 16 * lw, col = base + lane;
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = (i == lane) ? 1.f : 0.f;
#pragma unroll
        for (int s2 = 0; s2 < 16; ++s2) {
            const float xs = x[s2];
#pragma unroll
            for (int i = s2 + 1; i < 16; ++i) x[i] = fmaf(-Gs[(base + i) * kLd + base + s2], xs, x[i]);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) Ts[(base + i) * kLd + col] = x[i];
    }
    named_sync(bar_id, kPrepThreads);
    {
        const int i = lt >> 4, j = lt & 15;
        float a = 0.f;
#pragma unroll
        for (int m = 0; m < 16; ++m) a = fmaf(Gs[(16 + i) * kLd + m], Ts[m * kLd + j], a);
        Xs[i * 17 + j] = a;
    }
    named_sync(bar_id, kPrepThreads);
    {
        const int i = lt >> 4, j = lt & 15;
        float a = 0.f;
#pragma unroll
        for (int u = 0; u < 16; ++u)
            if (u <= i) a = fmaf(Ts[(16 + i) * kLd + 16 + u], Xs[u * 17 + j], a);
        Ts[(16 + i) * kLd + j] = -a;
    }
    named_sync(bar_id, kPrepThreads);

    // T diag(beta) and T diag(beta Gamma) as hi + lo bf16 tiles:
    // one (tile, row, 8-element chunk) per thread
    if (lt < (gated ? 256 : 128)) {
        const int pr = lt >> 7, i = (lt >> 2) & 31, ch = lt & 3;
        uint8_t *hi = tdst + 2 * pr * kTTile, *lo = hi + kTTile;
        uint32_t wh[4], wl[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int s0 = ch * 8 + 2 * e;
            float v0 = s0 <= i ? Ts[i * kLd + s0] * beta_s[s0] : 0.f;
            float v1 = s0 + 1 <= i ? Ts[i * kLd + s0 + 1] * beta_s[s0 + 1] : 0.f;
            if (pr) {
                v0 *= __expf(L_s[s0]);
                v1 *= __expf(L_s[s0 + 1]);
            }
            split_pack(v0, v1, wh[e], wl[e]);
        }
        *(uint4 *)(hi + sw128_offset(i, ch)) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
        *(uint4 *)(lo + sw128_offset(i, ch)) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
    }
}

// Row offsets of K^T and P inside the group's Y tile.
__device__ __forceinline__ int y_row_k(int g) { return g ? 0 : kNQ; }
__device__ __forceinline__ int y_row_p(int g) { return g ? kD : 0; }

// Phase B of chunk c (group g, stage st): the state pass's fp32 B tiles. P
// comes from `Psrc` (row stride `pld` floats), the cumulative log-gates from
// `L_s`, K and Q from the stage at `kq`. X = [-W; Gamma q] is signalled
// first (the chain starts the chunk's first half on it), then Y = [K^T; P]
// (decayed K^T, needed by the second half only) together with the release
// of the stage. `renorm` is the chunk's rescale flag for the chain. Returns
// false, uniformly over the group, if a wait failed or the CTA is aborting.
__device__ __forceinline__ bool phase_b_gated(const Smem &s, const Params &p, uint32_t tbase, uint8_t *gt,
                        const uint8_t *kq, const float *Psrc, int pld, const float *L_s, int c,
                        int g, int st, int lt, uint32_t bar_id, float ls_cur, float ls_next, bool renorm,
                        const float *kw16 = nullptr, const uint8_t *ksrc = nullptr,
                        uint32_t kblock = kKQBlock)
{
    const int lw = lt >> 5, lane = lt & 31, lq = lw & 3, hf = lw >> 2;
    const int nh = p.nh, ct = p.ct;
    constexpr bool gated = true;
    // the group's tiles are free once the state pass of chunk c - 2 has retired
    bool ok = (c < 2 || lt != 0) || wait_bar(s, kBarM2 + g, ((c - 2) >> 1) & 1, p.status);
    if (group_any(bar_id, kPrepThreads, !ok || *s.abort)) return false;
    // Gamma-scaled q: (token row i, dk block kb4, 8-element group q)
    {
        const int i = lt >> 4, kb4 = (lt >> 2) & 3, q = lt & 3;
        const bool valid = i < ct;
        const float gr = !valid ? 0.f : (gated ? __expf(L_s[i * nh + nh - 1] + ls_cur) : 1.f);
        const uint4 u = *(const uint4 *)(kq + (kb4 >> 1) * kKQBlock + sw128_offset(kC + i, (kb4 & 1) * 4 + q));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
        float f[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            f[2 * e] = __uint_as_float(w[e] << 16) * gr;
            f[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u) * gr;
        }
        uint8_t *dst = gt + kGX + kb4 * kXBlock;
        *(float4 *)(dst + sw128_offset(kC + i, 2 * q)) = make_float4(f[0], f[1], f[2], f[3]);
        *(float4 *)(dst + sw128_offset(kC + i, 2 * q + 1)) = make_float4(f[4], f[5], f[6], f[7]);
    }
    // -W (lane = dk; half hf takes chunk rows 16*hf .. 16*hf + 15)
    ok = (lt != 0) || wait_bar(s, kBarUW + g, (c >> 1) & 1, p.status);
    if (group_any(bar_id, kPrepThreads, !ok || *s.abort)) return false;
    tc_fence_after();
    {
        uint32_t r[16];
        tmem_ld16(tbase + ((uint32_t)(lq * 32) << 16) + kColW + g * 32 + 16 * hf, r);
        tmem_wait_ld();
        const int dk = 32 * lq + lane, pos = dk & 31;
        uint8_t *dst = gt + kGX + (dk >> 5) * kXBlock + (pos & 3) * 4;
        const float nsig = gated ? -__expf(ls_cur) : -1.f;
#pragma unroll
        for (int j = 0; j < 16; ++j)
            *(float *)(dst + sw128_offset(16 * hf + j, pos >> 2)) = nsig * __uint_as_float(r[j]);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    named_sync(bar_id, kPrepThreads);
    if (lt == 0) {
        // the chain reads the flag after the X barrier; its previous value
        // (chunk c - 2) was read before the state pass waited for above
        s.renorm[g] = renorm ? 1u : 0u;
        mbar_arrive(&s.bar[kBarReady + g]);
    }
    // P (16 rows x 8 float4)
    if (lt < kNQ * 8) {
        const int i = lt >> 3, ch = lt & 7;
        const float *src = Psrc + i * pld + 4 * ch;
        *(float4 *)(gt + kGY + sw128_offset(y_row_p(g) + i, ch)) = make_float4(src[0], src[1], src[2], src[3]);
    }
    // decayed K^T (write keys: decayed K~^T, from kw16 = this thread's 16
    // values, or from the K~ tile at ksrc with blocks kblock bytes apart):
    // row dk, four groups of 4 chunk rows per thread. The decay of chunk row
    // s2 is one exponential per row, taken by lane s2 - 4 q0 of every warp
    // and passed around (the warp's rows are 4 q0 .. 4 q0 + 15).
    {
        const int dk = lt & 127, q0 = (lt >> 7) * 4;
        const float Lend = L_s[kC - 1] - ls_next;
        const float dec = gated ? __expf(Lend - L_s[4 * q0 + (lane & 15)]) : 1.f;
        const uint8_t *src = (ksrc ? ksrc : kq) + (dk >> 6) * kblock;
        const int chunk = (dk & 63) >> 3, e = dk & 7;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float f[4];
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
                const int s2 = 4 * (q0 + q) + k4;
                const float x = kw16 ? kw16[4 * q + k4]
                                     : __bfloat162float(*(const __nv_bfloat16 *)(src + sw128_offset(s2, chunk) + e * 2));
                const float d = __shfl_sync(0xffffffffu, dec, 4 * q + k4);
                f[k4] = gated ? x * d : x;
            }
            *(float4 *)(gt + kGY + sw128_offset(y_row_k(g) + dk, q0 + q)) = make_float4(f[0], f[1], f[2], f[3]);
        }
    }
    fence_proxy_async_smem();
    named_sync(bar_id, kPrepThreads);
    if (lt == 0) {
        mbar_arrive(&s.bar[kBarReadyY + g]);
        mbar_arrive(&s.bar[kBarEmpty + st]);
    }
    return true;
}

// Phase B without a gate: the tiles are quick to make, so X and Y are
// signalled together at the end (same arguments as phase_b_gated; kw16 is
// unused: ungated write keys arrive in the record at ksrc).
__device__ __forceinline__ bool phase_b_plain(const Smem &s, const Params &p, uint32_t tbase, uint8_t *gt,
                        const uint8_t *kq, const float *Psrc, int pld, const float *L_s, int c,
                        int g, int st, int lt, uint32_t bar_id, float ls_cur, float ls_next, bool renorm,
                        const float *kw16 = nullptr, const uint8_t *ksrc = nullptr,
                        uint32_t kblock = kKQBlock)
{
    const int lw = lt >> 5, lane = lt & 31, lq = lw & 3, hf = lw >> 2;
    const int ct = p.ct;
    bool ok = (c < 2 || lt != 0) || wait_bar(s, kBarM2 + g, ((c - 2) >> 1) & 1, p.status);
    if (group_any(bar_id, kPrepThreads, !ok || *s.abort)) return false;
    // P (16 rows x 8 float4)
    if (lt < kNQ * 8) {
        const int i = lt >> 3, ch = lt & 7;
        const float *src = Psrc + i * pld + 4 * ch;
        *(float4 *)(gt + kGY + sw128_offset(y_row_p(g) + i, ch)) = make_float4(src[0], src[1], src[2], src[3]);
    }
    // q rows (token row i, dk block kb4, 8-element group q); zero past the chunk's tokens
    {
        const int i = lt >> 4, kb4 = (lt >> 2) & 3, q = lt & 3;
        const float gr = i < ct ? 1.f : 0.f;
        const uint4 u = *(const uint4 *)(kq + (kb4 >> 1) * kKQBlock + sw128_offset(kC + i, (kb4 & 1) * 4 + q));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
        float f[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            f[2 * e] = __uint_as_float(w[e] << 16) * gr;
            f[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u) * gr;
        }
        uint8_t *dst = gt + kGX + kb4 * kXBlock;
        *(float4 *)(dst + sw128_offset(kC + i, 2 * q)) = make_float4(f[0], f[1], f[2], f[3]);
        *(float4 *)(dst + sw128_offset(kC + i, 2 * q + 1)) = make_float4(f[4], f[5], f[6], f[7]);
    }
    // K^T (or K~^T from ksrc): row dk, four groups of 4 chunk rows per thread
    {
        const int dk = lt & 127, q0 = (lt >> 7) * 4;
        const uint8_t *src = (ksrc ? ksrc : kq) + (dk >> 6) * kblock;
        const int chunk = (dk & 63) >> 3, e = dk & 7;
#pragma unroll
        for (int q = q0; q < q0 + 4; ++q) {
            float f[4];
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4)
                f[k4] = __bfloat162float(*(const __nv_bfloat16 *)(src + sw128_offset(4 * q + k4, chunk) + e * 2));
            *(float4 *)(gt + kGY + sw128_offset(y_row_k(g) + dk, q)) = make_float4(f[0], f[1], f[2], f[3]);
        }
    }
    // -W (lane = dk; half hf takes chunk rows 16*hf .. 16*hf + 15)
    ok = (lt != 0) || wait_bar(s, kBarUW + g, (c >> 1) & 1, p.status);
    if (group_any(bar_id, kPrepThreads, !ok || *s.abort)) return false;
    tc_fence_after();
    {
        uint32_t r[16];
        tmem_ld16(tbase + ((uint32_t)(lq * 32) << 16) + kColW + g * 32 + 16 * hf, r);
        tmem_wait_ld();
        const int dk = 32 * lq + lane, pos = dk & 31;
        uint8_t *dst = gt + kGX + (dk >> 5) * kXBlock + (pos & 3) * 4;
#pragma unroll
        for (int j = 0; j < 16; ++j)
            *(float *)(dst + sw128_offset(16 * hf + j, pos >> 2)) = -__uint_as_float(r[j]);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    named_sync(bar_id, kPrepThreads);
    if (lt == 0) {
        s.renorm[g] = 0u;
        mbar_arrive(&s.bar[kBarReady + g]);
        mbar_arrive(&s.bar[kBarReadyY + g]);
        mbar_arrive(&s.bar[kBarEmpty + st]);
    }
    return true;
}

__device__ __forceinline__ bool phase_b(const Smem &s, const Params &p, uint32_t tbase, uint8_t *gt,
                        const uint8_t *kq, const float *Psrc, int pld, const float *L_s, int c,
                        int g, int st, int lt, uint32_t bar_id, float ls_cur, float ls_next, bool renorm,
                        const float *kw16 = nullptr, const uint8_t *ksrc = nullptr,
                        uint32_t kblock = kKQBlock)
{
    return p.g ? phase_b_gated(s, p, tbase, gt, kq, Psrc, pld, L_s, c, g, st, lt, bar_id, ls_cur, ls_next, renorm, kw16, ksrc, kblock)
               : phase_b_plain(s, p, tbase, gt, kq, Psrc, pld, L_s, c, g, st, lt, bar_id, ls_cur, ls_next, renorm, kw16, ksrc, kblock);
}

// Write keys of chunk c for phase B's decayed K~^T: thread lt's column
// dk = lt % 128 on chunk rows 16 (lt / 128) .. + 15 (zero past R or past the
// sequence), read from global memory ahead of the chunk's turn.
template <class J>
__device__ __forceinline__ void load_kw_rows(const Params &p, const J &jb, int c, int lt, float (&kwv)[16])
{
    const int dk = lt & 127, r0 = 16 * (lt >> 7), nh = p.nh, R = p.ct * nh;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int s2 = r0 + i, tl = s2 / nh, j = s2 - tl * nh, t = c * p.ct + tl;
        kwv[i] = (s2 < R && t < jb.tokens(p))
                     ? __bfloat162float(p.kw[(tok_row(p, jb, t) * nh + j) * kD + dk])
                     : 0.f;
    }
}

// The same rows of chunk c pulled into L2 ahead of load_kw_rows (no
// registers held: the kernel runs at its register cap).
template <class J>
__device__ __forceinline__ void prefetch_kw_rows(const Params &p, const J &jb, int c, int lt)
{
    const int dk = lt & 127, r0 = 16 * (lt >> 7), nh = p.nh, R = p.ct * nh;
    if ((dk & 63) != 0) return;   // one 128-byte line per 64 columns of a row
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int s2 = r0 + i, tl = s2 / nh, j = s2 - tl * nh, t = c * p.ct + tl;
        if (s2 < R && t < jb.tokens(p))
            asm volatile("prefetch.global.L2 [%0];" ::"l"(p.kw + (tok_row(p, jb, t) * nh + j) * kD + dk));
    }
}

// Prep group g of the state-pass kernel: chunks g, g + 2, ...
template <bool kSplit, class J>
__device__ void prep_role(const Smem &s, const Params &p, uint32_t tbase, int g, const J &jb)
{
    const int lt = threadIdx.x - (kPrepWarp + 8 * g) * 32, lw = lt >> 5, lane = lt & 31;
    const uint32_t bar_id = 1 + g;
    uint8_t *gt = s.group(g);
    const bool gated = p.g != nullptr;
    // gated: log sigma before the group's chunk (see kRenormLog), folded
    // over every chunk in order: the group's own previous chunk (c - 2, its
    // log Gamma_C kept) and the other group's (c - 1, its gates fetched one
    // iteration ahead)
    float ls = 0.f, lgc_own = 0.f;
    bool have_own = false;
    uint32_t graw_other = (p.g != nullptr && g == 1) ? gate_raw(p, jb, 0, lane) : kNoGate;
    auto advance_ls = [&](int c) {
        if (have_own) ls = ls_after(ls, lgc_own);
        if (c >= 1) ls = ls_after(ls, gate_lgc<J>(p, graw_other, lane));
        graw_other = gate_raw(p, jb, c + 1, lane);
    };

    if (kSplit) {
        for (int c = g; c < jb.chunks(p); c += 2) {
            const int st = c % kNS;
            const uint8_t *kq = s.stage(st), *rec = kq + kStageIn;
            // write keys: the chunk's rows from global memory, in flight
            // while the stage lands (fetching them a whole iteration ahead
            // costs registers the 80-register kernel spills: slower)
            float kwv[16];
            const bool kw_global = J::kWK && gated;   // ungated: K~ arrives in the record
            if (kw_global) {
                if (c + 2 < jb.chunks(p)) prefetch_kw_rows(p, jb, c + 2, lt);
                load_kw_rows(p, jb, c, lt, kwv);
            }
            if (gated) advance_ls(c);
            const bool ok = (lt != 0) || wait_bar(s, kBarFull + st, (c / kNS) & 1, p.status);
            if (group_any(bar_id, kPrepThreads, !ok || *s.abort)) break;
            const float *Lrec = (const float *)(rec + kRecL);
            const float lgc = gated ? Lrec[kC - 1] : 0.f, ls_next = ls_after(ls, lgc);
            // (with a key/query prologue the stage's K and Q arrive mapped, from the record)
            if (!phase_b(s, p, tbase, gt, kq, (const float *)(rec + kRecP), kC, Lrec, c, g, st, lt, bar_id, ls, ls_next,
                         gated && renorm_at(ls, lgc), kw_global ? kwv : nullptr,
                         (J::kWK && !gated) ? rec + kRecKW : nullptr, (J::kWK && !gated) ? kKWBlock : kKQBlock))
                break;
            // (after the chunk's signals: the group has time until the state pass frees its tiles)
            if (p.flags && !J::kSeg) discard_record(p, jb, c, lt, kPrepThreads);
            lgc_own = lgc;
            have_own = true;
        }
        return;
    }

    const PrepScratch w = prep_scratch(s.scratch(g));
    RowVals rv{0.f, 0.f};
    if (lw == 0) rv = load_rows(p, jb, g, lane);
    for (int c = g; c < jb.chunks(p); c += 2) {
        const int st = c % kNS;
        const uint8_t *kq = s.stage(st);
        if (gated) advance_ls(c);
        if (lw == 0) {
            scan_rows(rv, lane, w.beta_s, w.L_s);
            rv = load_rows(p, jb, c + 2, lane);          // next chunk of this group
        }
        if (J::kPro) {   // the prologue on the stage, before the Gram MMA reads it
            const bool okf = (lt != 0) || wait_bar(s, kBarFull + st, (c / kNS) & 1, p.status);
            if (group_any(bar_id, kPrepThreads, !okf || *s.abort)) break;
            normalise_rows(const_cast<uint8_t *>(kq), p.ct * p.nh, p.ct, p.prologue, lt, kPrepThreads);
            fence_proxy_async_smem();
            named_sync(bar_id, kPrepThreads);
            if (lt == 0) mbar_arrive(&s.bar[kBarNorm + g]);
        }
        // one thread polls the mbarriers; the group barrier spreads the outcome
        bool ok = true;
        if (lt == 0) {
            ok = wait_bar(s, kBarFull + st, (c / kNS) & 1, p.status);
            if (ok) ok = wait_bar(s, kBarGQ + g, (c >> 1) & 1, p.status);
        }
        if (group_any(bar_id, kPrepThreads, !ok || *s.abort)) break;
        tc_fence_after();
        phase_a(w, tbase, kColGQ + g * 32, gt + kGTb, lt, p.nh, p.ct, gated, bar_id);
        fence_proxy_async_smem();
        named_sync(bar_id, kPrepThreads);
        if (lt == 0) mbar_arrive(&s.bar[kBarTb + g]);
        const float lgc = gated ? w.L_s[kC - 1] : 0.f, ls_next = ls_after(ls, lgc);
        if (!phase_b(s, p, tbase, gt, kq, w.Ps, kLd, w.L_s, c, g, st, lt, bar_id, ls, ls_next,
                     gated && renorm_at(ls, lgc)))
            break;
        lgc_own = lgc;
        have_own = true;
    }
}

// ------------------------------------------------------------------ epilogue
template <typename TOut, class J>
__device__ void epi_role(const Smem &s, const Params &p, uint32_t tbase, const J &jb)
{
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t bar_id = 3;
    const uint32_t trow = tbase + ((uint32_t)(warp * 32) << 16);
    const size_t bh = (size_t)jb.b * p.H + jb.h;
    const bool gated = p.g != nullptr;
    // o row of the sequence's first token, this thread's value column.
    // Segmented mode, segments >= 1: the readout goes to fp32 workspace
    // arrays of o's layout (part 0: o from a zero start state; part 1: the
    // start state's weights q~ = A_{<=t}^T q_t), which the correction adds up.
    const bool ws_out = J::kSeg && jb.seg > 0;
    // (from this warp's block of 32 value columns)
    TOut *const o_seq = (TOut *)p.o + tok_row(p, jb, 0) * kD + warp * 32;
    float *const w_seq = J::kSeg ? (jb.part ? p.seg_qt : p.seg_o0) + tok_row(p, jb, 0) * kD + warp * 32 : nullptr;
    uint8_t *const stg = s.out_tile(warp);
    const size_t tok_stride = (size_t)p.H * kD;

    {   // S^T <- h0^T (lane = dv, column = dk), or zeros (or, for a segment's
        // transition part, the identity); readout accumulators zero
        const float *h0 = ws_out ? nullptr : p.h0;
        const bool ident = ws_out && jb.part == 1;
        uint32_t r[32];
        for (int c0 = 0; c0 < kD; c0 += 32) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                r[j] = __float_as_uint(ident ? (c0 + j == tid ? 1.f : 0.f)
                                             : (h0 ? h0[(bh * kD + c0 + j) * kD + tid] : 0.f));
            tmem_st32(trow + kColS + c0, r);
        }
        uint32_t z[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) z[j] = 0u;
        tmem_st16(trow + col_oa(0), z);
        tmem_st16(trow + col_oa(1), z);
        tmem_st16(trow + col_ob(0), z);
        tmem_st16(trow + col_ob(1), z);
        tmem_wait_st();
    }
    tc_fence_before();
    named_sync(bar_id, 128);
    if (tid == 0) mbar_arrive(&s.bar[kBarInit]);

    // Each warp owns 32 TMEM lanes (value columns) and runs on its own: it
    // waits for the chain's commits itself and arrives once per warp on the
    // barriers the chain waits for, and it releases a chunk's O buffers
    // before storing the outputs from registers.
    // Gated: the stored state is S^ = S / sigma (see kRenormLog); chunks
    // that rescale it are handled here, and h_final is sigma S^.
    bool failed = false;
    float ls = 0.f;
    uint32_t n_renorm = 0;
    uint32_t graw = gated ? gate_raw(p, jb, 0, lane) : kNoGate;   // gates one chunk ahead
    for (int c = 0; c < jb.chunks(p); ++c) {
        const int g = c & 1, t0 = c * p.ct;
        const float lgc = gated ? gate_lgc<J>(p, graw, lane) : 0.f;
        if (gated) graw = gate_raw(p, jb, c + 1, lane);
        if (gated && renorm_at(ls, lgc)) {
            // S^ <- sigma_c Gamma_C S^ between the chunk's two state-pass halves
            const float gC = __expf(ls + lgc);
            if (!warp_wait(s, kBarM1, n_renorm & 1, p.status)) { failed = true; break; }
            ++n_renorm;
            tc_fence_after();
            uint32_t r[32];
            for (int c0 = 0; c0 < kD; c0 += 32) {
                tmem_ld32(trow + kColS + c0, r);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * gC);
                tmem_st32(trow + kColS + c0, r);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            // (a release arrive, as for kBarOFree below)
            if (lane == 0) mbar_arrive(&s.bar[kBarScaled]);
        }
        ls = ls_after(ls, lgc);
        if (!warp_wait(s, kBarM2 + g, (c >> 1) & 1, p.status)) { failed = true; break; }
        tc_fence_after();
        uint32_t ra[16], rb[16];
        tmem_ld16(trow + col_oa(g), ra);
        tmem_ld16(trow + col_ob(g), rb);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < kNQ; ++i) {
            ra[i] = __float_as_uint(__uint_as_float(ra[i]) + __uint_as_float(rb[i]));
            rb[i] = 0u;
        }
        tmem_st16(trow + col_oa(g), rb);   // both parts accumulate: clear them for chunk c + 2
        tmem_st16(trow + col_ob(g), rb);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        // a release arrive: with the chain's acquiring wait and its
        // tcgen05.fence::after_thread_sync it orders the chain's next MMAs on
        // these columns after the clears above
        if (lane == 0) mbar_arrive(&s.bar[kBarOFree + g]);
        const int n_rows = min(p.ct, jb.tokens(p) - t0);
        if (ws_out)
            store_rows(w_seq + (size_t)t0 * tok_stride, tok_stride, ra, n_rows, stg, lane);
        else
            store_rows(o_seq + (size_t)t0 * tok_stride, tok_stride, ra, n_rows, stg, lane);
    }
    // segmented mode: every part's end state goes to the workspace (the
    // combine step turns them into start states and the final state)
    float *const hdst = J::kSeg ? p.seg_h + (((size_t)bh * p.seg_count + jb.seg) * 2 + jb.part) * kD * kD
                                : (p.h_final ? p.h_final + bh * kD * kD : nullptr);
    if (!failed && jb.ok() && hdst) {
        const float sig = gated ? __expf(ls) : 1.f;
        uint32_t r[32];
        for (int c0 = 0; c0 < kD; c0 += 32) {
            tmem_ld32(trow + kColS + c0, r);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) hdst[(size_t)(c0 + j) * kD + tid] = sig * __uint_as_float(r[j]);
        }
    }
}

// ------------------------------------------------------------------ state-pass kernel
template <typename TOut, bool kSplit, bool kCoop, bool kPacked, bool kPro, bool kWK = false, bool kSeg = false>
__device__ __forceinline__ void state_pass_cta(const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                                               const CUtensorMap &tm_q, const Params &p, int bh)
{
    using Lay = Layout<kSplit>;
    extern __shared__ uint8_t smem_raw[];
    Smem s;
    s.base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    s.bar = (uint64_t *)(s.base + Lay::kOffBar);
    s.tmem_slot = (uint32_t *)(s.bar + kNumBars);
    s.abort = s.tmem_slot + 1;
    s.renorm = s.tmem_slot + 2;
    s.stage_bytes = Lay::kStage;
    s.group_off = Lay::kOffGroup;
    s.group_bytes = Lay::kGroup;
    s.scratch_off = Lay::kOffScratch;
    s.out_off = Lay::kOffOut;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // a sequence with bad packed offsets runs no chunk
    const Job<kPacked, kPro, kWK, kSeg> jb = make_job<kPacked, kPro, kWK, kSeg>(p, bh);
    if (kPacked && threadIdx.x == 0 && !jb.ok()) report_bad_sequence(p.status);

    // Zero every tile once: rows TMA never writes (padding rows, query rows
    // beyond the chunk's tokens) must hold finite zeros.
    for (uint32_t i = threadIdx.x * 16; i < Lay::kOffScratch; i += kThreads * 16)
        *(uint4 *)(s.base + i) = make_uint4(0, 0, 0, 0);
    if (threadIdx.x == 0) {
        for (int i = 0; i < (int)kNumBars; ++i)
            mbar_init(&s.bar[i], (i == kBarOFree || i == kBarOFree + 1 || i == kBarScaled) ? kPrepWarp : 1);
        *s.abort = 0;
        fence_mbar_init();
    }
    if (warp == kTmaWarp && lane == 0) {
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_q);
    }
    if (warp == 0) tmem_alloc(s.tmem_slot, kTmemCols);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *s.tmem_slot;

    if (warp < kPrepWarp) {
        epi_role<TOut>(s, p, tbase, jb);
    } else if (warp < kTmaWarp) {
        prep_role<kSplit>(s, p, tbase, (warp - kPrepWarp) >> 3, jb);
    } else if (warp == kTmaWarp) {
        if (lane == 0) tma_role<kSplit, kCoop>(s, p, &tm_k, &tm_v, &tm_q, jb);
    } else if (warp == kChainWarp) {
        if (lane == 0) {
            if (p.g) chain_role_gated(s, p, tbase, jb.chunks(p));
            else chain_role_plain(s, p, tbase, jb.chunks(p));
        }
    } else {
        if (lane == 0) prep_mma_role<kSplit, kPro>(s, p, tbase, jb.chunks(p));
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, kTmemCols);
}

template <typename TOut, bool kSplit, bool kPacked, bool kPro, bool kWK = false>
__global__ void __launch_bounds__(kThreads, 1)
chunk_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                const __grid_constant__ CUtensorMap tm_q, const Params p)
{
    state_pass_cta<TOut, kSplit, false, kPacked, kPro, kWK>(tm_k, tm_v, tm_q, p, blockIdx.x);
}

// ------------------------------------------------------------------ chunk prep (split and cooperative modes)
// One prep group = 256 threads (`lt` 0..255; warps whose index mod 4 is
// lt / 32 mod 4, for TMEM lane access) working through its share of the
// chunks (every `stride`-th index of the chunk-major order from `first`),
// two deep: while the group solves chunk k (phase A, the T tiles straight
// into the chunk's record), the Gram MMA of chunk k + 1 runs and the K, Q
// tiles of chunk k + 2 are in flight. Per group: two stages (KQ tiles, and
// K~ tiles with write keys; rows TMA never writes are zero), two 32-column
// Gram accumulators, four mbarriers (loads into stage 0 / 1, Gram MMA into
// accumulator 0 / 1); chunk k uses stage and accumulator k % 2, as their
// (k / 2)-th use.
struct PrepGroup {
    uint8_t *stage;            // stage 0; stage 1 follows at pg_stage_bytes
    uint64_t *bar;             // [0, 1] stage loads, [2, 3] Gram MMAs
    uint32_t tcol;             // TMEM address of accumulator 0 (accumulator 1: + 32 columns)
    PrepScratch w;
    uint32_t bar_id;           // named barrier of the group
    int lt;
};
constexpr uint32_t kPGKQ = 2 * kKQBlock;   // KQ tiles of a stage (16 KB)
__host__ __device__ constexpr uint32_t pg_stage_bytes(bool wk) { return wk ? kPGKQ + 2 * kKWBlock : kPGKQ; }

// The next chunk index at or after `idx` in a group's share that holds a
// chunk (packed calls skip chunks past a sequence's end, and sequences with
// bad offsets); `total` when none is left.
template <bool kPacked, bool kPro, bool kWK>
__device__ __forceinline__ int next_chunk(const Params &p, int idx, int stride, int total)
{
    if (kPacked) {
        for (; idx < total; idx += stride) {
            const int c = idx / p.bh_count;
            if (c < make_job<kPacked, kPro, kWK>(p, idx - c * p.bh_count).chunks(p)) break;
        }
    }
    return idx < total ? idx : total;
}

// K and Q tiles (and K~ tiles) of chunk c of job jb into `stage`.
template <class J>
__device__ __forceinline__ void prep_issue_load(const Params &p, const CUtensorMap *tk, const CUtensorMap *tq,
                                                const CUtensorMap *tkw, uint8_t *stage, uint64_t *bar,
                                                const J &jb, int c)
{
    const int ct = p.ct, R = ct * p.nh, t0 = jb.first() + c * ct;
    mbar_arrive_expect_tx(bar, 256u * R + 256u * ct + (J::kWK ? 256u * R : 0u));
#pragma unroll
    for (int kb = 0; kb < 2; ++kb) {
        tma_load_5d(stage + kb * kKQBlock, tk, bar, kb * 64, 0, jb.h, t0, jb.row_b());
        tma_load_4d(stage + kb * kKQBlock + kC * 128, tq, bar, kb * 64, jb.h, t0, jb.row_b());
        if (J::kWK) tma_load_5d(stage + kPGKQ + kb * kKWBlock, tkw, bar, kb * 64, 0, jb.h, t0, jb.row_b());
    }
}

template <bool kPacked, bool kPro, bool kWK>
__device__ void prep_loop(const Params &p, const CUtensorMap *tk, const CUtensorMap *tq, const CUtensorMap *tkw,
                          const PrepGroup &G, volatile uint32_t *abort, int first, int stride, bool publish)
{
    using J = Job<kPacked, kPro, kWK>;
    constexpr uint32_t kSt = pg_stage_bytes(kWK);
    const int lt = G.lt, lane = lt & 31, ct = p.ct, R = ct * p.nh;
    const int total = p.n_chunks * p.bh_count;
    const bool gated = p.g != nullptr;
    // group work on a landed stage before its Gram MMA: the prologue's row
    // maps (and the mapped rows into the record), the K~ tile into the record
    constexpr bool kStageWork = kPro || kWK;
    // lt == 0: loads and MMAs issued and not yet waited for (drained on a timeout)
    bool ld_out[2] = {false, false}, mma_out[2] = {false, false};
    uint32_t ld_par[2] = {0, 0}, mma_par[2] = {0, 0};

    auto job_of = [&](int idx, int &c) {
        c = idx / p.bh_count;
        return make_job<kPacked, kPro, kWK>(p, idx - c * p.bh_count);
    };
    auto issue_load = [&](int idx, int st, uint32_t par) {
        int c;
        const J jb = job_of(idx, c);
        prep_issue_load(p, tk, tq, tkw, G.stage + st * kSt, &G.bar[st], jb, c);
        ld_out[st] = true;
        ld_par[st] = par;
    };
    // Gram MMA of local chunk k (index idx): wait for its stage, do the
    // stage work, issue. A failed wait sets the abort flag, which every
    // later group_any of the group sees.
    auto gram = [&](int k, int idx) {
        const int st = k & 1;
        const uint32_t par = (k >> 1) & 1;
        uint8_t *stage = G.stage + st * kSt;
        bool ok = true;
        if (kStageWork) {
            ok = (lt != 0) || mbar_wait(&G.bar[st], par, kWaitTries, abort);
            if (lt == 0) {
                if (ok) ld_out[st] = false;
                else flag_error(p.status, abort, kDevTimeout);
            }
            if (group_any(G.bar_id, kPrepThreads, !ok || *abort)) return false;
            int c;
            const J jb = job_of(idx, c);
            uint8_t *rec = p.rec + rec_index(p, jb, c) * p.rec_stride;
            if (kPro) {
                normalise_rows(stage, R, ct, p.prologue, lt, kPrepThreads);
                fence_proxy_async_smem();
                named_sync(G.bar_id, kPrepThreads);
                if (kq_in_record(p.prologue))   // the mapped rows, for the state pass
                    for (uint32_t i = lt * 16; i < kRecKQBytes; i += kPrepThreads * 16) {
                        const uint32_t kb = i / kRecKQBlock, off = i - kb * kRecKQBlock;
                        *(uint4 *)(rec + kRecKQ + i) = *(const uint4 *)(stage + kb * kKQBlock + off);
                    }
            }
            if (kWK && !gated)   // the K~ tile, for the state pass (see kRecKW)
                for (uint32_t i = lt * 16; i < 2 * kKWBlock; i += kPrepThreads * 16)
                    *(uint4 *)(rec + kRecKW + i) = *(const uint4 *)(stage + kPGKQ + i);
        }
        if (lt == 0) {
            if (!kStageWork) {
                ok = mbar_wait(&G.bar[st], par, kWaitTries, abort);
                if (ok) ld_out[st] = false;
                else flag_error(p.status, abort, kDevTimeout);
            }
            if (ok) {
                tc_fence_after();
                if (kWK)
                    issue_gram_wk(G.tcol + st * 32, smem_addr(stage), smem_addr(stage + kPGKQ));
                else
                    issue_gram(G.tcol + st * 32, smem_addr(stage));
                mma_commit(&G.bar[2 + st]);
                mma_out[st] = true;
                mma_par[st] = par;
            }
        }
        return true;
    };

    int idx = next_chunk<kPacked, kPro, kWK>(p, first, stride, total);
    bool ok = idx < total;
    int nxt = ok ? next_chunk<kPacked, kPro, kWK>(p, idx + stride, stride, total) : total;
    if (ok && lt == 0) {
        issue_load(idx, 0, 0);
        if (nxt < total) issue_load(nxt, 1, 0);
    }
    RowVals rv{0.f, 0.f};
    if (ok && lt < 32) {
        int c;
        const J jb = job_of(idx, c);
        rv = load_rows(p, jb, c, lane);
    }
    if (ok) ok = gram(0, idx);
    for (int k = 0; ok; ++k) {
        const int st = k & 1;
        // the Gram MMA of chunk k is done
        bool okw = true;
        if (lt == 0) {
            okw = mbar_wait(&G.bar[2 + st], (k >> 1) & 1, kWaitTries, abort);
            if (okw) mma_out[st] = false;
            else flag_error(p.status, abort, kDevTimeout);
        }
        if (group_any(G.bar_id, kPrepThreads, !okw || *abort)) {
            ok = false;
            break;
        }
        tc_fence_after();
        // stage st is free: the tiles of chunk k + 2 go into it
        const int nn = nxt < total ? next_chunk<kPacked, kPro, kWK>(p, nxt + stride, stride, total) : total;
        if (lt == 0 && nn < total) issue_load(nn, st, ((k + 2) >> 1) & 1);
        // the Gram MMA of chunk k + 1 (its tiles were requested one chunk ago)
        if (nxt < total && !(ok = gram(k + 1, nxt))) break;
        // betas and cumulative log-gates of chunk k; those of chunk k + 1 in flight
        if (lt < 32) {
            scan_rows(rv, lane, G.w.beta_s, G.w.L_s);
            rv = RowVals{0.f, 0.f};
            if (nxt < total) {
                int c;
                const J jb = job_of(nxt, c);
                rv = load_rows(p, jb, c, lane);
            }
        }
        named_sync(G.bar_id, kPrepThreads);
        int c;
        const J jb = job_of(idx, c);
        uint8_t *rec = p.rec + rec_index(p, jb, c) * p.rec_stride;
        phase_a(G.w, G.tcol, st * 32, rec + kRecT, lt, p.nh, ct, gated, G.bar_id);
        float *rp = (float *)(rec + kRecP);
        for (int i = lt; i < kNQ * kC; i += kPrepThreads) rp[i] = G.w.Ps[(i >> 5) * kLd + (i & 31)];
        if (lt < kC) {
            ((float *)(rec + kRecBeta))[lt] = G.w.beta_s[lt];
            ((float *)(rec + kRecL))[lt] = G.w.L_s[lt];
        }
        // the record is complete, the scratch and accumulator st free
        tc_fence_before();
        named_sync(G.bar_id, kPrepThreads);
        if (publish && lt == 0 && !(p.withhold_first && idx == 0)) {
            __threadfence();
            flag_publish(p.flags + rec_index(p, jb, c), 1u);
        }
        if (nxt >= total) break;
        idx = nxt;
        nxt = nn;
    }
    if (lt == 0) {   // after a timeout: let what is in flight finish before smem and TMEM go
        uint32_t no_abort = 0;
        for (int st = 0; st < 2; ++st) {
            if (ld_out[st]) mbar_wait(&G.bar[st], ld_par[st], kWaitTries, &no_abort);
            if (mma_out[st]) mbar_wait(&G.bar[2 + st], mma_par[st], kWaitTries, &no_abort);
        }
    }
}

// Split mode: every chunk of every head, by persistent CTAs of one prep
// group each (several per SM).
constexpr uint32_t pk_smem(bool wk)
{
    return 2 * pg_stage_bytes(wk) + kPrepScratch + 4 * 8 + 16 + 1024;
}
constexpr uint32_t kPKTmemCols = 64;

template <bool kPacked, bool kPro, bool kWK = false>
__global__ void __launch_bounds__(kPrepThreads, 4)
chunk_prep_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                  const __grid_constant__ CUtensorMap tm_kw, const Params p)
{
    extern __shared__ uint8_t smem_raw[];
    constexpr uint32_t kSt = pg_stage_bytes(kWK);
    uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t *bar = (uint64_t *)(base + 2 * kSt + kPrepScratch);
    uint32_t *tmem_slot = (uint32_t *)(bar + 4);
    volatile uint32_t *abort = tmem_slot + 1;
    const int lt = threadIdx.x, warp = lt >> 5;

    // rows TMA does not write (padding, queries beyond the chunk) stay zero
    for (uint32_t i = lt * 16; i < 2 * kSt; i += kPrepThreads * 16)
        *(uint4 *)(base + i) = make_uint4(0, 0, 0, 0);
    if (lt == 0) {
        for (int i = 0; i < 4; ++i) mbar_init(&bar[i], 1);
        *abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_q);
        if (kWK) tma_prefetch_desc(&tm_kw);
    }
    if (warp == 0) tmem_alloc(tmem_slot, kPKTmemCols);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;
    const PrepGroup G{base, bar, tbase, prep_scratch(base + 2 * kSt), 1, lt};
    prep_loop<kPacked, kPro, kWK>(p, &tm_k, &tm_q, &tm_kw, G, abort, blockIdx.x, gridDim.x, false);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, kPKTmemCols);
}

// ------------------------------------------------------------------ cooperative mode
// One launch: CTAs 0 .. B*H-1 run the state pass (split mode), the others
// prepare the chunks in chunk-major order, two prep groups per CTA (warps
// 0-7 and 8-15), and publish each record through its flag. The state pass
// waits for a record's flag (bounded) before loading it. All CTAs are
// resident together (cooperative launch), and no prep CTA waits on a
// state-pass CTA. The host zeroes the flags before the launch.
constexpr uint32_t kCoopScratch = (kPrepScratch + 127) & ~127u;

template <bool kPacked, bool kPro, bool kWK>
__device__ void prep_cta(const CUtensorMap &tm_k, const CUtensorMap &tm_q, const CUtensorMap &tm_kw,
                         const Params &p, int pcta, int n_pcta)
{
    extern __shared__ uint8_t smem_raw[];
    constexpr uint32_t kSt = pg_stage_bytes(kWK);
    uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *scr = base + 4 * kSt;                                   // [group 0 stages | group 1 stages]
    uint64_t *bar = (uint64_t *)(scr + 2 * kCoopScratch);            // [group][4]
    uint32_t *tmem_slot = (uint32_t *)(bar + 8);
    volatile uint32_t *abort = tmem_slot + 1;
    const int warp = threadIdx.x >> 5;

    for (uint32_t i = threadIdx.x * 16; i < 4 * kSt; i += kThreads * 16)
        *(uint4 *)(base + i) = make_uint4(0, 0, 0, 0);
    if (threadIdx.x == 0) {
        for (int i = 0; i < 8; ++i) mbar_init(&bar[i], 1);
        *abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_q);
        if (kWK) tma_prefetch_desc(&tm_kw);
    }
    if (warp == 0) tmem_alloc(tmem_slot, 128);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;

    if (warp < 16) {
        const int gi = warp >> 3, lt = threadIdx.x - gi * kPrepThreads;
        const PrepGroup G{base + gi * 2 * kSt, bar + 4 * gi, tbase + gi * 64,
                          prep_scratch(scr + gi * kCoopScratch), (uint32_t)(1 + gi), lt};
        prep_loop<kPacked, kPro, kWK>(p, &tm_k, &tm_q, &tm_kw, G, abort, pcta * 2 + gi, n_pcta * 2, true);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, 128);
}

// ------------------------------------------------------------------ warp-per-chunk prep
// The prep of the plain path (no prologue, no write keys) in the split and
// cooperative modes: each consumer warp solves whole chunks on its own
// (lane i = extended row i), so nothing waits on a group barrier, and
// producer threads keep the loads and Gram MMAs ahead of them.
//  * producer (one per 8 consumer warps, 4 slots; a loader thread and an
//    MMA thread, so that load issue and MMA issue overlap): TMA of the
//    chunk's K and Q tiles into the slot's stage, then one MMA
//    D = [K-rows at the consumer's TMEM lane quarter] x [K; Q]^T (M = 128,
//    N = 48: columns 0-31 the Gram row k_i.k_s, columns 32-47 k_i.q_t); the
//    A operand's start is moved back by 32 rows per quarter so that the K
//    rows land in the lanes the consumer warp may read (the other lanes get
//    rows of neighbouring shared memory and are never read).
//  * consumer warp: the rows' betas and log-gates, G^T (strictly lower
//    part, scaled) into its scratch, the readout weights P straight into the
//    record, then row i of T = (I + G)^-1 by back-substitution (row i needs
//    only G: T[i][j] = -sum_{s>j} T[i][s] G[s][j]), written as the bf16 hi/lo
//    tiles of T diag(beta) (and T diag(beta Gamma)) in the record's
//    swizzled layout; in the cooperative mode it publishes the record.
// Slot s of a producer holds local chunks k = s, s + 4, ... (its (k / 4)-th
// use), with mbarriers "loaded" (TMA bytes) and "free" (the consumer has
// read the accumulator: stage and TMEM columns reusable); the Gram MMA of
// chunk k completes on the mbarrier of its consumer warp k % 8, whose j-th
// phase is that warp's j-th chunk. (A per-slot completion barrier would
// let a warp that finished its chunk on a slot wait for its next one there
// while another warp's chunk still stands in between: two phases ahead,
// which a parity wait cannot tell from the phase before.)
constexpr int kWCons = 16;                       // consumer warps (8 per producer)
constexpr int kWConsPerProd = 8;
constexpr int kWSlots = 4;                       // slots per producer
constexpr int kWLg = 36;                         // G^T row stride (floats; 16-byte aligned rows)
constexpr uint32_t kWScr = 5120;                 // per consumer warp: G^T [32][36], L [32], beta [32]
constexpr uint32_t kWStage = 2 * kKQBlock;       // 16 KB: the KQ tiles
constexpr uint32_t kWStages = 8 * kWScr;         // stages after consumers 0-7's scratch (>= 12 KB lead)
constexpr uint32_t kWScr2 = kWStages + 2 * kWSlots * kWStage;   // consumers 8-15 (>= 8 KB tail)
constexpr uint32_t kWBar = kWScr2 + 8 * kWScr;
constexpr int kWBars = 2 * kWSlots + kWConsPerProd;   // per producer: [slot][loaded, free], [consumer] Gram done
constexpr uint32_t kWSmem = kWBar + 2 * kWBars * 8 + 16 + 1024;
static_assert(kWStages % 1024 == 0 && kWStages >= 3 * 4096, "stage alignment and A-shift lead");
// the M = 128 A operand of the last stage's second block (quarter 0) reads 16 KB from its start
static_assert(kWStages + (2 * kWSlots - 1) * kWStage + kKQBlock + 16 * 1024 <= kWBar, "A-operand tail");

static_assert(kWSmem <= smem_bytes<true>(), "the warp prep fits the cooperative kernel's shared memory");

__device__ __forceinline__ uint8_t *wprep_scratch(uint8_t *base, int w)
{
    return base + (w < 8 ? w * kWScr : kWScr2 + (w - 8) * kWScr);
}

// The chunk-index stream of producer `pr`: every (2 n_pcta)-th chunk from
// 2 pcta + pr, skipping chunks that do not exist (packed calls).
template <bool kPacked>
__device__ __forceinline__ int wstream_next(const Params &p, int idx, int stride, int total)
{
    return next_chunk<kPacked, false, false>(p, idx, stride, total);
}

// Producer pr's loader thread: the K and Q tiles of its chunks into the
// slots' stages, each slot once the consumer of the chunk four back has read
// its accumulator (which also means the Gram MMA that read the stage is done).
template <bool kPacked>
__device__ void wprep_loader(const Params &p, const CUtensorMap *tk, const CUtensorMap *tq, uint8_t *base,
                             uint64_t *bar, int pr, int first, int stride, volatile uint32_t *abort)
{
    using J = Job<kPacked, false, false>;
    const int total = p.n_chunks * p.bh_count, ct = p.ct, R = ct * p.nh;
    bool ok = true;
    int issued = 0;
    int idx = wstream_next<kPacked>(p, first, stride, total);
    for (int k = 0; idx < total; ++k) {
        const int sl = k & (kWSlots - 1);
        if (k >= kWSlots && !(ok = mbar_wait(&bar[sl * 2 + 1], ((k >> 2) - 1) & 1, kWaitTries, abort))) break;
        const int c = idx / p.bh_count;
        const J jb = make_job<kPacked, false, false>(p, idx - c * p.bh_count);
        const int t0 = jb.first() + c * ct;
        if (p.flags && c >= kPaceLead && c - kPaceLead < jb.chunks(p)) {
            // cooperative mode: no further than kPaceLead chunks ahead of the head's state pass
            const uint32_t *f = p.flags + rec_index(p, jb, c - kPaceLead);
            uint32_t tries = 0;
            while (flag_peek(f) != 2u && ++tries < p.flag_tries && !*abort) __nanosleep(128);
            if (flag_peek(f) != 2u) { ok = false; break; }
        }
        uint64_t *lb = &bar[sl * 2 + 0];
        uint8_t *stg = base + kWStages + (pr * kWSlots + sl) * kWStage;
        mbar_arrive_expect_tx(lb, 256u * R + 256u * ct);
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
            tma_load_5d(stg + kb * kKQBlock, tk, lb, kb * 64, 0, jb.h, t0, jb.row_b());
            tma_load_4d(stg + kb * kKQBlock + kC * 128, tq, lb, kb * 64, jb.h, t0, jb.row_b());
        }
        issued = k + 1;
        idx = wstream_next<kPacked>(p, idx + stride, stride, total);
    }
    if (!ok) {   // a wait expired: record it; the loads in flight land before smem goes
        flag_error(p.status, abort, kDevTimeout);
        uint32_t no_abort = 0;
        for (int k = issued > kWSlots ? issued - kWSlots : 0; k < issued; ++k)
            mbar_wait(&bar[(k & (kWSlots - 1)) * 2 + 0], (k >> 2) & 1, kWaitTries, &no_abort);
    }
}

// Producer pr's MMA thread: the Gram MMA of each chunk once its tiles have
// landed (the loader only refills a slot after its accumulator was read, so
// the MMA never overwrites one still needed), completing on the consumer
// warp's barrier.
template <bool kPacked>
__device__ void wprep_mma(const Params &p, uint8_t *base, uint64_t *bar, uint32_t tcol, int pr, int first, int stride,
                          volatile uint32_t *abort)
{
    const int total = p.n_chunks * p.bh_count;
    const uint32_t idesc = idesc_bf16(128, kC + kNQ, false, false);
    bool ok = true;
    int issued = 0;
    int idx = wstream_next<kPacked>(p, first, stride, total);
    for (int k = 0; idx < total; ++k) {
        const int sl = k & (kWSlots - 1);
        if (!(ok = mbar_wait(&bar[sl * 2 + 0], (k >> 2) & 1, kWaitTries, abort))) break;
        tc_fence_after();
        const int q = (pr * kWConsPerProd + (k & (kWConsPerProd - 1))) & 3;   // consumer warp's lane quarter
        const uint32_t st = smem_addr(base + kWStages + (pr * kWSlots + sl) * kWStage);
        const uint32_t d = tcol + sl * 64;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * kKQBlock + (kk & 3) * 32;
            mma_ss(d, sdesc_sw128(st + off - 4096u * q, 16, 1024), sdesc_sw128(st + off, 16, 1024), idesc, kk > 0);
        }
        mma_commit(&bar[2 * kWSlots + (k & (kWConsPerProd - 1))]);
        issued = k + 1;
        idx = wstream_next<kPacked>(p, idx + stride, stride, total);
    }
    if (!ok) {   // a wait expired: record it; the MMAs issued retire before TMEM goes
        flag_error(p.status, abort, kDevTimeout);
        uint32_t no_abort = 0;
        for (int k = issued > kWConsPerProd ? issued - kWConsPerProd : 0; k < issued; ++k)
            mbar_wait(&bar[2 * kWSlots + (k & (kWConsPerProd - 1))], (k >> 3) & 1, kWaitTries, &no_abort);
    }
}

template <bool kPacked>
__device__ void wprep_consumer(const Params &p, uint8_t *scr, uint64_t *bar, uint32_t tcol, int w, int first,
                               int stride, bool publish, volatile uint32_t *abort)
{
    using J = Job<kPacked, false, false>;
    const int lane = threadIdx.x & 31, q = w & 3, lc = w & (kWConsPerProd - 1);
    const int total = p.n_chunks * p.bh_count, nh = p.nh, ct = p.ct;
    const bool gated = p.g != nullptr;
    float *Gt = (float *)scr, *Ls = Gt + 32 * kWLg, *Bs = Ls + 32;
    int idx = wstream_next<kPacked>(p, first, stride, total);
    for (int k = 0; k < lc && idx < total; ++k) idx = wstream_next<kPacked>(p, idx + stride, stride, total);
    for (int k = lc; idx < total; k += kWConsPerProd) {
        const int sl = k & (kWSlots - 1);
        const int c = idx / p.bh_count;
        const J jb = make_job<kPacked, false, false>(p, idx - c * p.bh_count);
        const RowVals rv = load_rows(p, jb, c, lane);
        bool ok = true;
        if (lane == 0) {
            ok = mbar_wait(&bar[2 * kWSlots + lc], (k >> 3) & 1, kWaitTries, abort);
            if (!ok) flag_error(p.status, abort, kDevTimeout);
        }
        if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0) || *abort) break;
        tc_fence_after();
        uint32_t gr[32], pt[16];
        const uint32_t ta = tcol + sl * 64 + ((uint32_t)(32 * q) << 16);
        tmem_ld16(ta, *reinterpret_cast<uint32_t(*)[16]>(&gr[0]));
        tmem_ld16(ta + 16, *reinterpret_cast<uint32_t(*)[16]>(&gr[16]));
        tmem_ld16(ta + 32, pt);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[sl * 2 + 1]);   // accumulator read: the slot may be reused
        // betas and cumulative log-gates (lane = row), as scan_rows computes them
        float L = rv.lg;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, L, d);
            if (lane >= d) L += y;
        }
        Ls[lane] = L;
        Bs[lane] = rv.beta;
        __syncwarp();
        uint8_t *rec = p.rec + rec_index(p, jb, c) * p.rec_stride;
        // G^T[j][i] = G[i][j] = beta_i (k_i.k_j) E_ij for j < i, 0 otherwise
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            float gv = 0.f;
            if (j < lane) {
                gv = rv.beta * __uint_as_float(gr[j]);
                if (gated) gv *= __expf(L - Ls[j]);
            }
            Gt[j * kWLg + lane] = gv;
        }
        // readout weights P[t][s] (lane = s): (q_t.k_s) E_{r(t) s} for s <= r(t), the token's last row
        float *rp = (float *)(rec + kRecP);
#pragma unroll
        for (int t = 0; t < kNQ; ++t) {
            const int rr = t * nh + nh - 1;
            float x = 0.f;
            if (t < ct && lane <= rr) {
                x = __uint_as_float(pt[t]);
                if (gated) x *= __expf(Ls[rr] - L);
            }
            rp[t * kC + lane] = x;
        }
        ((float *)(rec + kRecBeta))[lane] = rv.beta;
        ((float *)(rec + kRecL))[lane] = L;
        __syncwarp();
        // row `lane` of T = (I + G)^-1: T[i][j] = -sum_{s > j} T[i][s] G[s][j] for j < i
        float t[32];
#pragma unroll
        for (int s2 = 0; s2 < 32; ++s2) t[s2] = (s2 == lane) ? 1.f : 0.f;
#pragma unroll
        for (int j = 30; j >= 0; --j) {
            const float *row = Gt + j * kWLg;
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int c4 = (j + 1) >> 2; c4 < 8; ++c4) {
                const float4 v = *(const float4 *)(row + 4 * c4);
                const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int s2 = 4 * c4 + e;
                    if (s2 > j) {
                        if (e & 1) a1 = fmaf(t[s2], vv[e], a1);
                        else a0 = fmaf(t[s2], vv[e], a0);
                    }
                }
            }
            if (j < lane) t[j] = -(a0 + a1);
        }
        // T diag(beta) and T diag(beta Gamma): bf16 hi + lo tiles, row `lane`
#pragma unroll
        for (int pr = 0; pr < 2; ++pr) {
            if (pr == 1 && !gated) break;
            uint8_t *hi = rec + kRecT + 2 * pr * kTTile, *lo = hi + kTTile;
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
                uint32_t wh[4], wl[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int s0 = ch * 8 + 2 * e;
                    float v0 = t[s0] * Bs[s0], v1 = t[s0 + 1] * Bs[s0 + 1];
                    if (pr) {
                        v0 *= __expf(Ls[s0]);
                        v1 *= __expf(Ls[s0 + 1]);
                    }
                    split_pack(v0, v1, wh[e], wl[e]);
                }
                *(uint4 *)(hi + sw128_offset(lane, ch)) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
                *(uint4 *)(lo + sw128_offset(lane, ch)) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
            }
        }
        __syncwarp();   // every lane's record writes happen before the publication
        if (publish && lane == 0 && !(p.withhold_first && idx == 0)) {
            __threadfence();
            flag_publish(p.flags + rec_index(p, jb, c), 1u);
        }
        for (int n = 0; n < kWConsPerProd && idx < total; ++n)
            idx = wstream_next<kPacked>(p, idx + stride, stride, total);
    }
}

// A prep CTA (kThreads threads): warps 0-15 consumers; for consumers 0-7
// and 8-15 the MMA threads of warps 16 and 17 and the loader threads of
// warps 18 and 19. Producer pr's chunk stream is every
// (2 n_pcta)-th chunk of the chunk-major order from 2 pcta + pr.
template <bool kPacked>
__device__ void wprep_cta(const CUtensorMap &tm_k, const CUtensorMap &tm_q, const Params &p, int pcta, int n_pcta,
                          bool publish)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t *bar = (uint64_t *)(base + kWBar);   // [producer][kWBars]
    uint32_t *tmem_slot = (uint32_t *)(bar + 2 * kWBars);
    volatile uint32_t *abort = tmem_slot + 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // rows TMA does not write (K padding rows, queries beyond the chunk) stay zero
    for (uint32_t i = threadIdx.x * 16; i < 2 * kWSlots * kWStage; i += kThreads * 16)
        *(uint4 *)(base + kWStages + i) = make_uint4(0, 0, 0, 0);
    if (threadIdx.x == 0) {
        for (int i = 0; i < 2 * kWBars; ++i) mbar_init(&bar[i], 1);
        *abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_q);
    }
    if (warp == 0) tmem_alloc(tmem_slot, 512);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;
    if (warp < kWCons) {
        const int pr = warp / kWConsPerProd;
        wprep_consumer<kPacked>(p, wprep_scratch(base, warp), bar + pr * kWBars, tbase + pr * 256, warp,
                                2 * pcta + pr, 2 * n_pcta, publish, abort);
    } else if (warp < kWCons + 2 && lane == 0) {
        const int pr = warp - kWCons;
        wprep_mma<kPacked>(p, base, bar + pr * kWBars, tbase + pr * 256, pr, 2 * pcta + pr, 2 * n_pcta, abort);
    } else if (warp < kWCons + 4 && lane == 0) {
        const int pr = warp - kWCons - 2;
        wprep_loader<kPacked>(p, &tm_k, &tm_q, base, bar + pr * kWBars, pr, 2 * pcta + pr, 2 * n_pcta, abort);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, 512);
}

// Split mode, plain path: one warp-per-chunk prep CTA per SM.
template <bool kPacked>
__global__ void __launch_bounds__(kThreads, 1)
chunk_wprep_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q, const Params p)
{
    wprep_cta<kPacked>(tm_k, tm_q, p, blockIdx.x, gridDim.x, false);
}

// ------------------------------------------------------------------ segmented mode
// For sequences too few to fill the GPU, each (b, h) sequence is cut into P
// segments of whole chunks, and the recurrence's affine form (DeltaProduct
// paper, Sec.2 Eq.(1): S_end = A S_start + B per segment, associative)
// lets the segments run at once:
//  1. state pass (chunk_seg_kernel, one CTA per job): segment 0 from h0,
//     writing o; every later segment twice, from a zero state (part 0:
//     readout o0, end state B_s) and, with its values left out, from the
//     identity (part 1: end state A_s, readout q~_t = A_{<=t}^T q_t);
//  2. seg_combine_kernel: S_1 = segment 0's end state, S_{s+1} = A_s S_s +
//     B_s, in order (fp32, CUDA cores); S_s^T for the correction, S_P is
//     h_final;
//  3. seg_correct_kernel: o_t = o0_t + S_s^T q~_t for the tokens of segment
//     s >= 1 (tf32 tensor-core MMA per tile of 128 tokens).
template <typename TOut>
__global__ void __launch_bounds__(kThreads, 1)
chunk_seg_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                 const __grid_constant__ CUtensorMap tm_q, const Params p)
{
    state_pass_cta<TOut, true, false, false, false, false, true>(tm_k, tm_v, tm_q, p, blockIdx.x);
}

constexpr int kCombThreads = 256;
constexpr int kCombLd = kD + 4;                          // A row stride in shared memory (floats)
constexpr uint32_t kCombSmem = (kD * kCombLd + kD * 33) * 4;
// grid: B*H x 4 blocks of 32 value columns (the columns of the state evolve
// independently: S[:, J] <- A S[:, J] + B[:, J]); A_s is staged in shared
// memory by coalesced loads, the block of S stays there.
__global__ void __launch_bounds__(kCombThreads)
seg_combine_kernel(const float *seg_h, float *seg_st, float *h_final, int P)
{
    extern __shared__ float comb_smem[];
    float *As = comb_smem;                               // [kD][kCombLd]
    float(*S)[33] = reinterpret_cast<float(*)[33]>(comb_smem + kD * kCombLd);
    const int bh = blockIdx.x >> 2, vb = (blockIdx.x & 3) * 32, tid = threadIdx.x;
    const float *base = seg_h + (size_t)bh * P * 2 * kD * kD;
    for (int i = tid; i < kD * 32; i += kCombThreads) S[i >> 5][i & 31] = base[(size_t)(i >> 5) * kD + vb + (i & 31)];
    __syncthreads();
    const int row = tid >> 1, v0 = (tid & 1) * 16;
    for (int sg = 1; sg < P; ++sg) {
        // start state of segment sg, transposed: [v][k]
        float *st = seg_st + ((size_t)bh * P + sg) * kD * kD;
        for (int i = tid; i < kD * 32; i += kCombThreads) st[(size_t)(vb + (i >> 7)) * kD + (i & 127)] = S[i & 127][i >> 7];
        const float *A = base + ((size_t)sg * 2 + 1) * kD * kD;
        for (int i = tid; i < kD * kD / 4; i += kCombThreads) {
            const float4 a = __ldg((const float4 *)A + i);
            *(float4 *)(As + (i >> 5) * kCombLd + 4 * (i & 31)) = a;
        }
        const float *Bm = base + ((size_t)sg * 2) * kD * kD + (size_t)row * kD + vb + v0;
        float acc[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) acc[j] = __ldg(Bm + j);
        __syncthreads();
        const float *Ar = As + row * kCombLd;
        for (int k4 = 0; k4 < kD / 4; ++k4) {
            const float4 a = *(const float4 *)(Ar + 4 * k4);
            const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
#pragma unroll
                for (int j = 0; j < 16; ++j) acc[j] = fmaf(av[e], S[4 * k4 + e][v0 + j], acc[j]);
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < 16; ++j) S[row][v0 + j] = acc[j];
        __syncthreads();
    }
    if (h_final)
        for (int i = tid; i < kD * 32; i += kCombThreads)
            h_final[(size_t)bh * kD * kD + (size_t)(i >> 5) * kD + vb + (i & 31)] = S[i >> 5][i & 31];
}

constexpr int kCorrTok = 64;                             // tokens per tile (two CTAs per SM)
constexpr uint32_t kCorrBlock = 128 * 128;               // A: 128 rows x 32 fp32
constexpr uint32_t kCorrBBlock = kCorrTok * 128;         // B: kCorrTok rows x 32 fp32
constexpr uint32_t kCorrSmem = 4 * kCorrBlock + 4 * kCorrBBlock + 2 * 8 + 16 + 1024;

template <typename TOut>
__global__ void __launch_bounds__(128, 2)
seg_correct_kernel(const __grid_constant__ CUtensorMap tm_st, const __grid_constant__ CUtensorMap tm_qt,
                   const Params p, int tiles)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *sA = base, *sB = base + 4 * kCorrBlock;    // S_s^T (rows v), q~ tile (rows t)
    uint64_t *bar = (uint64_t *)(sB + 4 * kCorrBBlock);
    uint32_t *tmem_slot = (uint32_t *)(bar + 2);
    volatile uint32_t *abort = tmem_slot + 1;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int tile = blockIdx.x % tiles, r = blockIdx.x / tiles, nseg = p.seg_count - 1;
    const int sg = 1 + r % nseg, bh = r / nseg, b = bh / p.H, h = bh - b * p.H;
    const int seg0 = sg * p.seg_chunks * p.ct, seg_len = min(p.seg_chunks * p.ct, p.T - seg0);
    const int tok0 = seg0 + tile * kCorrTok, ntok = min(kCorrTok, seg_len - tile * kCorrTok);
    if (ntok <= 0) return;   // the same for the whole CTA
    if (tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        *abort = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(tmem_slot, kCorrTok);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;
    // every thread's o0 values (lane = value column v, kCorrTok tokens) are
    // fetched before the tiles land and the MMAs run, so that their DRAM
    // latency overlaps those
    const size_t tok_stride = (size_t)p.H * kD;
    const size_t row0 = (((size_t)b * p.T + tok0) * p.H + h) * kD + tid;
    float a[kCorrTok];
#pragma unroll
    for (int j = 0; j < kCorrTok; ++j) a[j] = j < ntok ? __ldg(p.seg_o0 + row0 + (size_t)j * tok_stride) : 0.f;
    bool ok = true;
    if (tid == 0) {
        mbar_arrive_expect_tx(&bar[0], 4 * kCorrBlock + 4 * kCorrBBlock);
#pragma unroll
        for (int kb = 0; kb < 4; ++kb) {
            tma_load_3d(sA + kb * kCorrBlock, &tm_st, &bar[0], kb * 32, 0, bh * p.seg_count + sg);
            tma_load_4d(sB + kb * kCorrBBlock, &tm_qt, &bar[0], kb * 32, h, tok0, b);
        }
        uint32_t no_abort = 0;
        ok = mbar_wait(&bar[0], 0, kWaitTries, &no_abort);
        if (ok) {
            tc_fence_after();
            const uint32_t idesc = idesc_tf32(128, kCorrTok);
#pragma unroll
            for (int kk = 0; kk < 16; ++kk) {
                const uint32_t ka = (kk >> 2) * kCorrBlock + (kk & 3) * 32, kb = (kk >> 2) * kCorrBBlock + (kk & 3) * 32;
                mma_ss_tf32(tbase, sdesc_sw128(smem_addr(sA) + ka, 16, 1024), sdesc_sw128(smem_addr(sB) + kb, 16, 1024),
                            idesc, kk > 0);
            }
            mma_commit(&bar[1]);
            ok = mbar_wait(&bar[1], 0, kWaitTries, &no_abort);
        }
        if (!ok) {
            if (p.status) atomicCAS(p.status, 0u, kDevTimeout);
            *abort = 1;
            mbar_wait(&bar[0], 0, kWaitTries, &no_abort);   // let what is in flight land
            mbar_wait(&bar[1], 0, kWaitTries, &no_abort);
        }
    }
    __syncthreads();
    tc_fence_after();
    if (!*abort) {
        // lane = value column v; TMEM column = token of the tile
        const uint32_t trow = tbase + ((uint32_t)(warp * 32) << 16);
#pragma unroll
        for (int c0 = 0; c0 < kCorrTok; c0 += 32) {
            uint32_t d[32];
            tmem_ld32(trow + c0, d);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (c0 + j < ntok)
                    store_out((TOut *)p.o, row0 + (size_t)(c0 + j) * tok_stride, __uint_as_float(d[j]) + a[c0 + j]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, kCorrTok);
}

template <typename TOut, bool kPacked, bool kPro, bool kWK = false>
__global__ void __launch_bounds__(kThreads, 1)
chunk_coop_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kw,
                  const Params p)
{
    if ((int)blockIdx.x < p.bh_count)
        state_pass_cta<TOut, true, true, kPacked, kPro, kWK>(tm_k, tm_v, tm_q, p, blockIdx.x);
    else if (!kPro && !kWK)
        wprep_cta<kPacked>(tm_k, tm_q, p, blockIdx.x - p.bh_count, gridDim.x - p.bh_count, true);
    else
        prep_cta<kPacked, kPro, kWK>(tm_k, tm_q, tm_kw, p, blockIdx.x - p.bh_count, gridDim.x - p.bh_count);
}

}  // namespace

namespace {
std::atomic<uint32_t> g_fault_tries{0};
std::atomic<int> g_fault_withhold{0};
}  // namespace

CoopFault coop_fault() { return {g_fault_tries.load(), g_fault_withhold.load()}; }

void set_coop_fault(CoopFault f)
{
    g_fault_tries.store(f.flag_tries);
    g_fault_withhold.store(f.withhold_first);
}

bool chunk_tc_supported(const Problem &p)
{
    return p.dtype == DP_BF16 && p.Dk == kD && p.Dv == kD && p.nh >= 1 && p.nh <= 4 && p.T > 0 &&
           tensor_map_encoder() != nullptr;
}

namespace {
int chunk_tokens(int nh) { return (kC / nh < kNQ) ? kC / nh : kNQ; }
}  // namespace

namespace {
size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }
// Records are laid out for the longest sequence: ceil(max_T / ct) per (sequence, head).
size_t chunks_per_seq(const Problem &p)
{
    const int ct = chunk_tokens(p.nh);
    return p.T > 0 ? (size_t)(p.max_T + ct - 1) / ct : 0;
}
size_t n_chunks_total(const Problem &p) { return (size_t)p.B * p.H * chunks_per_seq(p); }
}  // namespace

// Records, then one flag per chunk (cooperative mode).
size_t chunk_tc_records_bytes(const Problem &p)
{
    const size_t n = n_chunks_total(p);
    return n ? round256(n * record_stride(p.prologue)) + round256(n * 4) : 0;
}

namespace {
constexpr int kSegMinChunks = 16;   // shortest segment worth a CTA pair

// Segments per sequence for the segmented mode (>= 2) and their length in
// chunks, or 0 when the mode does not apply: dense plain problems whose
// B*H (2P - 1) state-pass CTAs fit the SMs at once with P >= 2.
int seg_plan(const Problem &p, int *seg_chunks)
{
    *seg_chunks = 0;
    if (p.cu || p.prologue || p.kw || p.T <= 0) return 0;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    const long long bh = (long long)p.B * p.H, nch = (long long)chunks_per_seq(p);
    if (bh <= 0) return 0;
    long long P = (sms / bh + 1) / 2;
    if (P > nch / kSegMinChunks) P = nch / kSegMinChunks;
    // two segments do not pay for the separate prep, combine and correction
    // (measured: the cooperative launch is faster there)
    if (P < 3) return 0;
    const long long L = (nch + P - 1) / P;
    P = (nch + L - 1) / L;   // no empty segment
    if (P < 3) return 0;
    *seg_chunks = (int)L;
    return (int)P;
}

// Segmented-mode workspace after the status block: records, the parts' end
// states [B*H][P][2] and the start states S_s^T [B*H][P] (D x D fp32 each),
// the two fp32 readouts of o's size.
struct SegLayout {
    size_t rec, h, st, o0, qt, total;
};
SegLayout seg_layout(const Problem &p, int P)
{
    const size_t bh = (size_t)p.B * p.H, d2 = (size_t)kD * kD * 4, tok = (size_t)p.B * p.T * p.H * kD * 4;
    SegLayout l;
    l.rec = 0;
    l.h = round256(n_chunks_total(p) * record_stride(0));
    l.st = l.h + round256(bh * P * 2 * d2);
    l.o0 = l.st + round256(bh * P * d2);
    l.qt = l.o0 + round256(tok);
    l.total = l.qt + round256(tok);
    return l;
}
}  // namespace

size_t chunk_tc_fast_bytes(const Problem &p)
{
    size_t r = chunk_tc_records_bytes(p);
    int L = 0;
    const int P = seg_plan(p, &L);
    if (P >= 2) {
        const size_t sb = seg_layout(p, P).total;
        if (sb > r) r = sb;
    }
    return r;
}

namespace {
// The kernel instantiation for a problem: output type, mode, packed
// offsets, input prologue; write keys (dense, no prologue, split modes).
template <typename TOut, bool kSplit>
auto tc_kernel_mode(bool packed, bool pro)
{
    return packed ? (pro ? chunk_tc_kernel<TOut, kSplit, true, true> : chunk_tc_kernel<TOut, kSplit, true, false>)
                  : (pro ? chunk_tc_kernel<TOut, kSplit, false, true> : chunk_tc_kernel<TOut, kSplit, false, false>);
}
template <typename TOut>
auto tc_kernel_for(bool split, bool packed, bool pro, bool wk)
{
    if (wk) return chunk_tc_kernel<TOut, true, false, false, true>;
    return split ? tc_kernel_mode<TOut, true>(packed, pro) : tc_kernel_mode<TOut, false>(packed, pro);
}
template <typename TOut>
auto coop_kernel_typed(bool packed, bool pro)
{
    return packed ? (pro ? chunk_coop_kernel<TOut, true, true> : chunk_coop_kernel<TOut, true, false>)
                  : (pro ? chunk_coop_kernel<TOut, false, true> : chunk_coop_kernel<TOut, false, false>);
}
auto coop_kernel_for(const Problem &p)
{
    const bool packed = p.cu != nullptr, pro = p.prologue != 0, f32 = p.out_dtype == DP_F32;
    if (p.kw) return f32 ? chunk_coop_kernel<float, false, false, true> : chunk_coop_kernel<__nv_bfloat16, false, false, true>;
    return f32 ? coop_kernel_typed<float>(packed, pro) : coop_kernel_typed<__nv_bfloat16>(packed, pro);
}

// Grid of the cooperative launch (state-pass CTAs + prep CTAs), or 0 when
// this problem and device do not take it.
cudaError_t coop_grid(const Problem &p, long long *grid)
{
    *grid = 0;
    const size_t n_total = n_chunks_total(p);
    if (n_total == 0 || p.scratch_bytes < chunk_tc_records_bytes(p)) return cudaSuccess;
    int dev = 0, sms = 0, coop = 0, per_sm = 0;
    auto kernel = coop_kernel_for(p);
    const uint32_t smem = smem_bytes<true>();
    cudaError_t e;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev)) != cudaSuccess ||
        (e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess ||
        (e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, smem)) != cudaSuccess)
        return e;
    const long long bh = (long long)p.B * p.H, slots = (long long)sms * per_sm;
    if (coop && per_sm >= 1 && 2 * bh <= slots) {
        const long long want_prep = ((long long)n_total + 1) / 2;
        *grid = bh + (slots - bh < want_prep ? slots - bh : want_prep);
    }
    return cudaSuccess;
}
}  // namespace

cudaError_t chunk_tc_path(const Problem &p, int *path)
{
    int L = 0;
    const int P = seg_plan(p, &L);
    if (P >= 2 && p.scratch_bytes >= seg_layout(p, P).total) {
        *path = DP_PATH_CHUNK_SEG;
        return cudaSuccess;
    }
    long long grid = 0;
    const cudaError_t e = coop_grid(p, &grid);
    if (e != cudaSuccess) return e;
    const size_t n_total = n_chunks_total(p);
    if (grid > 0)
        *path = DP_PATH_CHUNK_COOP;
    else if (n_total > 0 && p.scratch_bytes >= round256(n_total * record_stride(p.prologue)))
        *path = DP_PATH_CHUNK_SPLIT;
    else
        *path = DP_PATH_CHUNK_FUSED;
    return cudaSuccess;
}

namespace {
// Segmented mode (see seg_combine_kernel): prep of every chunk, the state
// pass over B*H (2P - 1) jobs, the combine, the correction.
cudaError_t launch_segmented(const Problem &p, Params pr, const CUtensorMap &tk, const CUtensorMap &tv,
                             const CUtensorMap &tq, int P, int L, const SegLayout &lay)
{
    uint8_t *ws = (uint8_t *)p.scratch;
    pr.rec = ws + lay.rec;
    pr.seg_count = P;
    pr.seg_chunks = L;
    pr.seg_h = (float *)(ws + lay.h);
    pr.seg_o0 = (float *)(ws + lay.o0);
    pr.seg_qt = (float *)(ws + lay.qt);
    float *seg_st = (float *)(ws + lay.st);
    const size_t n_total = n_chunks_total(p), bh = (size_t)p.B * p.H;
    cudaError_t e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return e;
    {   // 1. records
        auto prep = chunk_wprep_kernel<false>;
        if ((e = cudaFuncSetAttribute(prep, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kWSmem)) != cudaSuccess)
            return e;
        const unsigned n_ctas = (unsigned)((n_total + 1) / 2 < (size_t)sms ? (n_total + 1) / 2 : sms);
        prep<<<n_ctas, kThreads, kWSmem, p.stream>>>(tk, tq, pr);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    {   // 2. state pass of every job
        auto kernel = p.out_dtype == DP_F32 ? chunk_seg_kernel<float> : chunk_seg_kernel<__nv_bfloat16>;
        const uint32_t smem = smem_bytes<true>();
        if ((e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
            return e;
        kernel<<<(unsigned)(bh * (2 * P - 1)), kThreads, smem, p.stream>>>(tk, tv, tq, pr);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    // 3. start states and the final state
    if ((e = cudaFuncSetAttribute(seg_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kCombSmem)) !=
        cudaSuccess)
        return e;
    seg_combine_kernel<<<(unsigned)(bh * 4), kCombThreads, kCombSmem, p.stream>>>(pr.seg_h, seg_st, p.h_final, P);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    {   // 4. correction of the outputs of segments >= 1
        CUtensorMap tm_st, tm_qt;
        const cuuint64_t dst[3] = {kD, kD, (cuuint64_t)bh * P};
        const cuuint64_t sst[2] = {kD * 4, kD * kD * 4};
        const cuuint32_t bst[3] = {32, 128, 1};
        const cuuint64_t dqt[4] = {kD, (cuuint64_t)p.H, (cuuint64_t)p.T, (cuuint64_t)p.B};
        const cuuint64_t sqt[3] = {kD * 4, (cuuint64_t)p.H * kD * 4, (cuuint64_t)p.T * p.H * kD * 4};
        const cuuint32_t bqt[4] = {32, 1, (cuuint32_t)kCorrTok, 1};
        if (!encode(&tm_st, seg_st, 3, dst, sst, bst, CU_TENSOR_MAP_DATA_TYPE_FLOAT32) ||
            !encode(&tm_qt, pr.seg_qt, 4, dqt, sqt, bqt, CU_TENSOR_MAP_DATA_TYPE_FLOAT32))
            return cudaErrorInvalidValue;
        const int tiles = (L * pr.ct + kCorrTok - 1) / kCorrTok;
        auto kernel = p.out_dtype == DP_F32 ? seg_correct_kernel<float> : seg_correct_kernel<__nv_bfloat16>;
        if ((e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kCorrSmem)) != cudaSuccess)
            return e;
        const size_t grid = bh * (P - 1) * tiles;
        if (grid > 0x7fffffffu) return cudaErrorInvalidValue;
        kernel<<<(unsigned)grid, 128, kCorrSmem, p.stream>>>(tm_st, tm_qt, pr, tiles);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}
}  // namespace

cudaError_t launch_chunk_tc(const Problem &p)
{
    const int nh = p.nh, ct = chunk_tokens(nh);
    // packed calls: one batch row of T tokens, sequences found through cu
    const cuuint64_t B = p.cu ? 1 : p.B, T = p.T, H = p.H;
    CUtensorMap tk, tv, tq, tkw;
    const cuuint64_t dk[5] = {kD, (cuuint64_t)nh, H, T, B};
    const cuuint64_t sk[4] = {kD * 2, (cuuint64_t)nh * kD * 2, H * nh * kD * 2, T * H * nh * kD * 2};
    const cuuint32_t bk[5] = {64, (cuuint32_t)nh, 1, (cuuint32_t)ct, 1};
    const cuuint64_t dq[4] = {kD, H, T, B};
    const cuuint64_t sq[3] = {kD * 2, H * kD * 2, T * H * kD * 2};
    const cuuint32_t bq[4] = {64, 1, (cuuint32_t)ct, 1};
    if (!encode(&tk, p.k, 5, dk, sk, bk) || !encode(&tv, p.v, 5, dk, sk, bk) ||
        !encode(&tq, p.q, 4, dq, sq, bq) || !encode(&tkw, p.kw ? p.kw : p.k, 5, dk, sk, bk))
        return cudaErrorInvalidValue;
    Params pr;
    pr.beta = (const __nv_bfloat16 *)p.beta;
    pr.g = (const __nv_bfloat16 *)p.g;
    pr.h0 = p.h0;
    pr.o = p.o;
    pr.h_final = p.h_final;
    pr.status = p.status;
    pr.rec = (uint8_t *)p.scratch;
    pr.flags = nullptr;
    pr.flag_tries = kFlagTries;
    pr.withhold_first = 0;
    pr.bh_count = p.B * p.H;
    pr.cu = p.cu;
    pr.B = p.B;
    pr.T = p.T;
    pr.H = p.H;
    pr.nh = nh;
    pr.ct = ct;
    pr.max_T = p.max_T;
    pr.prologue = p.prologue;
    pr.rec_stride = record_stride(p.prologue);
    pr.kw = (const __nv_bfloat16 *)p.kw;
    pr.n_chunks = (int)chunks_per_seq(p);

    pr.seg_count = pr.seg_chunks = 0;
    pr.seg_h = pr.seg_o0 = pr.seg_qt = nullptr;
    const size_t n_total = n_chunks_total(p);
    cudaError_t e;
    {
        int L = 0;
        const int P = seg_plan(p, &L);
        if (P >= 2 && p.scratch != nullptr && p.scratch_bytes >= seg_layout(p, P).total)
            return launch_segmented(p, pr, tk, tv, tq, P, L, seg_layout(p, P));
    }
    // split whenever the workspace holds every chunk's record; cooperative
    // (one launch) when it also holds the flags and the heads leave at least
    // as many SMs for the prep CTAs as the state pass takes
    const size_t rec_bytes = round256(n_total * record_stride(p.prologue));
    const bool split = p.scratch != nullptr && n_total > 0 && p.scratch_bytes >= rec_bytes;
    // write keys: the split modes only (dense, no prologue; checked by the caller)
    if (p.kw && (!split || p.cu || p.prologue)) return cudaErrorInvalidValue;
    long long grid = 0;
    if (split && (e = coop_grid(p, &grid)) != cudaSuccess) return e;
    if (grid > 0) {
        auto kernel = coop_kernel_for(p);
        pr.flags = (uint32_t *)((uint8_t *)p.scratch + rec_bytes);
        const CoopFault f = coop_fault();
        if (f.flag_tries) pr.flag_tries = f.flag_tries;
        pr.withhold_first = f.withhold_first;
        // every flag starts at zero, whatever an earlier call left in the workspace
        if ((e = cudaMemsetAsync(pr.flags, 0, n_total * 4, p.stream)) != cudaSuccess) return e;
        void *args[] = {(void *)&tk, (void *)&tv, (void *)&tq, (void *)&tkw, (void *)&pr};
        e = cudaLaunchCooperativeKernel((const void *)kernel, dim3((unsigned)grid), dim3(kThreads), args,
                                        smem_bytes<true>(), p.stream);
        if (e == cudaSuccess) return cudaSuccess;
        cudaGetLastError();   // not launchable together here: two launches instead
    }
    const bool packed = p.cu != nullptr, pro = p.prologue != 0;
    if (split && !pro && !p.kw) {
        auto prep = packed ? chunk_wprep_kernel<true> : chunk_wprep_kernel<false>;
        int dev = 0, sms = 0;
        if ((e = cudaFuncSetAttribute(prep, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kWSmem)) != cudaSuccess ||
            (e = cudaGetDevice(&dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return e;
        if (n_total > 0x7fffffffu) return cudaErrorInvalidValue;
        // persistent: one CTA per SM, each with two producers of 8 consumer warps
        const unsigned n_ctas = (unsigned)((n_total + 1) / 2 < (size_t)sms ? (n_total + 1) / 2 : sms);
        prep<<<n_ctas, kThreads, kWSmem, p.stream>>>(tk, tq, pr);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    } else if (split) {
        auto prep = p.kw     ? chunk_prep_kernel<false, false, true>
                    : packed ? (pro ? chunk_prep_kernel<true, true> : chunk_prep_kernel<true, false>)
                             : (pro ? chunk_prep_kernel<false, true> : chunk_prep_kernel<false, false>);
        const uint32_t psmem = pk_smem(p.kw != nullptr);
        int dev = 0, sms = 0, per_sm = 0;
        if ((e = cudaFuncSetAttribute(prep, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)psmem)) != cudaSuccess ||
            (e = cudaFuncSetAttribute(prep, cudaFuncAttributePreferredSharedMemoryCarveout,
                                      (int)cudaSharedmemCarveoutMaxShared)) != cudaSuccess ||
            (e = cudaGetDevice(&dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
            (e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, prep, kPrepThreads, psmem)) != cudaSuccess)
            return e;
        if (n_total > 0x7fffffffu) return cudaErrorInvalidValue;
        // persistent: as many one-group CTAs as fit, each taking every grid-th chunk
        const size_t slots = (size_t)sms * (per_sm > 0 ? per_sm : 1);
        const unsigned n_ctas = (unsigned)(n_total < slots ? n_total : slots);
        prep<<<n_ctas, kPrepThreads, psmem, p.stream>>>(tk, tq, tkw, pr);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    auto kernel = p.out_dtype == DP_F32 ? tc_kernel_for<float>(split, packed, pro, p.kw != nullptr)
                                        : tc_kernel_for<__nv_bfloat16>(split, packed, pro, p.kw != nullptr);
    const uint32_t smem = split ? smem_bytes<true>() : smem_bytes<false>();
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kernel<<<p.B * p.H, kThreads, smem, p.stream>>>(tk, tv, tq, pr);
    return cudaGetLastError();
}

}  // namespace dp
