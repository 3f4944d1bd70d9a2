// Internal declarations shared by the host planner and the kernel launchers.
// Not part of the public ABI (include/gla.h is).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/gla.h"

namespace gla {

constexpr int kChunk = 64;        // primary chunk length C of the tensor-core path
constexpr int kSimtChunk = 16;    // chunk length of the CUDA-core path
constexpr int kDvTile = 128;      // dv columns per CTA on the tensor-core path
constexpr int kSimtDvTile = 64;   // dv columns per CTA on the CUDA-core path
constexpr int kMaxDk = 256;       // widest keys of the tensor-core path and of the 16-row CUDA-core form
constexpr int kStateCtasPerSm = 1;  // resident CTAs per SM of the state pass (gla_chunk_state)
constexpr int kMinStateChunks = 4;  // shortest piece the planner gives the state pass
// CUDA-core forward for dk > kMaxDk: 8-row chunks and 32 columns per CTA keep
// the fp32 state tile (dk x 32) and five [8 x dk] row buffers within the
// 227 KB of shared memory a CTA may hold, up to dk = kSimtMaxDk.
constexpr int kSimtChunkWide = 8;
constexpr int kSimtDvTileWide = 32;
constexpr int kSimtMaxDk = 768;
// Bilinear gate on the tensor-core path: the largest |in-chunk partial sum of
// log beta| for which one reference per chunk stays exact to rounding.
constexpr float kVGuard = 60.f;
// Per-head scalar gate on the tensor-core path: a chunk whose in-chunk log
// decay B_end = rows * log(lambda) stays above -kQGuard takes the query row
// factor lambda^(r+1) out of the inter and intra products (the chunk pass reads
// raw q and scales its output rows), so the prep writes no Q (.) Lambda for it.
// The prep and the chunk pass decide with this same test on the same float.
constexpr float kQGuard = 60.f;
__host__ __device__ __forceinline__ bool q_factored(float b_end) { return b_end >= -kQGuard; }
// Whether a pass takes that form at all: the per-head scalar gate with dk <= 128 (at
// dk = 256 the chunk pass's extra drain work spills registers).
inline bool q_factor_offload(const gla_fwd_params& p) { return p.gate == GLA_GATE_HEAD_SCALAR && p.dk <= 128; }

enum StageKind {
    STAGE_SIMT = 0,        // whole pass on CUDA cores
    STAGE_PREP = 1,        // gate prep + intra-chunk scores
    STAGE_SEG_STATE = 2,   // per-segment state from a zero start (sequence split)
    STAGE_SEG_SCAN = 3,    // serial recurrence over segments
    STAGE_CHUNK_FWD = 4,   // chunk-serial tensor-core pass: state, inter + intra output
    STAGE_COPY_STATE = 5,  // T == 0: ST <- S0 (or 0)
    STAGE_VALUE_PREP = 6,  // bilinear gate: V (.) D', the chunks' column decays, range flags
    STAGE_SIMT_FLAGGED = 7,  // bilinear gate: the CUDA-core pass for the heads flagged out of range
    STAGE_CHUNK_FWD_HI = 8,  // dk = 512: the chunk pass over keys 256-511, adding the first half's partial O
    STAGE_FUSED = 9,         // per-key gate, dk = 256: gate prep inside the chunk pass (one cluster per head)
    STAGE_SEG_WINDOW = 10,   // sliding-window split: each segment's start state from the window before it
};

struct Plan {
    int path = GLA_PATH_SIMT;
    int nchunks = 0;       // ceil(T / 64)
    int Tpad = 0;          // nchunks * 64
    int n_dvt = 0;         // number of dv tiles
    int nseg = 1;          // sequence segments per (b,h)
    int chunks_per_seg = 0;
    int window = 0;        // sliding-window split: chunks of the window (0: exact split)
    // exact split: the state pass covers the chunks before the last segment in st_nseg
    // pieces of st_cps chunks, sub of them per segment (finer than the segments, so that
    // it fills the SMs), and the workspace keeps segin_n start states per (b,h): one per
    // piece and the state after the last (the sliding window keeps one per segment)
    int sub = 1, st_nseg = 0, st_cps = 0, segin_n = 0;
    bool raw_qk = false;   // tensor path reads q,k directly (no gate)
    // the chunk pass forms the intra-chunk scores itself (dk <= 128, no gate or a per-head
    // gate's chunks with the query factor left to it); no gate then needs no prep at all
    bool sc = false;
    int sms = 0;           // multiprocessors of the device the plan was made for
    // workspace layout (byte offsets from the workspace base)
    size_t off_qt = 0, off_kt = 0, off_A = 0, off_gam = 0, off_segS = 0, off_segin = 0;
    size_t off_vh = 0, off_lbc = 0, off_flag = 0;   // bilinear gate only
    size_t off_opart = 0;  // dk = 512: the first key half's O, fp32 [BH][T][dv]
    size_t ws_bytes = 0;
    int nstages = 0;
    StageKind stages[8];
};

// Argument checks of the C ABI (gla_api.cu). validate_args: sizes, modes and
// which pointers are present. validate_pointers: no output overlaps an input
// (ST may equal S0 exactly) and, when `device`, the alignment the kernels need.
gla_status validate_args(const gla_fwd_params* p);
gla_status validate_pointers(const gla_fwd_params* p, bool device);
// Workspace bytes of the plan for *p from its shapes alone (the pointers are
// not looked at); the status of validate_args or of planning.
gla_status plan_workspace(const gla_fwd_params* p, size_t* bytes);

// Device status word (per device), written by kernels whose bounded waits run out.
int* device_status_ptr();   // nullptr on failure

// Launchers. Each returns cudaSuccess or the launch error.
// launch_simt: with `only` non-null, just the heads bh with only[bh] != 0.
cudaError_t launch_simt(const gla_fwd_params& p, int* status, cudaStream_t s, const int* only = nullptr);
cudaError_t launch_value_prep(const gla_fwd_params& p, const Plan& pl, void* ws, cudaStream_t s);
// allow_qfac = false: the per-head scalar gate's chunks always get Q (.) Lambda and plain
// scores (the backward reads them as such)
cudaError_t launch_prep(const gla_fwd_params& p, const Plan& pl, void* ws, int* status, cudaStream_t s,
                        bool allow_qfac = true);
// kh: 0, or for dk = 512 the key half (1: keys 0-255 with the intra term, O as an fp32
// partial; 2: keys 256-511, adding that partial)
cudaError_t launch_chunk_fwd(const gla_fwd_params& p, const Plan& pl, void* ws, int mode,
                             int* status, cudaStream_t s, int kh = 0);
// The fused per-key pass (gla_fused.cu): the shapes it takes, whether the device can run
// its clusters, and the launch.
bool fused_shape_ok(const gla_fwd_params& p);
bool fused_available(int dv);
cudaError_t launch_fused(const gla_fwd_params& p, int* status, cudaStream_t s);
// launch_seg_state: with S_out non-null and a one-segment plan, the segment's state goes
// there ([BH][dk][dv]) instead of the workspace.
cudaError_t launch_seg_state(const gla_fwd_params& p, const Plan& pl, void* ws, int* status, cudaStream_t s,
                             float* S_out = nullptr);
// The sliding-window split: segment 0's start state is S0 (or zero); segment s > 0's is the
// state the pl.window chunks before it leave from a zero start.
cudaError_t launch_seg_window(const gla_fwd_params& p, const Plan& pl, void* ws, int* status, cudaStream_t s);
cudaError_t launch_seg_scan(const gla_fwd_params& p, const Plan& pl, void* ws, int* status,
                            cudaStream_t s);

// The sequence exchange (gla_seqpar.cu): log Gamma of a segment (the per-key sum of the log
// gate; ws holds seg_logsum_ws_bytes(p) bytes, 8-byte aligned), the recurrence over P pairs,
// and one composition of two pairs.
size_t seg_logsum_ws_bytes(const gla_fwd_params& p);
cudaError_t launch_seg_logsum(const gla_fwd_params& p, float* log_Gamma, void* ws, cudaStream_t s);
cudaError_t launch_pair_scan(int P, const float* log_G, const float* S_star, const float* S0, float* S_in,
                             float* S_T, long long BH, int dk, int dv, int sms, cudaStream_t s);
cudaError_t launch_pair_combine(const float* log_G2, const float* S2, float* log_G1, float* S1, long long BH,
                                int dk, int dv, int sms, cudaStream_t s);

// One warp waiting, with the pipelined kernels' bounded mbarrier wait, on a barrier that
// nothing arrives on (unless `arrive`): a timeout recorded in the status word (gla_selftest.cu).
cudaError_t launch_wait_selftest(int* status, unsigned limit_us, bool arrive, cudaStream_t s);

// chunk_fwd modes
constexpr int kModeFull = 0;        // O and final state from S0 (single segment)
constexpr int kModeSegState = 1;    // per-segment state from zero, no O
constexpr int kModeSegOut = 2;      // O from per-segment start states, no final state
constexpr int kModeSweep = 3;       // no O: the state entering every chunk to Hst, the final state
constexpr int kModeSweepRev = 4;    // the same over the chunks from the last (dL/dS for the backward)

// The chunk pass as a state sweep for the backward (gla_chunk_fwd.cu): with X = S_in,
// for each chunk c in order (from the last when `reverse`): Hst[c] <- bf16(X), then
// X <- Diag(gam[c]) X + KT[c]^T V[c]; S_out <- X at the end. KT: [BH][kt_rows][dk] bf16
// (rows past T zero), V: [BH][T][dv] bf16, gam: [BH][nch][dk] or null (no gate), S_in,
// S_out: [BH][dk][dv] fp32 or null, Hst: [BH][nch][dv][dk] bf16. dk in {64, 128, 256},
// dv a multiple of 128.
struct StateSweep {
    const void* kt; long long kt_rows;
    const void* v;
    const float* gam;
    const float* S_in;
    float* S_out;
    void* Hst;
    bool reverse;
    int BH, T, dk, dv, nch;
    // sequence split (nseg > 1): segment s covers chunks [s cps, (s + 1) cps) and starts from
    // S_in + (bh nseg + s) dk dv; S_out is written by the last segment (the first, reverse)
    int nseg = 1, cps = 0;
};
cudaError_t launch_state_sweep(const StateSweep& w, int* status, cudaStream_t s);

// The sequence split for the backward's sweeps. launch_seg_state_job (gla_state.cu): each
// segment's state from a zero start, S*_s = sum over its chunks n of (KT_n (.) d_n)^T V_n, d_n
// the product of the segment's gates after chunk n (before it when `reverse`), to S_out
// [BH][nseg][dk][dv]. launch_seg_scan_job (gla_scan.cu): segin[s] = the state entering segment
// s from S_start (the recurrence over segments, from the last when `reverse`), S_end the
// state after all of them (either may be null).
struct SegStateJob {
    const void* kt; long long kt_rows;
    const void* v;
    const float* gam;
    float* S_out;
    bool reverse;
    int BH, T, dk, dv, nch, cps, nseg;
};
cudaError_t launch_seg_state_job(const SegStateJob& j, int* status, cudaStream_t s);
struct SegScanJob {
    const float* S_start;
    float* S_end;
    const float* gam;
    const float* segS;
    float* segin;
    bool reverse;
    int BH, dk, dv, nch, cps, nseg;
};
cudaError_t launch_seg_scan_job(const SegScanJob& j, cudaStream_t s);

// The chunk-parallel gradients of the backward (gla_bwd_chunk.cu): dq, dk, dv and the gate
// terms q (.) dq - k (.) dk per token, from the prep's Kt, Qt ([BH][kt_rows][dk] bf16), A and
// gamma, and the two sweeps' H and D ([BH][nch][dv][dk] bf16). dk in {128, 256}, dv a
// multiple of 128, T > 0. gam null without a gate; bnd ([BH][dk]) may be null. With R
// ([BH][T][dk]) and ctot ([BH][nch][dk]): R gets each gate term summed over the later rows of
// its chunk, ctot each chunk's total.
struct BwdGrads {
    const void* q; const void* k; const void* v; const void* dO;
    const float* log_g;
    const void* qt; const void* kt; long long kt_rows;
    const void* A; const float* gam;
    const void* Hst; const void* Dst;
    const float* bnd;
    float* gq; float* gk; float* gv; float* R; float* ctot;
    int BH, H, T, dk, dv, gate, sms;
};
cudaError_t launch_bwd_grads(const BwdGrads& g, int* status, cudaStream_t s);
// out [BH][T][dk] += crev [BH][nch][dk] of the chunk after each row's (none for the last)
cudaError_t launch_bwd_gate_fixup(float* out, const float* crev, long long BH, int T, int dk, int sms, cudaStream_t s);
// rowsum(dST (.) ST) over each of `rows` rows of dv values
cudaError_t launch_bwd_boundary(const float* dST, const float* ST, float* bnd, long long rows, int dv, int sms,
                                cudaStream_t s);

}  // namespace gla
