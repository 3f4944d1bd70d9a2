// Host side of the C ABI: argument validation, planning, workspace layout and
// launch order. No arithmetic of the method happens here; every step of the
// pass runs in the kernels.
#include <cstdint>
#include <cstring>
#include <mutex>

#include "gla_internal.h"

namespace gla {

namespace {

constexpr int kVersion = 100;  // 0.1.0

__device__ int g_status[1];   // device status word: 0 ok, else the kernel's timeout code

struct DevCache {
    bool init = false;
    int major = 0, minor = 0, sms = 0;
    int* status = nullptr;
};
std::mutex g_mu;
DevCache g_dev[64];

DevCache* dev_cache()
{
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    DevCache& c = g_dev[d];
    if (!c.init) {
        if (cudaDeviceGetAttribute(&c.major, cudaDevAttrComputeCapabilityMajor, d) != cudaSuccess) return nullptr;
        if (cudaDeviceGetAttribute(&c.minor, cudaDevAttrComputeCapabilityMinor, d) != cudaSuccess) return nullptr;
        if (cudaDeviceGetAttribute(&c.sms, cudaDevAttrMultiProcessorCount, d) != cudaSuccess) return nullptr;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return nullptr;
        c.status = static_cast<int*>(p);
        c.init = true;
    }
    return &c;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Range { uintptr_t lo, hi; };
Range rng(const void* p, size_t bytes) {
    uintptr_t a = reinterpret_cast<uintptr_t>(p);
    return Range{a, a + bytes};
}
bool overlap(Range a, Range b) {
    if (a.lo == a.hi || b.lo == b.hi || a.lo == 0 || b.lo == 0) return false;
    return a.lo < b.hi && b.lo < a.hi;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace

// Host-only checks of sizes, modes and which pointers are present.
gla_status validate_args(const gla_fwd_params* p)
{
    if (!p) return GLA_ERR_INVALID_ARG;
    if (p->B <= 0 || p->H <= 0 || p->T < 0 || p->dk <= 0 || p->dv <= 0) return GLA_ERR_INVALID_ARG;
    if (p->dtype != GLA_BF16 && p->dtype != GLA_FP32) return GLA_ERR_INVALID_ARG;
    if (p->gate != GLA_GATE_NONE && p->gate != GLA_GATE_HEAD_SCALAR && p->gate != GLA_GATE_PER_KEY &&
        p->gate != GLA_GATE_TOKEN_SCALAR && p->gate != GLA_GATE_BILINEAR)
        return GLA_ERR_INVALID_ARG;
    if ((p->gate == GLA_GATE_BILINEAR) != (p->log_b != nullptr) && !(p->gate == GLA_GATE_BILINEAR && p->T == 0))
        return GLA_ERR_INVALID_ARG;
    if (p->path != GLA_PATH_AUTO && p->path != GLA_PATH_TENSOR && p->path != GLA_PATH_SIMT &&
        p->path != GLA_PATH_STAGED && p->path != GLA_PATH_FUSED)
        return GLA_ERR_INVALID_ARG;
    if (p->force_segments < 0 || p->window_chunks < 0) return GLA_ERR_INVALID_ARG;
    if (p->dk % 16 != 0 || p->dv % 16 != 0) return GLA_ERR_INVALID_ARG;
    if ((long long)p->B * p->H > (1LL << 30)) return GLA_ERR_INVALID_ARG;
    if (p->gate == GLA_GATE_NONE && p->log_g) return GLA_ERR_INVALID_ARG;
    if (p->gate == GLA_GATE_HEAD_SCALAR && !p->log_g) return GLA_ERR_INVALID_ARG;
    if ((p->gate == GLA_GATE_PER_KEY || p->gate == GLA_GATE_TOKEN_SCALAR || p->gate == GLA_GATE_BILINEAR) &&
        !p->log_g && p->T > 0)
        return GLA_ERR_INVALID_ARG;
    if (p->T > 0 && (!p->q || !p->k || !p->v || !p->O)) return GLA_ERR_INVALID_ARG;
    if (p->chunk != 0 && p->chunk != kChunk) return GLA_ERR_UNSUPPORTED;
    if (p->dk > kSimtMaxDk) return GLA_ERR_UNSUPPORTED;
    return GLA_OK;
}

// Checks of the pointer values: outputs overlap no input (ST may equal S0
// exactly), and, for device pointers, the alignment the kernels' TMA and
// vector accesses need.
gla_status validate_pointers(const gla_fwd_params* p, bool device)
{
    const size_t e = p->dtype == GLA_BF16 ? 2 : 4;
    const size_t BH = (size_t)p->B * p->H;
    const size_t nq = BH * p->T * p->dk * e, nv = BH * p->T * p->dv * e;
    const size_t ng = (p->gate == GLA_GATE_PER_KEY || p->gate == GLA_GATE_BILINEAR) ? BH * p->T * p->dk * 4
                    : p->gate == GLA_GATE_TOKEN_SCALAR ? BH * p->T * 4
                    : p->gate == GLA_GATE_HEAD_SCALAR ? (size_t)p->H * 4 : 0;
    const size_t ns = BH * p->dk * p->dv * 4;
    if (device) {
        // TMA and vector loads need 16-byte aligned bases
        for (const void* ptr : {p->q, p->k, p->v, (const void*)p->O, (const void*)p->S0, (const void*)p->ST})
            if (ptr && !aligned(ptr, 16)) return GLA_ERR_INVALID_ARG;
        if (p->log_g && !aligned(p->log_g, p->gate == GLA_GATE_PER_KEY ? 16 : 4)) return GLA_ERR_INVALID_ARG;
        if (p->log_b && !aligned(p->log_b, 4)) return GLA_ERR_INVALID_ARG;
        if (p->workspace && !aligned(p->workspace, 256)) return GLA_ERR_INVALID_ARG;
    }
    // outputs must not overlap inputs; ST may equal S0 exactly (in-place state carry)
    Range rO = rng(p->O, nv), rST = rng(p->ST, p->ST ? ns : 0);
    Range ins[] = {rng(p->q, nq), rng(p->k, nq), rng(p->v, nv), rng(p->log_g, ng), rng(p->S0, p->S0 ? ns : 0)};
    for (Range r : ins) if (overlap(rO, r)) return GLA_ERR_INVALID_ARG;
    const Range rb = rng(p->log_b, p->log_b ? BH * p->T * p->dv * 4 : 0);
    if (overlap(rO, rb) || overlap(rST, rb)) return GLA_ERR_INVALID_ARG;
    if (overlap(rO, rST)) return GLA_ERR_INVALID_ARG;
    for (int i = 0; i < 4; ++i) if (overlap(rST, ins[i])) return GLA_ERR_INVALID_ARG;
    if (p->ST && p->S0 && overlap(rST, ins[4]) && (const void*)p->ST != (const void*)p->S0)
        return GLA_ERR_INVALID_ARG;
    return GLA_OK;
}

namespace {

gla_status validate(const gla_fwd_params* p)
{
    gla_status st = validate_args(p);
    return st != GLA_OK ? st : validate_pointers(p, true);
}

bool tensor_shape_ok(const gla_fwd_params* p)
{
    const long long BH = (long long)p->B * p->H;
    const long long Tpad = ((long long)p->T + kChunk - 1) / kChunk * kChunk;
    // dk = 512 runs as two chunk passes over key halves (not with the bilinear gate)
    const bool dk_ok = p->dk == 64 || p->dk == 128 || p->dk == 256 ||
                       (p->dk == 512 && p->gate != GLA_GATE_BILINEAR);
    return p->dtype == GLA_BF16 && dk_ok && p->dv % kDvTile == 0 && BH <= 65535 && BH * Tpad < (1LL << 31);
}

// Number of sequence segments per (b,h). A single chunk-serial pass per
// (b,h, dv tile) leaves SMs idle when B*H*tiles is small; splitting the
// sequence into n segments costs one extra state-only pass and a short
// serial recurrence over segments, so it pays only when the pass is long
// and the grid is well under one wave.
int choose_segments(const gla_fwd_params* p, int units, int nchunks, int sms)
{
    if (p->force_segments > 0) return p->force_segments < nchunks ? p->force_segments : (nchunks > 0 ? nchunks : 1);
    if (units * 2 > sms || nchunks < 16) return 1;
    int n = sms / units;
    if (n > nchunks / 8) n = nchunks / 8;
    return n < 1 ? 1 : n;
}

// Callers check the pointers (validate or validate_pointers) themselves.
gla_status make_plan(const gla_fwd_params* p, Plan& pl, int sms)
{
    gla_status st = validate_args(p);
    if (st != GLA_OK) return st;
    pl = Plan{};
    if (p->T == 0) {
        pl.path = GLA_PATH_SIMT;
        pl.nstages = 1;
        pl.stages[0] = STAGE_COPY_STATE;
        return GLA_OK;
    }
    if (p->path == GLA_PATH_FUSED) {
        // the fused per-key pass: one kernel, no workspace, never a sequence split
        if (!fused_shape_ok(*p) || (sms > 0 && !fused_available(p->dv))) return GLA_ERR_UNSUPPORTED;
        pl.path = GLA_PATH_TENSOR;
        pl.nchunks = (p->T + kChunk - 1) / kChunk;
        pl.Tpad = pl.nchunks * kChunk;
        pl.n_dvt = p->dv / kDvTile;
        pl.sms = sms;
        pl.nstages = 1;
        pl.stages[0] = STAGE_FUSED;
        pl.ws_bytes = 0;
        return GLA_OK;
    }
    bool want_tensor = false;
    if (p->path == GLA_PATH_TENSOR || p->path == GLA_PATH_STAGED) {
        if (!tensor_shape_ok(p)) return GLA_ERR_UNSUPPORTED;
        want_tensor = true;
    } else if (p->path == GLA_PATH_AUTO) {
        want_tensor = tensor_shape_ok(p);
    }
    if (!want_tensor) {
        pl.path = GLA_PATH_SIMT;
        pl.nstages = 1;
        pl.stages[0] = STAGE_SIMT;
        return GLA_OK;
    }
    pl.path = GLA_PATH_TENSOR;
    pl.nchunks = (p->T + kChunk - 1) / kChunk;
    pl.Tpad = pl.nchunks * kChunk;
    pl.n_dvt = p->dv / kDvTile;
    pl.raw_qk = (p->gate == GLA_GATE_NONE);
    // the intra-chunk scores formed in the chunk pass: dk <= 128 (its tensor memory has room
    // for the score accumulator), no gate, or a per-head gate with the query factor left to it
    pl.sc = p->dk <= 128 && (p->gate == GLA_GATE_NONE || q_factor_offload(*p));
    pl.sms = sms;
    const int units = p->B * p->H * pl.n_dvt;
    const bool bil = p->gate == GLA_GATE_BILINEAR;
    // the sequence split carries only a per-key decay between segments: none with the bilinear gate
    const bool halves = p->dk == 512;   // two chunk passes over key halves; no sequence split
    pl.nseg = (bil || halves) ? 1 : choose_segments(p, units, pl.nchunks, sms > 0 ? sms : 148);
    pl.chunks_per_seg = (pl.nchunks + pl.nseg - 1) / pl.nseg;
    pl.nseg = (pl.nchunks + pl.chunks_per_seg - 1) / pl.chunks_per_seg;
    pl.window = pl.nseg > 1 ? p->window_chunks : 0;
    if (pl.nseg > 1 && pl.window == 0) {
        // The last segment's own chunk pass ends at S_T, so the state pass only covers the
        // chunks before it. It cuts them into the most pieces that still fit in one wave,
        // each a whole fraction of a segment and at least kMinStateChunks long.
        const int cps = pl.chunks_per_seg, slots = (sms > 0 ? sms : 148) * kStateCtasPerSm;
        const long long fit = slots / ((long long)(pl.nseg - 1) * units);   // pieces per segment in one wave
        pl.sub = 1;
        for (int f = (int)(fit < cps / kMinStateChunks ? fit : cps / kMinStateChunks); f > 1; --f)
            if (cps % f == 0) {
                pl.sub = f;
                break;
            }
        pl.st_nseg = (pl.nseg - 1) * pl.sub;
        pl.st_cps = cps / pl.sub;
        pl.segin_n = pl.st_nseg + 1;
    } else if (pl.nseg > 1) {
        pl.segin_n = pl.nseg;
    }

    const size_t BH = (size_t)p->B * p->H;
    size_t off = 0;
    if (!pl.raw_qk) {
        pl.off_qt = off; off = align_up(off + BH * pl.Tpad * p->dk * 2, 256);
        pl.off_kt = off; off = align_up(off + BH * pl.Tpad * p->dk * 2, 256);
    }
    const bool prep = !(pl.sc && p->gate == GLA_GATE_NONE);   // no gate, scores in the pass: nothing to prepare
    if (prep) {
        pl.off_A = off;   off = align_up(off + BH * pl.nchunks * kChunk * kChunk * 2, 256);
    }
    if (p->gate != GLA_GATE_NONE) {
        pl.off_gam = off; off = align_up(off + BH * pl.nchunks * p->dk * 4, 256);
    }
    if (pl.nseg > 1) {
        pl.off_segS = off;  off = align_up(off + BH * pl.st_nseg * p->dk * p->dv * 4, 256);
        pl.off_segin = off; off = align_up(off + BH * pl.segin_n * p->dk * p->dv * 4, 256);
    }
    if (halves) {
        pl.off_opart = off; off = align_up(off + BH * p->T * p->dv * 4, 256);
    }
    if (bil) {
        pl.off_vh = off;   off = align_up(off + BH * p->T * p->dv * 2, 256);
        pl.off_lbc = off;  off = align_up(off + BH * pl.nchunks * p->dv * 4, 256);
        pl.off_flag = off; off = align_up(off + BH * 4, 256);
    }
    pl.ws_bytes = off;
    int n = 0;
    if (prep) pl.stages[n++] = STAGE_PREP;
    if (bil) pl.stages[n++] = STAGE_VALUE_PREP;
    if (pl.nseg > 1 && pl.window > 0) {
        pl.stages[n++] = STAGE_SEG_WINDOW;
    } else if (pl.nseg > 1) {
        pl.stages[n++] = STAGE_SEG_STATE;
        pl.stages[n++] = STAGE_SEG_SCAN;
    }
    pl.stages[n++] = STAGE_CHUNK_FWD;
    if (halves) pl.stages[n++] = STAGE_CHUNK_FWD_HI;
    if (bil) pl.stages[n++] = STAGE_SIMT_FLAGGED;
    pl.nstages = n;
    return GLA_OK;
}

const char* stage_name(StageKind k)
{
    switch (k) {
    case STAGE_SIMT: return "gla_fwd_simt";
    case STAGE_PREP: return "gla_chunk_prep";
    case STAGE_SEG_STATE: return "gla_chunk_state";
    case STAGE_SEG_SCAN: return "gla_state_scan";
    case STAGE_CHUNK_FWD: return "gla_chunk_fwd";
    case STAGE_COPY_STATE: return "gla_copy_state";
    case STAGE_VALUE_PREP: return "gla_value_prep";
    case STAGE_SIMT_FLAGGED: return "gla_fwd_simt_flagged";
    case STAGE_CHUNK_FWD_HI: return "gla_chunk_fwd_keys_hi";
    case STAGE_FUSED: return "gla_chunk_fused";
    case STAGE_SEG_WINDOW: return "gla_chunk_state_window";
    }
    return "?";
}

int device_sms()
{
    DevCache* c = dev_cache();
    return c ? c->sms : 0;
}

gla_status run_stage(const gla_fwd_params* p, const Plan& pl, int i, cudaStream_t s)
{
    DevCache* c = dev_cache();
    if (!c) return GLA_ERR_CUDA;
    if (c->major != 10 || c->minor != 3) return GLA_ERR_UNSUPPORTED;  // built for sm_103a only
    const StageKind k = pl.stages[i];
    if (pl.ws_bytes > 0 && k != STAGE_SIMT && k != STAGE_COPY_STATE) {
        if (!p->workspace || p->workspace_bytes < pl.ws_bytes) return GLA_ERR_WORKSPACE;
    }
    cudaError_t e = cudaSuccess;
    switch (k) {
    case STAGE_COPY_STATE:
        if (p->ST && p->ST != p->S0) {
            const size_t ns = (size_t)p->B * p->H * p->dk * p->dv * 4;
            e = p->S0 ? cudaMemcpyAsync(p->ST, p->S0, ns, cudaMemcpyDeviceToDevice, s)
                      : cudaMemsetAsync(p->ST, 0, ns, s);
        }
        break;
    case STAGE_SIMT: e = launch_simt(*p, c->status, s); break;
    case STAGE_PREP: e = launch_prep(*p, pl, p->workspace, c->status, s); break;
    case STAGE_SEG_STATE: e = launch_seg_state(*p, pl, p->workspace, c->status, s); break;
    case STAGE_SEG_SCAN: e = launch_seg_scan(*p, pl, p->workspace, c->status, s); break;
    case STAGE_SEG_WINDOW: e = launch_seg_window(*p, pl, p->workspace, c->status, s); break;
    case STAGE_CHUNK_FWD:
        e = launch_chunk_fwd(*p, pl, p->workspace, pl.nseg > 1 ? kModeSegOut : kModeFull, c->status, s,
                             p->dk == 512 ? 1 : 0);
        break;
    case STAGE_CHUNK_FWD_HI: e = launch_chunk_fwd(*p, pl, p->workspace, kModeFull, c->status, s, 2); break;
    case STAGE_FUSED: e = launch_fused(*p, c->status, s); break;
    case STAGE_VALUE_PREP: e = launch_value_prep(*p, pl, p->workspace, s); break;
    case STAGE_SIMT_FLAGGED:
        e = launch_simt(*p, c->status, s, reinterpret_cast<const int*>(static_cast<uint8_t*>(p->workspace) + pl.off_flag));
        break;
    }
    return e == cudaSuccess ? GLA_OK : GLA_ERR_CUDA;
}

// The sequence-exchange pair of one segment: the call's parameters as the segment's
// forward pass sees them, and where each part of the work goes.
struct PairPlan {
    gla_fwd_params pp;     // *p with S0 = none, ST = S_star, q = k when absent
    bool tensor = false;   // gate prep + state-only pass (else the CUDA-core pass, O discarded)
    Plan pl;               // tensor route: the prep's workspace layout, one segment
    size_t off_o = 0;      // CUDA-core route: the discarded O
    size_t off_sum = 0;    // the log gate's partial sums
    size_t ws_bytes = 0;
};

// shapes_only: check sizes, modes and which inputs are present, not the pointer values
// (the workspace query, which gets no output pointers).
gla_status plan_pair(const gla_fwd_params* p, const float* log_Gamma, const float* S_star, int sms, PairPlan& pp,
                     bool shapes_only = false)
{
    if (!p || (!shapes_only && (!log_Gamma || !S_star))) return GLA_ERR_INVALID_ARG;
    if (p->gate == GLA_GATE_BILINEAR) return GLA_ERR_UNSUPPORTED;   // its decay is a dk x dv matrix
    gla_fwd_params& q = pp.pp;
    q = *p;
    q.S0 = nullptr;
    q.ST = const_cast<float*>(S_star);
    q.force_segments = 1;
    if (!q.q) q.q = q.k;   // read by the gate prep; the pair does not depend on it
    // presence checks want an O; the pair never writes the caller's
    q.O = const_cast<void*>(q.v);
    gla_status st = validate_args(&q);
    if (st != GLA_OK) return st;
    q.O = nullptr;
    const size_t BH = (size_t)q.B * q.H;
    const size_t e = q.dtype == GLA_BF16 ? 2 : 4;
    if (!shapes_only) {
        st = validate_pointers(&q, true);
        if (st != GLA_OK) return st;
        if (!aligned(log_Gamma, 4)) return GLA_ERR_INVALID_ARG;
        const Range rG = rng(log_Gamma, BH * q.dk * 4);
        const size_t ng = q.gate == GLA_GATE_PER_KEY ? BH * q.T * q.dk * 4
                        : q.gate == GLA_GATE_TOKEN_SCALAR ? BH * q.T * 4
                        : q.gate == GLA_GATE_HEAD_SCALAR ? (size_t)q.H * 4 : 0;
        const Range ins[] = {rng(p->q, BH * q.T * q.dk * e), rng(q.k, BH * q.T * q.dk * e),
                             rng(q.v, BH * q.T * q.dv * e), rng(q.log_g, ng), rng(S_star, BH * q.dk * q.dv * 4)};
        for (const Range& r : ins) if (overlap(rG, r)) return GLA_ERR_INVALID_ARG;
    }
    size_t off = 0;
    pp.tensor = q.T > 0 && p->path != GLA_PATH_SIMT && tensor_shape_ok(&q) && q.dk <= kMaxDk;
    if (q.T > 0) {
        if (pp.tensor) {
            gla_fwd_params t = q;
            t.O = const_cast<void*>(q.v);   // placeholder for the presence check; prep and state ignore O
            t.path = GLA_PATH_STAGED;
            st = make_plan(&t, pp.pl, sms);
            if (st != GLA_OK) return st;
            if (pp.pl.nseg != 1) return GLA_ERR_UNSUPPORTED;
            off = pp.pl.ws_bytes;
        } else {
            pp.off_o = off;
            off = align_up(off + BH * q.T * q.dv * e, 256);
        }
    }
    pp.off_sum = off;
    off = align_up(off + seg_logsum_ws_bytes(q), 256);
    pp.ws_bytes = off;
    return GLA_OK;
}

}  // namespace

gla_status plan_workspace(const gla_fwd_params* p, size_t* bytes)
{
    Plan pl;
    gla_status st = make_plan(p, pl, device_sms());
    *bytes = st == GLA_OK ? pl.ws_bytes : 0;
    return st;
}

int* device_status_ptr()
{
    DevCache* c = dev_cache();
    return c ? c->status : nullptr;
}

}  // namespace gla

using namespace gla;

extern "C" {

size_t gla_fwd_workspace_size(const gla_fwd_params* p)
{
    Plan pl;
    if (validate(p) != GLA_OK) return 0;
    if (make_plan(p, pl, device_sms()) != GLA_OK) return 0;
    return pl.ws_bytes;
}

int gla_fwd_num_stages(const gla_fwd_params* p)
{
    Plan pl;
    if (validate(p) != GLA_OK) return -1;
    if (make_plan(p, pl, device_sms()) != GLA_OK) return -1;
    return pl.nstages;
}

const char* gla_fwd_stage_name(const gla_fwd_params* p, int stage)
{
    Plan pl;
    if (validate(p) != GLA_OK) return "invalid";
    if (make_plan(p, pl, device_sms()) != GLA_OK || stage < 0 || stage >= pl.nstages) return "invalid";
    return stage_name(pl.stages[stage]);
}

gla_status gla_fwd_stage(const gla_fwd_params* p, int stage, cudaStream_t stream)
{
    gla_status st = validate(p);
    if (st != GLA_OK) return st;
    Plan pl;
    st = make_plan(p, pl, device_sms());
    if (st != GLA_OK) return st;
    if (stage < 0 || stage >= pl.nstages) return GLA_ERR_INVALID_ARG;
    return run_stage(p, pl, stage, stream);
}

gla_status gla_fwd_ex(const gla_fwd_params* p, cudaStream_t stream)
{
    gla_status st = validate(p);
    if (st != GLA_OK) return st;
    Plan pl;
    st = make_plan(p, pl, device_sms());
    if (st != GLA_OK) return st;
    for (int i = 0; i < pl.nstages; ++i) {
        st = run_stage(p, pl, i, stream);
        if (st != GLA_OK) return st;
    }
    return GLA_OK;
}

gla_status gla_fwd(const void* q, const void* k, const void* v, const float* log_g,
                   const float* S0, void* O, float* ST,
                   int B, int H, int T, int dk, int dv, int chunk, cudaStream_t stream)
{
    gla_fwd_params p;
    std::memset(&p, 0, sizeof(p));
    p.q = q; p.k = k; p.v = v; p.log_g = log_g; p.S0 = S0; p.O = O; p.ST = ST;
    p.B = B; p.H = H; p.T = T; p.dk = dk; p.dv = dv; p.chunk = chunk;
    p.dtype = GLA_BF16;
    p.gate = log_g ? GLA_GATE_PER_KEY : GLA_GATE_NONE;
    p.path = GLA_PATH_AUTO;
    gla_status st = validate(&p);
    if (st != GLA_OK) return st;
    Plan pl;
    st = make_plan(&p, pl, device_sms());
    if (st != GLA_OK) return st;
    void* ws = nullptr;
    if (pl.ws_bytes > 0) {
        if (cudaMallocAsync(&ws, pl.ws_bytes, stream) != cudaSuccess) return GLA_ERR_WORKSPACE;
        p.workspace = ws;
        p.workspace_bytes = pl.ws_bytes;
    }
    for (int i = 0; i < pl.nstages && st == GLA_OK; ++i) st = run_stage(&p, pl, i, stream);
    if (ws) {
        if (cudaFreeAsync(ws, stream) != cudaSuccess && st == GLA_OK) st = GLA_ERR_CUDA;
    }
    return st;
}

size_t gla_segment_pair_workspace_size(const gla_fwd_params* p)
{
    PairPlan pp;
    if (plan_pair(p, nullptr, nullptr, device_sms(), pp, true) != GLA_OK) return 0;
    return pp.ws_bytes;
}

gla_status gla_segment_pair(const gla_fwd_params* p, float* log_Gamma, float* S_star, cudaStream_t stream)
{
    PairPlan pp;
    gla_status st = plan_pair(p, log_Gamma, S_star, device_sms(), pp);
    if (st != GLA_OK) return st;
    DevCache* c = dev_cache();
    if (!c) return GLA_ERR_CUDA;
    if (c->major != 10 || c->minor != 3) return GLA_ERR_UNSUPPORTED;
    gla_fwd_params& q = pp.pp;
    if (pp.ws_bytes > 0 && (!p->workspace || p->workspace_bytes < pp.ws_bytes)) return GLA_ERR_WORKSPACE;
    uint8_t* ws = static_cast<uint8_t*>(p->workspace);
    const size_t ns = (size_t)q.B * q.H * q.dk * q.dv * 4;
    cudaError_t e = cudaSuccess;
    if (q.T == 0) {
        e = cudaMemsetAsync(S_star, 0, ns, stream);
    } else if (pp.tensor) {
        // (no gate with the scores formed in the chunk pass: nothing to prepare, the state
        // pass reads k itself)
        if (pp.pl.nstages > 0 && pp.pl.stages[0] == STAGE_PREP) e = launch_prep(q, pp.pl, ws, c->status, stream);
        if (e == cudaSuccess) e = launch_seg_state(q, pp.pl, ws, c->status, stream, S_star);
    } else {
        q.O = ws + pp.off_o;
        e = launch_simt(q, c->status, stream);
    }
    if (e == cudaSuccess) e = launch_seg_logsum(q, log_Gamma, ws ? ws + pp.off_sum : nullptr, stream);
    return e == cudaSuccess ? GLA_OK : GLA_ERR_CUDA;
}

gla_status gla_pair_scan(int P, const float* log_Gamma, const float* S_star, const float* S0, float* S_in,
                         float* S_T, int B, int H, int dk, int dv, cudaStream_t stream)
{
    if (P < 0 || B <= 0 || H <= 0 || dk <= 0 || dv <= 0) return GLA_ERR_INVALID_ARG;
    if (P > 0 && (!log_Gamma || !S_star)) return GLA_ERR_INVALID_ARG;
    if (!S_in && !S_T) return GLA_ERR_INVALID_ARG;
    const size_t BH = (size_t)B * H, ns = BH * dk * dv * 4;
    for (const void* ptr : {(const void*)log_Gamma, (const void*)S_star, (const void*)S0, (const void*)S_in,
                            (const void*)S_T})
        if (ptr && !aligned(ptr, 4)) return GLA_ERR_INVALID_ARG;
    const Range rG = rng(log_Gamma, P * BH * dk * 4), rS = rng(S_star, P * ns), r0 = rng(S0, S0 ? ns : 0);
    const Range rI = rng(S_in, S_in ? P * ns : 0), rT = rng(S_T, S_T ? ns : 0);
    // S_in may be S_star exactly and S_T may be S0 exactly (each element is read before it is written)
    if (overlap(rI, rG) || overlap(rI, r0) || overlap(rI, rT)) return GLA_ERR_INVALID_ARG;
    if (overlap(rI, rS) && (const void*)S_in != (const void*)S_star) return GLA_ERR_INVALID_ARG;
    if (overlap(rT, rG) || overlap(rT, rS)) return GLA_ERR_INVALID_ARG;
    if (overlap(rT, r0) && (const void*)S_T != (const void*)S0) return GLA_ERR_INVALID_ARG;
    if (!dev_cache()) return GLA_ERR_CUDA;
    return launch_pair_scan(P, log_Gamma, S_star, S0, S_in, S_T, (long long)BH, dk, dv, device_sms(), stream) ==
                   cudaSuccess ? GLA_OK : GLA_ERR_CUDA;
}

gla_status gla_pair_combine(const float* log_Gamma2, const float* S2, float* log_Gamma1, float* S1,
                            int B, int H, int dk, int dv, cudaStream_t stream)
{
    if (!log_Gamma2 || !S2 || !log_Gamma1 || !S1 || B <= 0 || H <= 0 || dk <= 0 || dv <= 0)
        return GLA_ERR_INVALID_ARG;
    for (const void* ptr : {(const void*)log_Gamma2, (const void*)S2, (const void*)log_Gamma1, (const void*)S1})
        if (!aligned(ptr, 4)) return GLA_ERR_INVALID_ARG;
    const size_t BH = (size_t)B * H, ns = BH * dk * dv * 4, ng = BH * dk * 4;
    const Range a[] = {rng(log_Gamma2, ng), rng(S2, ns)}, b[] = {rng(log_Gamma1, ng), rng(S1, ns)};
    for (const Range& x : a)
        for (const Range& y : b) if (overlap(x, y)) return GLA_ERR_INVALID_ARG;
    if (overlap(b[0], b[1])) return GLA_ERR_INVALID_ARG;
    if (!dev_cache()) return GLA_ERR_CUDA;
    return launch_pair_combine(log_Gamma2, S2, log_Gamma1, S1, (long long)BH, dk, dv, device_sms(), stream) ==
                   cudaSuccess ? GLA_OK : GLA_ERR_CUDA;
}

gla_status gla_selftest_bounded_wait(unsigned limit_us, int arrive, cudaStream_t stream)
{
    if (limit_us == 0 || limit_us > 1000000u) return GLA_ERR_INVALID_ARG;
    DevCache* c = dev_cache();
    if (!c) return GLA_ERR_CUDA;
    if (c->major != 10 || c->minor != 3) return GLA_ERR_UNSUPPORTED;
    return launch_wait_selftest(c->status, limit_us, arrive != 0, stream) == cudaSuccess ? GLA_OK : GLA_ERR_CUDA;
}

gla_status gla_device_status(cudaStream_t stream)
{
    if (cudaStreamSynchronize(stream) != cudaSuccess) return GLA_ERR_CUDA;
    int* d = device_status_ptr();
    if (!d) return GLA_ERR_CUDA;
    int h = 0;
    if (cudaMemcpy(&h, d, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return GLA_ERR_CUDA;
    if (h != 0) {
        int z = 0;
        if (cudaMemcpy(d, &z, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return GLA_ERR_CUDA;
        return GLA_ERR_TIMEOUT;
    }
    return GLA_OK;
}

const char* gla_status_string(gla_status s)
{
    switch (s) {
    case GLA_OK: return "GLA_OK";
    case GLA_ERR_INVALID_ARG: return "GLA_ERR_INVALID_ARG: invalid argument";
    case GLA_ERR_UNSUPPORTED: return "GLA_ERR_UNSUPPORTED: request not supported by this build or device";
    case GLA_ERR_CUDA: return "GLA_ERR_CUDA: a CUDA call or kernel launch failed";
    case GLA_ERR_WORKSPACE: return "GLA_ERR_WORKSPACE: workspace missing, too small or not allocatable";
    case GLA_ERR_TIMEOUT: return "GLA_ERR_TIMEOUT: a kernel's bounded wait ran out";
    }
    return "unknown gla_status";
}

int gla_version(void) { return kVersion; }

}  // extern "C"
