// gla_state_scan: the short serial recurrence over sequence segments that
// lets small B*H fill the GPU. Each segment s was first run from a zero state
// (gla_chunk_state), giving S*_s. Because the recurrence is
// linear in S and the gate only scales rows, the true state entering segment
// s+1 is
//     S_in(s+1) = Diag(Gamma_s) S_in(s) + S*_s,   Gamma_s = prod over the
//                 segment's chunks of gamma (per key),
// the state correction of the FlashQLA talk ("core technical principles":
// a wrongly started segment is fixed by one matrix per rank), which for a
// diagonal gate collapses from a dk x dk matrix to the vector Gamma_s. With
// S_in(0) = S0 this also yields S_in(nseg), the state after the last one.
//
// In the forward pass the "segments" here are the state pass's pieces: they
// cover the chunks before the chunk pass's last segment, sub pieces per
// segment, and the chunk pass's segment j starts from S_in(j sub); the state
// after the last piece is where its last segment starts (that segment's own
// pass then ends at S_T). The backward runs the same recurrence over its
// sweeps' segments, forward or from the last one.
//
// One CTA covers 256 consecutive state elements of one (b,h) (they share a
// key row k when dv >= 256, else two rows); one thread per element. The
// per-segment decays of the CTA's rows are formed first (one warp per
// (row, segment), a product over that segment's chunks); then each thread
// runs the recurrence with the loads of the next segments already in flight.
#include "gla_internal.h"

namespace gla {
namespace {

constexpr int NT = 256;
constexpr int AHEAD = 4;   // segment loads kept in flight per thread

struct ScanArgs {
    const float* S0;     // [BH][dk][dv] or null
    float* ST;           // [BH][dk][dv] or null
    const float* gam;    // [BH][nchunks][dk] or null (no gate)
    const float* segS;   // [BH][nseg][dk][dv]
    float* segin;        // segment s of (b,h) at segin + bh in_bh + s dk dv
    long long in_bh;
    long long st_bh;     // ST of (b,h) at ST + bh st_bh
    int dk, dv, nchunks, nseg, cps;
    int rev;             // from the last segment to the first (the backward's dL/dS)
};

__global__ void __launch_bounds__(NT) gla_state_scan_kernel(ScanArgs a)
{
    // the chunk pass may start its set-up now; it waits for this grid's writes before it reads them
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    extern __shared__ float Gs[];   // [rows][nseg]
    const int bh = blockIdx.y;
    const size_t st = (size_t)a.dk * a.dv;
    const size_t e0 = (size_t)blockIdx.x * NT;           // first element of this CTA
    const int k0 = (int)(e0 / a.dv);
    const int rows = (int)((e0 + NT - 1) / a.dv) - k0 + 1;
    // Gamma per (row, segment): one warp per product, lanes stride over the chunks
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    for (int p = warp; p < rows * a.nseg; p += NT / 32) {
        const int r = p / a.nseg, s = p % a.nseg;
        float g = 1.f;
        if (a.gam) {
            const int c0 = s * a.cps, c1 = min(a.nchunks, c0 + a.cps);
            const float* gp = a.gam + (size_t)bh * a.nchunks * a.dk + k0 + r;
            for (int c = c0 + lane; c < c1; c += 32) g *= gp[(size_t)c * a.dk];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) g *= __shfl_xor_sync(0xffffffffu, g, o);
        }
        if (lane == 0) Gs[p] = g;
    }
    __syncthreads();
    const size_t e = e0 + threadIdx.x;
    if (e >= st) return;
    const int r = (int)(e / a.dv) - k0;
    const float* sp = a.segS + (size_t)bh * a.nseg * st + e;
    float* ip = a.segin + (size_t)bh * a.in_bh + e;
    float S = a.S0 ? a.S0[(size_t)bh * st + e] : 0.f;
    float buf[AHEAD];
    // step i visits segment seg(i): i in the forward order, nseg - 1 - i in the reverse one
    auto seg = [&](int i) { return a.rev ? a.nseg - 1 - i : i; };
#pragma unroll
    for (int i = 0; i < AHEAD; ++i) buf[i] = (i < a.nseg) ? sp[(size_t)seg(i) * st] : 0.f;
    for (int s = 0; s < a.nseg; s += AHEAD) {
#pragma unroll
        for (int i = 0; i < AHEAD; ++i) {
            const int ss = s + i;
            if (ss < a.nseg) {
                const float cur = buf[i];
                if (ss + AHEAD < a.nseg) buf[i] = sp[(size_t)seg(ss + AHEAD) * st];
                ip[(size_t)seg(ss) * st] = S;
                S = fmaf(Gs[r * a.nseg + seg(ss)], S, cur);
            }
        }
    }
    if (a.ST) a.ST[(size_t)bh * a.st_bh + e] = S;
}

}  // namespace

cudaError_t launch_seg_scan(const gla_fwd_params& p, const Plan& pl, void* ws, int* status, cudaStream_t s)
{
    (void)status;
    uint8_t* base = static_cast<uint8_t*>(ws);
    if (pl.st_nseg < 1 || pl.segin_n != pl.st_nseg + 1) return cudaErrorInvalidValue;
    const size_t st = (size_t)p.dk * p.dv;
    ScanArgs a;
    // the state pass's pieces from S0; the state after the last piece, where the last
    // segment starts, is kept as the final start state (its chunk pass writes S_T)
    a.S0 = p.S0;
    a.gam = p.gate == GLA_GATE_NONE ? nullptr : reinterpret_cast<const float*>(base + pl.off_gam);
    a.segS = reinterpret_cast<const float*>(base + pl.off_segS);
    a.segin = reinterpret_cast<float*>(base + pl.off_segin);
    a.in_bh = (long long)pl.segin_n * st;
    a.ST = a.segin + (size_t)pl.st_nseg * st;
    a.st_bh = a.in_bh;
    a.dk = p.dk; a.dv = p.dv; a.nchunks = pl.nchunks; a.nseg = pl.st_nseg; a.cps = pl.st_cps;
    a.rev = 0;
    dim3 grid((unsigned)((st + NT - 1) / NT), p.B * p.H);
    // rows one CTA touches: NT elements span at most NT / dv + 2 rows
    const int max_rows = NT / p.dv + 2;
    const size_t smem = (size_t)max_rows * a.nseg * sizeof(float);
    gla_state_scan_kernel<<<grid, NT, smem, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_seg_scan_job(const SegScanJob& j, cudaStream_t s)
{
    ScanArgs a;
    a.S0 = j.S_start;
    a.ST = j.S_end;
    a.gam = j.gam;
    a.segS = j.segS;
    a.segin = j.segin;
    a.in_bh = (long long)j.nseg * j.dk * j.dv;
    a.st_bh = (long long)j.dk * j.dv;
    a.dk = j.dk; a.dv = j.dv; a.nchunks = j.nch; a.nseg = j.nseg; a.cps = j.cps;
    a.rev = j.reverse ? 1 : 0;
    const size_t st = (size_t)j.dk * j.dv;
    dim3 grid((unsigned)((st + NT - 1) / NT), (unsigned)j.BH);
    const int max_rows = NT / j.dv + 2;
    const size_t smem = (size_t)max_rows * j.nseg * sizeof(float);
    gla_state_scan_kernel<<<grid, NT, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace gla
