// gla_state_scan: the short serial recurrence over sequence segments that
// lets small B*H fill the GPU. Each segment s was first run from a zero state
// (gla_chunk_fwd in state-only mode), giving S*_s. Because the recurrence is
// linear in S and the gate only scales rows, the true state entering segment
// s+1 is
//     S_in(s+1) = Diag(Gamma_s) S_in(s) + S*_s,   Gamma_s = prod over the
//                 segment's chunks of gamma (per key),
// the state correction of the FlashQLA talk ("core technical principles":
// a wrongly started segment is fixed by one matrix per rank), which for a
// diagonal gate collapses from a dk x dk matrix to the vector Gamma_s. With
// S_in(0) = S0 this also yields S_T = S_in(nseg). One CTA handles 8 rows of
// the state of one (b,h) for all dv columns.
#include "gla_internal.h"

namespace gla {
namespace {

constexpr int ROWS = 8;
constexpr int NT = 256;

struct ScanArgs {
    const float* S0;     // [BH][dk][dv] or null
    float* ST;           // [BH][dk][dv] or null
    const float* gam;    // [BH][nchunks][dk] or null (no gate)
    const float* segS;   // [BH][nseg][dk][dv]
    float* segin;        // [BH][nseg][dk][dv]
    int dk, dv, nchunks, nseg, cps;
};

__global__ void __launch_bounds__(NT) gla_state_scan_kernel(ScanArgs a)
{
    extern __shared__ float Gs[];   // [nseg][ROWS]
    const int bh = blockIdx.x, k0 = blockIdx.y * ROWS;
    for (int p = threadIdx.x; p < a.nseg * ROWS; p += NT) {
        const int s = p / ROWS, r = p % ROWS;
        float g = 1.f;
        if (a.gam) {
            const int c0 = s * a.cps, c1 = min(a.nchunks, c0 + a.cps);
            const float* gp = a.gam + ((size_t)bh * a.nchunks) * a.dk + k0 + r;
            for (int c = c0; c < c1; ++c) g *= gp[(size_t)c * a.dk];
        }
        Gs[p] = g;
    }
    __syncthreads();
    const size_t st = (size_t)a.dk * a.dv;
    for (int e = threadIdx.x; e < ROWS * a.dv; e += NT) {
        const int r = e / a.dv, j = e % a.dv;
        const size_t off = (size_t)(k0 + r) * a.dv + j;
        float S = a.S0 ? a.S0[(size_t)bh * st + off] : 0.f;
        for (int s = 0; s < a.nseg; ++s) {
            const size_t o = ((size_t)bh * a.nseg + s) * st + off;
            a.segin[o] = S;
            S = fmaf(Gs[s * ROWS + r], S, a.segS[o]);
        }
        if (a.ST) a.ST[(size_t)bh * st + off] = S;
    }
}

}  // namespace

cudaError_t launch_seg_scan(const gla_fwd_params& p, const Plan& pl, void* ws, int* status, cudaStream_t s)
{
    (void)status;
    uint8_t* base = static_cast<uint8_t*>(ws);
    ScanArgs a;
    a.S0 = p.S0;
    a.ST = p.ST;
    a.gam = p.gate == GLA_GATE_NONE ? nullptr : reinterpret_cast<const float*>(base + pl.off_gam);
    a.segS = reinterpret_cast<const float*>(base + pl.off_segS);
    a.segin = reinterpret_cast<float*>(base + pl.off_segin);
    a.dk = p.dk; a.dv = p.dv; a.nchunks = pl.nchunks; a.nseg = pl.nseg; a.cps = pl.chunks_per_seg;
    dim3 grid(p.B * p.H, p.dk / ROWS);
    const size_t smem = (size_t)pl.nseg * ROWS * sizeof(float);
    gla_state_scan_kernel<<<grid, NT, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace gla
