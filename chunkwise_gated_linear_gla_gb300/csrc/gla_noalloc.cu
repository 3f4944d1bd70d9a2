// gla_fwd_noalloc: the forward pass for callers that cannot allocate device
// memory. Its workspace is a fixed array of GLA_NOALLOC_SCRATCH_BYTES in the
// library's own device memory instead of a cudaMalloc/cudaMallocAsync
// buffer.
//
// Who needs this: a host that has handed (nearly) all of the GPU's memory to
// its own pool allocator, so a raw cudaMalloc would fail or fragment it; a
// latency-critical loop where cudaMalloc/cudaFree are forbidden because they
// can synchronise the device; a plugin interface that gives the kernel no
// allocator at all. Such a caller still owns and passes every input and
// output; only the intermediate workspace lives here.
//
// The array is a file-scope __device__ object, so every GPU that loads this
// library holds its 32 MiB until the process exits. Host code cannot use the
// array's name as a device address (on the host it is only a stand-in), so
// the first call on each device looks the address up with
// cudaGetSymbolAddress while that device is current and caches it; make that
// first call before any stream capture. The kernels write every workspace
// byte they later read, so nothing has to be cleared between calls. All calls
// on a device share the one array: calls whose work overlaps on the GPU (on
// different streams, or from different host threads without ordering) race
// on it and must be serialised by the caller.
#include <cstring>
#include <mutex>

#include "gla_internal.h"

namespace gla {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[GLA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once).
cudaError_t scratch_address(void** out)
{
    int d = 0;
    cudaError_t e = cudaGetDevice(&d);
    if (e != cudaSuccess) return e;
    if (d < 0 || d >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[d]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[d] = p;
    }
    *out = g_scratch_ptr[d];
    return cudaSuccess;
}

}  // namespace
}  // namespace gla

extern "C" gla_status gla_fwd_noalloc(const void* q, const void* k, const void* v, const float* log_g,
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
    p.force_segments = 1;   // one segment: no per-segment state buffers in the scratch
    if (gla_fwd_num_stages(&p) < 0) return gla_fwd_ex(&p, stream);   // reports the argument error
    const size_t need = gla_fwd_workspace_size(&p);
    if (need > (size_t)GLA_NOALLOC_SCRATCH_BYTES) return GLA_ERR_WORKSPACE;
    if (need > 0) {
        void* ws = nullptr;
        if (gla::scratch_address(&ws) != cudaSuccess) return GLA_ERR_CUDA;
        p.workspace = ws;
        p.workspace_bytes = need;
    }
    return gla_fwd_ex(&p, stream);
}
