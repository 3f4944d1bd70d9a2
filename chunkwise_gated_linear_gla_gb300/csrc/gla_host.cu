// gla_fwd_host: the forward pass with every tensor in host memory. The call
// copies the inputs to the device, runs the pass and copies O and S_T back,
// one slice of the batch at a time, so that on the GPU the copy-in of slice
// j+1, the compute of slice j and the copy-out of slice j-1 run together:
//
//   copy-in stream   H2D(0) H2D(1) H2D(2) H2D(3) ...
//   compute stream          C(0)   C(1)   C(2)   ...
//   copy-out stream                D2H(0) D2H(1) ...
//
// A slice is a run of whole batch rows, or, when there are fewer batch rows
// than slices wanted, a run of heads of one batch row; every (b, h) pair is an
// independent problem, so each slice is an ordinary gla_fwd_ex call on its
// own device buffers. Three slots of device buffers (inputs, O, S_T) rotate
// through the three stages; the compute stream runs one slice at a time, so
// all slices share one workspace. The device memory comes from a memory pool
// private to the library that keeps its pages between calls (returned by
// gla_host_release), so a steady stream of calls maps no memory.
//
// The library's three streams and their events exist once per device; a
// mutex makes calls on one device take turns (the call is synchronous).
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "gla_internal.h"

namespace gla {
namespace {

constexpr int kSlots = 3;
constexpr size_t kDefaultSliceBytes = size_t(48) << 20;
constexpr int kMaxDevices = 64;

struct HostCtx {
    std::mutex mu;   // held for the whole of a call
    bool init = false;
    cudaMemPool_t pool = nullptr;
    cudaStream_t s_in = nullptr, s_cmp = nullptr, s_out = nullptr;
    cudaEvent_t ev_start = nullptr, ev_done = nullptr;
    cudaEvent_t ev_in[kSlots] = {}, ev_cmp[kSlots] = {}, ev_out[kSlots] = {};
};
HostCtx g_host[kMaxDevices];

cudaError_t init_ctx(HostCtx& c, int dev)
{
    if (c.init) return cudaSuccess;
    cudaMemPoolProps props;
    std::memset(&props, 0, sizeof(props));
    props.allocType = cudaMemAllocationTypePinned;
    props.handleTypes = cudaMemHandleTypeNone;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaError_t e = cudaMemPoolCreate(&c.pool, &props);
    if (e != cudaSuccess) return e;
    uint64_t keep = UINT64_MAX;   // never hand pages back at a synchronisation point
    e = cudaMemPoolSetAttribute(c.pool, cudaMemPoolAttrReleaseThreshold, &keep);
    if (e != cudaSuccess) return e;
    for (cudaStream_t* s : {&c.s_in, &c.s_cmp, &c.s_out})
        if ((e = cudaStreamCreateWithFlags(s, cudaStreamNonBlocking)) != cudaSuccess) return e;
    std::vector<cudaEvent_t*> evs = {&c.ev_start, &c.ev_done};
    for (int i = 0; i < kSlots; ++i) {
        evs.push_back(&c.ev_in[i]);
        evs.push_back(&c.ev_cmp[i]);
        evs.push_back(&c.ev_out[i]);
    }
    for (cudaEvent_t* ev : evs)
        if ((e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming)) != cudaSuccess) return e;
    c.init = true;
    return cudaSuccess;
}

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

struct Slice {
    int b0, nb, h0, nh;   // batch rows b0..b0+nb-1, heads h0..h0+nh-1 of each
};

// Splits x in two (rows if it has several, else heads); false if x is one (b, h) pair.
bool halve(const Slice& x, Slice& a, Slice& b)
{
    if (x.nb > 1) {
        a = {x.b0, x.nb / 2, x.h0, x.nh};
        b = {x.b0 + x.nb / 2, x.nb - x.nb / 2, x.h0, x.nh};
        return true;
    }
    if (x.nh > 1) {
        a = {x.b0, 1, x.h0, x.nh / 2};
        b = {x.b0, 1, x.h0 + x.nh / 2, x.nh - x.nh / 2};
        return true;
    }
    return false;
}

// Slices of about `target` bytes of copy traffic each. The last slice is
// halved twice: after the final copy-in only the last slice's compute and
// copy-out remain, so a small last slice shortens that tail.
std::vector<Slice> plan_slices(const gla_fwd_params& p, size_t per_unit, size_t target)
{
    std::vector<Slice> out;
    const long long units = (long long)p.B * p.H;
    long long want = per_unit == 0 ? 1 : (long long)((units * per_unit + target - 1) / target);
    want = std::max(1LL, std::min(want, units));
    if (want == 1) {
        out.push_back({0, p.B, 0, p.H});
    } else if (want <= p.B) {
        const int nb = (int)((p.B + want - 1) / want);
        for (int b = 0; b < p.B; b += nb) out.push_back({b, std::min(nb, p.B - b), 0, p.H});
    } else {
        const long long groups = (want + p.B - 1) / p.B;   // head groups per batch row
        const int nh = (int)((p.H + groups - 1) / groups);
        for (int b = 0; b < p.B; ++b)
            for (int h = 0; h < p.H; h += nh) out.push_back({b, 1, h, std::min(nh, p.H - h)});
    }
    if (out.size() > 1) {
        for (int i = 0; i < 2; ++i) {
            Slice a, b;
            if (!halve(out.back(), a, b)) break;
            out.back() = a;
            out.push_back(b);
        }
    }
    return out;
}

struct Sizes {   // bytes per (b, h) pair of each tensor
    size_t q, v, g, b, s;
};

Sizes unit_sizes(const gla_fwd_params& p)
{
    const size_t e = p.dtype == GLA_BF16 ? 2 : 4;
    Sizes z;
    z.q = (size_t)p.T * p.dk * e;
    z.v = (size_t)p.T * p.dv * e;
    z.g = (p.gate == GLA_GATE_PER_KEY || p.gate == GLA_GATE_BILINEAR) ? (size_t)p.T * p.dk * 4
        : p.gate == GLA_GATE_TOKEN_SCALAR ? (size_t)p.T * 4 : 0;
    z.b = p.gate == GLA_GATE_BILINEAR ? (size_t)p.T * p.dv * 4 : 0;
    z.s = (size_t)p.dk * p.dv * 4;
    return z;
}

cudaError_t h2d(void* dst, const void* src, size_t n, cudaStream_t s)
{
    return n == 0 ? cudaSuccess : cudaMemcpyAsync(dst, src, n, cudaMemcpyHostToDevice, s);
}

cudaError_t d2h(void* dst, const void* src, size_t n, cudaStream_t s)
{
    return n == 0 ? cudaSuccess : cudaMemcpyAsync(dst, src, n, cudaMemcpyDeviceToHost, s);
}

}  // namespace
}  // namespace gla

using namespace gla;

extern "C" gla_status gla_fwd_host(const gla_fwd_params* hp, size_t slice_bytes, cudaStream_t stream)
{
    gla_status st = validate_args(hp);
    if (st != GLA_OK) return st;
    st = validate_pointers(hp, false);
    if (st != GLA_OK) return st;
    const gla_fwd_params& p = *hp;
    const Sizes z = unit_sizes(p);
    const size_t per_unit = 2 * z.q + 2 * z.v + z.g + z.b + (p.S0 ? z.s : 0) + (p.ST ? z.s : 0);
    const std::vector<Slice> sl = plan_slices(p, per_unit, slice_bytes ? slice_bytes : kDefaultSliceBytes);
    const int nsl = (int)sl.size();
    const int nslot = std::min(kSlots, nsl);

    // per-slot buffers sized for the largest slice; one workspace for all slices
    size_t umax = 0, ws = 0;
    for (const Slice& x : sl) {
        umax = std::max(umax, (size_t)x.nb * x.nh);
        gla_fwd_params t = p;
        t.B = x.nb;
        t.H = x.nh;
        size_t w = 0;
        if ((st = plan_workspace(&t, &w)) != GLA_OK) return st;
        ws = std::max(ws, w);
    }
    const size_t o_q = 0, o_k = o_q + up256(umax * z.q), o_v = o_k + up256(umax * z.q);
    const size_t o_g = o_v + up256(umax * z.v), o_b = o_g + up256(umax * z.g), o_s0 = o_b + up256(umax * z.b);
    const size_t o_o = o_s0 + up256(p.S0 ? umax * z.s : 0), o_st = o_o + up256(umax * z.v);
    const size_t slot = o_st + up256(p.ST ? umax * z.s : 0);
    const size_t scal = p.gate == GLA_GATE_HEAD_SCALAR ? up256((size_t)p.H * 4) : 0;
    const size_t total = nslot * slot + up256(ws) + scal;

    // every argument error is reported above, before the device is touched
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GLA_ERR_CUDA;
    HostCtx& c = g_host[dev];
    std::lock_guard<std::mutex> lk(c.mu);
    if (init_ctx(c, dev) != cudaSuccess) return GLA_ERR_CUDA;

    const uint8_t* hq = static_cast<const uint8_t*>(p.q);
    const uint8_t* hk = static_cast<const uint8_t*>(p.k);
    const uint8_t* hv = static_cast<const uint8_t*>(p.v);
    const uint8_t* hg = reinterpret_cast<const uint8_t*>(p.log_g);
    const uint8_t* hb = reinterpret_cast<const uint8_t*>(p.log_b);
    const uint8_t* hs0 = reinterpret_cast<const uint8_t*>(p.S0);
    uint8_t* ho = static_cast<uint8_t*>(p.O);
    uint8_t* hst = reinterpret_cast<uint8_t*>(p.ST);

    bool ok = cudaEventRecord(c.ev_start, stream) == cudaSuccess;
    for (cudaStream_t s : {c.s_in, c.s_cmp, c.s_out})
        ok = ok && cudaStreamWaitEvent(s, c.ev_start, 0) == cudaSuccess;
    uint8_t* base = nullptr;
    ok = ok && cudaMallocFromPoolAsync(reinterpret_cast<void**>(&base), total, c.pool, c.s_in) == cudaSuccess;
    if (!ok) {
        cudaStreamSynchronize(c.s_in);
        return GLA_ERR_CUDA;
    }
    uint8_t* dws = base + nslot * slot;
    float* dscal = reinterpret_cast<float*>(dws + up256(ws));
    if (scal) ok = h2d(dscal, p.log_g, (size_t)p.H * 4, c.s_in) == cudaSuccess;

    // copy-out of slice j is enqueued after the copy-in and compute of slice j+1, so
    // that a copy to pageable memory (which blocks the host) never holds back the next slice
    auto copy_out = [&](int j) -> bool {
        const Slice& x = sl[j];
        const int s = j % kSlots;
        uint8_t* b = base + s * slot;
        const size_t u0 = (size_t)x.b0 * p.H + x.h0, nu = (size_t)x.nb * x.nh;
        bool r = cudaStreamWaitEvent(c.s_out, c.ev_cmp[s], 0) == cudaSuccess;
        r = r && d2h(ho + u0 * z.v, b + o_o, nu * z.v, c.s_out) == cudaSuccess;
        if (p.ST) r = r && d2h(hst + u0 * z.s, b + o_st, nu * z.s, c.s_out) == cudaSuccess;
        return r && cudaEventRecord(c.ev_out[s], c.s_out) == cudaSuccess;
    };
    for (int j = 0; j < nsl && ok && st == GLA_OK; ++j) {
        const Slice& x = sl[j];
        const int s = j % kSlots;
        uint8_t* b = base + s * slot;
        const size_t u0 = (size_t)x.b0 * p.H + x.h0, nu = (size_t)x.nb * x.nh;
        if (j >= kSlots) ok = cudaStreamWaitEvent(c.s_in, c.ev_out[s], 0) == cudaSuccess;
        ok = ok && h2d(b + o_q, hq + u0 * z.q, nu * z.q, c.s_in) == cudaSuccess;
        ok = ok && h2d(b + o_k, hk + u0 * z.q, nu * z.q, c.s_in) == cudaSuccess;
        ok = ok && h2d(b + o_v, hv + u0 * z.v, nu * z.v, c.s_in) == cudaSuccess;
        if (z.g) ok = ok && h2d(b + o_g, hg + u0 * z.g, nu * z.g, c.s_in) == cudaSuccess;
        if (z.b) ok = ok && h2d(b + o_b, hb + u0 * z.b, nu * z.b, c.s_in) == cudaSuccess;
        if (p.S0) ok = ok && h2d(b + o_s0, hs0 + u0 * z.s, nu * z.s, c.s_in) == cudaSuccess;
        ok = ok && cudaEventRecord(c.ev_in[s], c.s_in) == cudaSuccess;
        ok = ok && cudaStreamWaitEvent(c.s_cmp, c.ev_in[s], 0) == cudaSuccess;
        if (!ok) break;

        gla_fwd_params t = p;
        t.B = x.nb;
        t.H = x.nh;
        t.q = b + o_q;
        t.k = b + o_k;
        t.v = b + o_v;
        t.log_g = z.g ? reinterpret_cast<const float*>(b + o_g)
                : p.gate == GLA_GATE_HEAD_SCALAR ? dscal + x.h0 : nullptr;
        t.log_b = z.b ? reinterpret_cast<const float*>(b + o_b) : nullptr;
        t.S0 = p.S0 ? reinterpret_cast<const float*>(b + o_s0) : nullptr;
        t.O = b + o_o;
        t.ST = p.ST ? reinterpret_cast<float*>(b + o_st) : nullptr;
        t.workspace = ws ? dws : nullptr;
        t.workspace_bytes = ws;
        st = gla_fwd_ex(&t, c.s_cmp);
        ok = st == GLA_OK && cudaEventRecord(c.ev_cmp[s], c.s_cmp) == cudaSuccess;
        if (ok && j >= 1) ok = copy_out(j - 1);
    }
    if (ok && st == GLA_OK && nsl > 0) ok = copy_out(nsl - 1);

    // the buffers go back to the pool once every stream is done with them
    bool fin = cudaEventRecord(c.ev_done, c.s_cmp) == cudaSuccess &&
               cudaStreamWaitEvent(c.s_out, c.ev_done, 0) == cudaSuccess &&
               cudaEventRecord(c.ev_done, c.s_in) == cudaSuccess &&
               cudaStreamWaitEvent(c.s_out, c.ev_done, 0) == cudaSuccess &&
               cudaFreeAsync(base, c.s_out) == cudaSuccess &&
               cudaEventRecord(c.ev_done, c.s_out) == cudaSuccess &&
               cudaStreamWaitEvent(stream, c.ev_done, 0) == cudaSuccess;
    for (cudaStream_t s : {c.s_in, c.s_cmp, c.s_out})
        fin = (cudaStreamSynchronize(s) == cudaSuccess) && fin;
    if (st != GLA_OK) return st;
    return ok && fin ? GLA_OK : GLA_ERR_CUDA;
}

extern "C" gla_status gla_host_release(void)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GLA_ERR_CUDA;
    HostCtx& c = g_host[dev];
    std::lock_guard<std::mutex> lk(c.mu);
    if (!c.init) return GLA_OK;
    return cudaMemPoolTrimTo(c.pool, 0) == cudaSuccess ? GLA_OK : GLA_ERR_CUDA;
}
