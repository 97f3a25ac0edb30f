// host_step.cu -- la_causal_step_host: one training step (causal forward, then
// the backward that reads the forward's segment states) on host-resident data,
// with the transfers overlapped with the kernels.
//
// Heads are independent ("Transformers은 RNN이다" digest, 핵심 구성요소 2-3:
// every head carries its own state), so the B*H heads are cut into groups of
// consecutive heads, which are contiguous in the [B,H,N,D] layout.  Three
// streams form a pipeline over the groups: host->device copies of group g+1,
// the kernels of group g and device->host copies of group g-1 run at the same
// time.  The device side holds two slots of group buffers (inputs q, k, v,
// dout and outputs o, dq, dk, dv), so a slot is refilled only after the
// kernels of the group two back have read it and its outputs have been copied
// out.  The streams and events are created once per device and kept.
#include <algorithm>
#include <mutex>

#include "la_internal.cuh"

namespace la {
la_status checked_shape(const la_shape& s);
la_status checked_device();
la_status checked_ptr(const void* p, const char* what);
la_status failed(la_status st, const char* msg);
void clear_detail();

namespace {

constexpr int kMaxDev = 64;
constexpr int kSlots = 2;

struct Pipe {
    cudaStream_t in = nullptr, comp = nullptr, out = nullptr;
    cudaEvent_t start = nullptr;
    cudaEvent_t in_ready[kSlots] = {}, computed[kSlots] = {}, out_done[kSlots] = {};
};
Pipe g_pipe[kMaxDev];
std::mutex g_pipe_mu;

cudaError_t get_pipe(Pipe** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> g(g_pipe_mu);
    Pipe& p = g_pipe[dev];
    if (!p.in) {
        Pipe n;
        const unsigned ef = cudaEventDisableTiming;
        if ((e = cudaStreamCreateWithFlags(&n.in, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaStreamCreateWithFlags(&n.comp, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaStreamCreateWithFlags(&n.out, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&n.start, ef)) != cudaSuccess)
            return e;
        for (int i = 0; i < kSlots; ++i)
            if ((e = cudaEventCreateWithFlags(&n.in_ready[i], ef)) != cudaSuccess ||
                (e = cudaEventCreateWithFlags(&n.computed[i], ef)) != cudaSuccess ||
                (e = cudaEventCreateWithFlags(&n.out_done[i], ef)) != cudaSuccess)
                return e;
        p = n;
    }
    *out = &p;
    return cudaSuccess;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

la_shape group_shape(const la_shape& s, int heads) {
    la_shape g = s;
    g.B = 1;
    g.H = heads;
    return g;
}

// Byte layout of the device scratch for groups of `G` heads.
struct HostStepLayout {
    size_t q, k, v, dout, o, dq, dk, dv;  // offsets inside a slot
    size_t slot;                          // bytes per slot
    size_t ws_f, ws_b;                    // offsets of the two workspaces
    size_t ws_f_bytes, ws_b_bytes;
    size_t bytes;
};

HostStepLayout host_step_layout(const la_shape& s, int G) {
    HostStepLayout L{};
    const size_t es = s.dtype == LA_BF16 ? 2 : 4;
    const size_t nk = align256((size_t)G * s.N * s.Dk * es), nv = align256((size_t)G * s.N * s.Dv * es);
    size_t off = 0;
    L.q = off, off += nk;
    L.k = off, off += nk;
    L.v = off, off += nv;
    L.dout = off, off += nv;
    L.o = off, off += nv;
    L.dq = off, off += nk;
    L.dk = off, off += nk;
    L.dv = off, off += nv;
    L.slot = off;
    // the last group may be smaller, and a smaller group may be cut into more segments
    const int BH = s.B * s.H, rem = BH % G;
    size_t wf = la_workspace_bytes(LA_OP_CAUSAL_FWD, group_shape(s, G));
    size_t wb = la_workspace_bytes(LA_OP_CAUSAL_BWD, group_shape(s, G));
    if (rem) {
        wf = std::max(wf, la_workspace_bytes(LA_OP_CAUSAL_FWD, group_shape(s, rem)));
        wb = std::max(wb, la_workspace_bytes(LA_OP_CAUSAL_BWD, group_shape(s, rem)));
    }
    L.ws_f_bytes = wf;
    L.ws_b_bytes = wb;
    L.ws_f = kSlots * L.slot;
    L.ws_b = L.ws_f + align256(wf);
    L.bytes = L.ws_b + align256(wb);
    return L;
}

la_status check_host(const void* p, const char* what) {
    if (!p) return failed(LA_ERR_INVALID_ARG, what);
    if (reinterpret_cast<uintptr_t>(p) & 15) return failed(LA_ERR_INVALID_ARG, "host buffer not 16-byte aligned");
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return failed(LA_ERR_INVALID_ARG, "host buffer: pointer query failed");
    }
    if (a.type != cudaMemoryTypeHost)
        return failed(LA_ERR_INVALID_ARG, "host buffers must be pinned (page-locked) host memory");
    return LA_OK;
}

}  // namespace
}  // namespace la

using namespace la;

extern "C" size_t la_host_step_bytes(la_shape s, int group_heads) {
    if (checked_shape(s) != LA_OK || group_heads < 1 || s.B == 0 || s.H == 0 || s.N == 0) return 0;
    return host_step_layout(s, std::min(group_heads, s.B * s.H)).bytes;
}

extern "C" la_status la_causal_step_host(const void* q, const void* k, const void* v, const void* dout, void* o,
                                         void* dq, void* dk, void* dv, la_shape s, int group_heads, void* dev_buf,
                                         size_t dev_bytes, la_stream_t stream) {
    clear_detail();
    la_status st = checked_shape(s);
    if (st != LA_OK) return st;
    if (group_heads < 1) return failed(LA_ERR_INVALID_ARG, "group_heads must be at least 1");
    if (s.B == 0 || s.H == 0 || s.N == 0) return LA_OK;
    if ((st = checked_device()) != LA_OK) return st;
    const void* hosts[8] = {q, k, v, dout, o, dq, dk, dv};
    const char* names[8] = {"q is NULL", "k is NULL", "v is NULL", "dout is NULL",
                            "o is NULL", "dq is NULL", "dk is NULL", "dv is NULL"};
    for (int i = 0; i < 8; ++i)
        if ((st = check_host(hosts[i], names[i])) != LA_OK) return st;
    const int BH = s.B * s.H, G = std::min(group_heads, BH);
    const HostStepLayout L = host_step_layout(s, G);
    if (!dev_buf || dev_bytes < L.bytes)
        return failed(LA_ERR_WORKSPACE, "device scratch smaller than la_host_step_bytes()");
    if ((st = checked_ptr(dev_buf, "dev_buf")) != LA_OK) return st;
    Pipe* P = nullptr;
    if (get_pipe(&P) != cudaSuccess) return failed(LA_ERR_CUDA, "la_causal_step_host: stream set-up failed");

    const size_t es = s.dtype == LA_BF16 ? 2 : 4;
    const size_t hk = (size_t)s.N * s.Dk * es, hv = (size_t)s.N * s.Dv * es;  // bytes per head
    char* base = static_cast<char*>(dev_buf);
    char* ws_f = base + L.ws_f;
    char* ws_b = base + L.ws_b;
    cudaStream_t user = reinterpret_cast<cudaStream_t>(stream);
#define LA_CU(x)                                                                        \
    do {                                                                                \
        if ((x) != cudaSuccess) return failed(LA_ERR_CUDA, "la_causal_step_host: " #x); \
    } while (0)
    // the pipeline starts after the work already queued on the caller's stream
    LA_CU(cudaEventRecord(P->start, user));
    LA_CU(cudaStreamWaitEvent(P->in, P->start, 0));
    LA_CU(cudaStreamWaitEvent(P->comp, P->start, 0));
    LA_CU(cudaStreamWaitEvent(P->out, P->start, 0));
    const int ngroups = (BH + G - 1) / G;
    for (int g = 0; g < ngroups; ++g) {
        const int slot = g % kSlots, h0 = g * G, nh = std::min(G, BH - h0);
        char* sb = base + slot * L.slot;
        const size_t bk = nh * hk, bv = nh * hv;
        const size_t ok = (size_t)h0 * hk, ov = (size_t)h0 * hv;
        // host -> device, once the kernels of the group that last used this slot are done
        if (g >= kSlots) LA_CU(cudaStreamWaitEvent(P->in, P->computed[slot], 0));
        LA_CU(cudaMemcpyAsync(sb + L.q, static_cast<const char*>(q) + ok, bk, cudaMemcpyHostToDevice, P->in));
        LA_CU(cudaMemcpyAsync(sb + L.k, static_cast<const char*>(k) + ok, bk, cudaMemcpyHostToDevice, P->in));
        LA_CU(cudaMemcpyAsync(sb + L.v, static_cast<const char*>(v) + ov, bv, cudaMemcpyHostToDevice, P->in));
        LA_CU(cudaMemcpyAsync(sb + L.dout, static_cast<const char*>(dout) + ov, bv, cudaMemcpyHostToDevice, P->in));
        LA_CU(cudaEventRecord(P->in_ready[slot], P->in));
        // the step's kernels, once the inputs are in and the slot's previous outputs are out
        LA_CU(cudaStreamWaitEvent(P->comp, P->in_ready[slot], 0));
        if (g >= kSlots) LA_CU(cudaStreamWaitEvent(P->comp, P->out_done[slot], 0));
        const la_shape gs = group_shape(s, nh);
        la_stream_t cs = reinterpret_cast<la_stream_t>(P->comp);
        if ((st = la_causal_fwd(sb + L.q, sb + L.k, sb + L.v, sb + L.o, gs, ws_f, L.ws_f_bytes, cs)) != LA_OK)
            return st;
        if ((st = la_causal_bwd_after_fwd(sb + L.q, sb + L.k, sb + L.v, sb + L.dout, sb + L.dq, sb + L.dk, sb + L.dv,
                                          gs, ws_f, L.ws_f_bytes, ws_b, L.ws_b_bytes, cs)) != LA_OK)
            return st;
        LA_CU(cudaEventRecord(P->computed[slot], P->comp));
        // device -> host
        LA_CU(cudaStreamWaitEvent(P->out, P->computed[slot], 0));
        LA_CU(cudaMemcpyAsync(static_cast<char*>(o) + ov, sb + L.o, bv, cudaMemcpyDeviceToHost, P->out));
        LA_CU(cudaMemcpyAsync(static_cast<char*>(dq) + ok, sb + L.dq, bk, cudaMemcpyDeviceToHost, P->out));
        LA_CU(cudaMemcpyAsync(static_cast<char*>(dk) + ok, sb + L.dk, bk, cudaMemcpyDeviceToHost, P->out));
        LA_CU(cudaMemcpyAsync(static_cast<char*>(dv) + ov, sb + L.dv, bv, cudaMemcpyDeviceToHost, P->out));
        LA_CU(cudaEventRecord(P->out_done[slot], P->out));
    }
    // the caller's stream continues after the last copy out (which follows every kernel)
    LA_CU(cudaStreamWaitEvent(user, P->out_done[(ngroups - 1) % kSlots], 0));
#undef LA_CU
    return LA_OK;
}
