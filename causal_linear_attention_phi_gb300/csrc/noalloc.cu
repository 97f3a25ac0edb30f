// noalloc.cu -- la_causal_fwd_noalloc: the causal forward with its scratch in a
// fixed, library-owned device array instead of a caller-provided workspace.
//
// Who needs it: callers that cannot allocate device memory when they call the
// library -- for example a plugin running inside a host framework that owns
// every device allocation and hands its plugins no workspace, or a
// latency-critical loop in which a cudaMalloc (which may synchronise the
// device) is not allowed after start-up.  They still pass q, k, v and o.
//
// The scratch is one file-scope __device__ array of kNoallocScratchBytes
// (16 MiB).  Every GPU that loads the library holds it until the process
// exits.  Its device address is looked up with cudaGetSymbolAddress by the
// first call on a device (that device current) and cached together with the
// CUDA context it belongs to; a call under another context of that device (the
// primary context destroyed and re-created, e.g. after cudaDeviceReset) looks
// it up again instead of using a stale address.  Make the first call on a
// device before any stream capture.  All calls share the array: two calls
// whose work overlaps on the GPU (different streams, or different host
// threads) race on it and give wrong results; serialise them.  The array keeps
// the previous call's contents; every call overwrites all of the part it reads
// (segment sums and their scan, or an explicit clear when there is a single
// segment), so nothing stale is read.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>
#include <mutex>

#include "la_internal.cuh"

namespace la {
la_status checked_shape(const la_shape& s);
la_status checked_device();
la_status checked_ptr(const void* p, const char* what);
la_status failed(la_status st, const char* msg);
void clear_detail();

namespace {

constexpr size_t kNoallocScratchBytes = size_t(16) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDev = 64;
void* g_scratch_ptr[kMaxDev] = {};
CUcontext g_scratch_ctx[kMaxDev] = {};
std::mutex g_scratch_mu;

// cuCtxGetCurrent through the runtime's driver entry-point query (the library
// links the runtime only).
PFN_cuCtxGetCurrent_v4000 ctx_get_current() {
    static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(ptr);
    });
    return fn;
}

// Device address of the scratch array on the current device, looked up again
// whenever the current context is not the one the cached address came from.
cudaError_t scratch_address(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    CUcontext ctx = nullptr;
    auto get = ctx_get_current();
    if (!get || get(&ctx) != CUDA_SUCCESS) return cudaErrorInitializationError;
    std::lock_guard<std::mutex> g(g_scratch_mu);
    if (!ctx || !g_scratch_ptr[dev] || g_scratch_ctx[dev] != ctx) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);  // initialises the context if none is current yet
        if (e != cudaSuccess) return e;
        if (!ctx && get(&ctx) != CUDA_SUCCESS) return cudaErrorInitializationError;
        g_scratch_ptr[dev] = p;
        g_scratch_ctx[dev] = ctx;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

// The regular plan, with fewer segments if its segment states would not fit.
// A state record holds plan_state_elems(p) floats: Dk*Dv + Dk on the CUDA-core
// path, and 128*128 + 128 on the tensor-core path (bf16 heads of 64 or 128),
// whose records keep the padded 128-wide layout.
size_t record_bytes(const Plan& p) { return plan_state_elems(p) * sizeof(float); }

bool fit_plan(const la_shape& s, Plan* p) {
    *p = make_plan(s, LA_OP_CAUSAL_FWD);
    const size_t per_seg = (size_t)s.B * s.H * record_bytes(*p);
    const size_t max_P = kNoallocScratchBytes / per_seg;
    if (max_P < 1) return false;
    if ((size_t)p->P > max_P) {
        const int P = (int)max_P;
        p->cps = (p->nchunks + P - 1) / P;
        p->P = (p->nchunks + p->cps - 1) / p->cps;
    }
    return (size_t)p->P * per_seg <= kNoallocScratchBytes;
}

// LA_ERR_CUDA with the failing stage and CUDA's message in la_error_detail().
la_status stage_failed(const char* stage, cudaError_t e) {
    char msg[256];
    snprintf(msg, sizeof msg, "la_causal_fwd_noalloc: %s failed: %s", stage, cudaGetErrorString(e));
    return failed(LA_ERR_CUDA, msg);
}

}  // namespace
}  // namespace la

using namespace la;

extern "C" la_status la_causal_fwd_noalloc(const void* q, const void* k, const void* v, void* o, la_shape s,
                                           la_stream_t stream) {
    // the same argument checks as la_causal_fwd, all before any launch
    clear_detail();
    la_status st0 = checked_shape(s);
    if (st0 != LA_OK) return st0;
    if (s.B == 0 || s.H == 0 || s.N == 0) return LA_OK;
    if ((st0 = checked_device()) != LA_OK) return st0;
    if ((st0 = checked_ptr(q, "q")) != LA_OK || (st0 = checked_ptr(k, "k")) != LA_OK ||
        (st0 = checked_ptr(v, "v")) != LA_OK || (st0 = checked_ptr(o, "o")) != LA_OK)
        return st0;
    Plan p;
    if (!fit_plan(s, &p)) {
        char msg[320];
        snprintf(msg, sizeof msg,
                 "la_causal_fwd_noalloc: B*H = %lld state records of %zu bytes (%s) exceed its 16 MiB static "
                 "scratch; use la_causal_fwd with a caller workspace",
                 (long long)s.B * s.H, record_bytes(p),
                 p.tc ? "128 x 128 + 128 floats, the padded tensor-core layout" : "(Dk*Dv + Dk) floats");
        return failed(LA_ERR_WORKSPACE, msg);
    }
    void* scratch = nullptr;
    cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess) return stage_failed("cudaGetSymbolAddress of the static scratch", e);
    float* seg = static_cast<float*>(scratch);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const size_t seg_bytes = (size_t)s.B * s.H * p.P * plan_state_elems(p) * sizeof(float);
    if (p.P > 1) {
        e = p.tc ? tc_causal_fwd(nullptr, k, v, nullptr, seg, s, p, false, st) : simt_segment_sums(k, v, seg, s, p, st);
        if (e != cudaSuccess) return stage_failed("segment sums", e);
        e = scan_segments(seg, nullptr, s, p, SCAN_EXCLUSIVE_PREFIX, st);
        if (e != cudaSuccess) return stage_failed("segment scan", e);
    } else if ((e = cudaMemsetAsync(seg, 0, seg_bytes, st)) != cudaSuccess) {
        return stage_failed("state clear", e);
    }
    e = p.tc ? tc_causal_fwd(q, k, v, o, seg, s, p, true, st) : simt_causal_fwd_out(q, k, v, o, seg, s, p, st);
    return e == cudaSuccess ? LA_OK : stage_failed("causal forward", e);
}
