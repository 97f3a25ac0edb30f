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
// exits.  Its device address is looked up once per device, with that device
// current, by the first call on the device (cudaGetSymbolAddress); make that
// first call before any stream capture.  All calls share the array: two calls
// whose work overlaps on the GPU (different streams, or different host
// threads) race on it and give wrong results; serialise them.  The array keeps
// the previous call's contents; every call overwrites all of the part it reads
// (segment sums and their scan, or an explicit clear when there is a single
// segment), so nothing stale is read.
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

constexpr size_t kNoallocScratchBytes = size_t(16) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDev = 64;
void* g_scratch_ptr[kMaxDev] = {};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device.
cudaError_t scratch_address(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> g(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

// The regular plan, with fewer segments if its segment states would not fit.
bool fit_plan(const la_shape& s, Plan* p) {
    *p = make_plan(s, LA_OP_CAUSAL_FWD);
    const size_t per_seg = (size_t)s.B * s.H * plan_state_elems(*p) * sizeof(float);
    const size_t max_P = kNoallocScratchBytes / per_seg;
    if (max_P < 1) return false;
    if ((size_t)p->P > max_P) {
        const int P = (int)max_P;
        p->cps = (p->nchunks + P - 1) / P;
        p->P = (p->nchunks + p->cps - 1) / p->cps;
    }
    return (size_t)p->P * per_seg <= kNoallocScratchBytes;
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
    if (!fit_plan(s, &p))
        return failed(LA_ERR_WORKSPACE,
                      "la_causal_fwd_noalloc: B*H*(Dk*Dv+Dk)*4 bytes exceed its 16 MiB static scratch; "
                      "use la_causal_fwd with a caller workspace");
    void* scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess)
        return failed(LA_ERR_CUDA, "la_causal_fwd_noalloc: cudaGetSymbolAddress of the static scratch failed");
    float* seg = static_cast<float*>(scratch);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const size_t seg_bytes = (size_t)s.B * s.H * p.P * plan_state_elems(p) * sizeof(float);
    cudaError_t e;
    if (p.P > 1) {
        e = p.tc ? tc_causal_fwd(nullptr, k, v, nullptr, seg, s, p, false, st) : simt_segment_sums(k, v, seg, s, p, st);
        if (e != cudaSuccess) return LA_ERR_CUDA;
        if (scan_segments(seg, nullptr, s, p, SCAN_EXCLUSIVE_PREFIX, st) != cudaSuccess) return LA_ERR_CUDA;
    } else if (cudaMemsetAsync(seg, 0, seg_bytes, st) != cudaSuccess) {
        return LA_ERR_CUDA;
    }
    e = p.tc ? tc_causal_fwd(q, k, v, o, seg, s, p, true, st) : simt_causal_fwd_out(q, k, v, o, seg, s, p, st);
    return e == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}
