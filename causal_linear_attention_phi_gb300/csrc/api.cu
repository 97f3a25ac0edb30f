// api.cu -- the extern "C" entry points of libla: argument checks, work
// planning, workspace carving and kernel dispatch, plus the sticky device
// error word and the optional per-kernel timing.
#include <cstdarg>
#include <cstdio>
#include <algorithm>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "la_internal.cuh"

namespace la {

// ------------------------------------------------------------------ sticky error word
__device__ int g_error_word = 0;
#ifdef LA_DEBUG
__device__ unsigned int g_debug_site = 0;  // (file tag << 16) | line of the first failed index check
#endif

namespace {
thread_local std::string t_detail;

la_status fail(la_status st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_detail = buf;
    return st;
}

constexpr int kMaxDevices = 64;
int* g_err_ptr[kMaxDevices] = {};
int g_cc_ok[kMaxDevices] = {};  // 0 unknown, 1 sm_103, -1 other
std::mutex g_dev_mu;

int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    return dev;
}
}  // namespace

int* device_error_word() {
    int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> g(g_dev_mu);
    if (!g_err_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
        g_err_ptr[dev] = static_cast<int*>(p);
    }
    return g_err_ptr[dev];
}

// ------------------------------------------------------------------ timing
namespace {
struct Pending {
    const char* name;
    cudaEvent_t a, b;
};
struct Total {
    const char* name;
    int launches;
    double ms;
};
std::mutex g_t_mu;
bool g_timing = false;
std::vector<Pending> g_pending;
std::vector<Total> g_totals;
std::vector<cudaEvent_t> g_event_pool;
thread_local cudaEvent_t t_open = nullptr;

cudaEvent_t take_event() {
    if (!g_event_pool.empty()) {
        cudaEvent_t e = g_event_pool.back();
        g_event_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}

void drain_locked() {
    for (auto& p : g_pending) {
        float ms = 0.f;
        cudaEventSynchronize(p.b);
        cudaEventElapsedTime(&ms, p.a, p.b);
        Total* t = nullptr;
        for (auto& x : g_totals)
            if (strcmp(x.name, p.name) == 0) t = &x;
        if (!t) {
            g_totals.push_back({p.name, 0, 0.0});
            t = &g_totals.back();
        }
        t->launches += 1;
        t->ms += ms;
        g_event_pool.push_back(p.a);
        g_event_pool.push_back(p.b);
    }
    g_pending.clear();
}
}  // namespace

void launch_begin(const char* /*name*/, cudaStream_t st) {
    if (!g_timing) return;
    std::lock_guard<std::mutex> g(g_t_mu);
    t_open = take_event();
    cudaEventRecord(t_open, st);
}

cudaError_t launch_end(const char* name, cudaStream_t st) {
    cudaError_t err = cudaGetLastError();
    if (g_timing && t_open) {
        std::lock_guard<std::mutex> g(g_t_mu);
        cudaEvent_t b = take_event();
        cudaEventRecord(b, st);
        g_pending.push_back({name, t_open, b});
        t_open = nullptr;
        if (g_pending.size() > 4096) drain_locked();
    }
    return err;
}

// ------------------------------------------------------------------ planning
// CUDA-core kernels: one CTA per SM (about 215 KB of shared memory at D = 128),
// so aim for a few hundred CTAs.  Tensor-core kernels: one CTA per SM as well;
// the segment count is chosen so the CTAs fill whole waves of the GB300's 152
// SMs with equal chunk counts.  Both are fixed functions of the shape so that
// la_workspace_bytes stays device independent.
static constexpr int kSimtChunk = 64;
static constexpr int kTargetCtas = 304;
static constexpr int kTcChunk = 128;
static constexpr int kSms = 152;
static constexpr int kMaxWaves = 8;

// bf16 heads with Dk = Dv = 128, or 64 (padded to 128 on chip: the tile loads
// zero-fill the upper columns, phi keeps them zero and their stores are skipped).
// The non-causal forward and gradient run entirely on the tensor cores as well.
bool tc_supported(const la_shape& s, int op) {
    return s.dtype == LA_BF16 && s.Dk == s.Dv && (s.Dk == 128 || s.Dk == 64) &&
           (op == LA_OP_CAUSAL_FWD || op == LA_OP_CAUSAL_BWD || op == LA_OP_NONCAUSAL_FWD ||
            op == LA_OP_NONCAUSAL_BWD || op == LA_OP_RETENTION_FWD);
}

static void finish_plan(Plan& p, int P) {
    if (P < 1) P = 1;
    if (P > p.nchunks) P = p.nchunks;
    if (P < 1) P = 1;
    p.cps = (p.nchunks + P - 1) / P;
    p.P = (p.nchunks + p.cps - 1) / p.cps;
    if (p.P < 1) p.P = 1;
}

Plan make_plan(const la_shape& s, int op) {
    Plan p{};
    const int BH = s.B * s.H;
    p.tc = tc_supported(s, op);
    p.C = p.tc ? kTcChunk : kSimtChunk;
    p.sk = p.tc ? 128 : s.Dk;
    p.sv = p.tc ? 128 : s.Dv;
    p.nchunks = (s.N + p.C - 1) / p.C;
    if (!p.tc) {
        finish_plan(p, (kTargetCtas + BH - 1) / BH);
        return p;
    }
    // maximise useful chunk work / (waves * SMs * chunks per CTA)
    int best_P = 1;
    double best = -1.0;
    const int pmax = std::max(1, std::min(p.nchunks, kMaxWaves * kSms / std::max(BH, 1)));
    for (int P = 1; P <= pmax; ++P) {
        const int cps = (p.nchunks + P - 1) / P;
        const int Pr = (p.nchunks + cps - 1) / cps;
        const long long ctas = (long long)BH * Pr;
        const long long waves = (ctas + kSms - 1) / kSms;
        const double eff = (double)p.nchunks * BH / ((double)waves * kSms * cps);
        if (eff > best + 1e-9) {
            best = eff;
            best_P = P;
        }
    }
    finish_plan(p, best_P);
    return p;
}

static size_t align256(size_t x) { return (x + 255) / 256 * 256; }

WsLayout make_ws_layout(const la_shape& s, int op, const Plan& p) {
    WsLayout w{};
    const size_t BH = (size_t)s.B * s.H;
    // retention records hold S only (no normaliser)
    const size_t E = op == LA_OP_RETENTION_FWD ? (size_t)p.sk * p.sv : plan_state_elems(p);
    const size_t seg = align256(BH * p.P * E * sizeof(float));
    size_t off = 0;
    w.seg_states = off;
    off += seg;
    if (op == LA_OP_CAUSAL_BWD || op == LA_OP_NONCAUSAL_BWD) {
        w.seg_states2 = off;
        off += seg;
        w.den_g = off;
        off += align256(BH * (size_t)s.N * 2 * sizeof(float));
    }
    if (op == LA_OP_NONCAUSAL_FWD || op == LA_OP_NONCAUSAL_BWD) {
        w.totals = off;
        off += align256(BH * E * sizeof(float));
    }
    if (op == LA_OP_NONCAUSAL_BWD) {
        w.totals2 = off;
        off += align256(BH * E * sizeof(float));
    }
    if (op == LA_OP_CAUSAL_FWD && p.tc) {  // the one-launch forward's chained scan
        w.agg = off;
        off += seg;
        w.flags = off;
        off += align256((BH * p.P + 1) * sizeof(unsigned));
    }
    w.bytes = off;
    return w;
}

// ------------------------------------------------------------------ argument checks
namespace {

bool pow2_head(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }

la_status check_shape(const la_shape& s) {
    if (s.B < 0 || s.H < 0 || s.N < 0) return fail(LA_ERR_INVALID_ARG, "negative size B=%d H=%d N=%d", s.B, s.H, s.N);
    if (s.dtype != LA_F32 && s.dtype != LA_BF16) return fail(LA_ERR_INVALID_ARG, "bad dtype %d", s.dtype);
    if (s.Dk <= 0 || s.Dv <= 0) return fail(LA_ERR_INVALID_ARG, "bad head size Dk=%d Dv=%d", s.Dk, s.Dv);
    if (!pow2_head(s.Dk) || !pow2_head(s.Dv))
        return fail(LA_ERR_UNSUPPORTED, "head sizes must be 16, 32, 64 or 128 (Dk=%d Dv=%d)", s.Dk, s.Dv);
    if ((long long)s.B * s.H > 65535) return fail(LA_ERR_UNSUPPORTED, "B*H=%lld exceeds 65535", (long long)s.B * s.H);
    const double elems = (double)s.B * s.H * (double)s.N * (s.Dk > s.Dv ? s.Dk : s.Dv);
    if (elems >= 1099511627776.0) return fail(LA_ERR_INVALID_ARG, "problem too large");
    return LA_OK;
}

bool empty(const la_shape& s) { return s.B == 0 || s.H == 0 || s.N == 0; }

la_status check_device() {
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return fail(LA_ERR_CUDA, "no current CUDA device");
    int ok = g_cc_ok[dev];
    if (ok == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return fail(LA_ERR_CUDA, "cannot query device %d", dev);
        ok = (major == 10 && minor == 3) ? 1 : -1;
        g_cc_ok[dev] = ok;
        if (ok < 0) return fail(LA_ERR_UNSUPPORTED, "device %d is sm_%d%d; the library is compiled for sm_103a", dev, major, minor);
    }
    return ok > 0 ? LA_OK : fail(LA_ERR_UNSUPPORTED, "device is not sm_103");
}

// A tensor argument must be a 16-byte aligned (`align`) pointer to device (or
// managed) memory of the current device.  Host pointers are refused here,
// before any kernel could dereference them.
la_status check_ptr(const void* p, const char* what, uintptr_t align = 16) {
    if (!p) return fail(LA_ERR_INVALID_ARG, "%s is NULL", what);
    if (reinterpret_cast<uintptr_t>(p) & (align - 1))
        return fail(LA_ERR_INVALID_ARG, "%s is not %d-byte aligned", what, (int)align);
    cudaPointerAttributes attr;
    cudaError_t e = cudaPointerGetAttributes(&attr, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(LA_ERR_INVALID_ARG, "%s: not a CUDA pointer", what);
    }
    if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged)
        return fail(LA_ERR_INVALID_ARG, "%s is not device memory", what);
    if (attr.type == cudaMemoryTypeDevice && attr.device != current_device())
        return fail(LA_ERR_INVALID_ARG, "%s lives on device %d, not the current device", what, attr.device);
    return LA_OK;
}

la_status check_ws(void* ws, size_t ws_bytes, size_t need) {
    if (need == 0) return LA_OK;
    if (!ws) return fail(LA_ERR_WORKSPACE, "workspace is NULL (%zu bytes needed)", need);
    if (ws_bytes < need) return fail(LA_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", ws_bytes, need);
    return check_ptr(ws, "workspace") == LA_OK ? LA_OK : LA_ERR_INVALID_ARG;
}

la_status cuda_status(cudaError_t e, const char* where) {
    if (e == cudaSuccess) return LA_OK;
    return fail(LA_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

#define LA_TRY(expr)                        \
    do {                                    \
        la_status _st = (expr);             \
        if (_st != LA_OK) return _st;       \
    } while (0)

}  // namespace

// Argument checks for entry points defined in other translation units.
la_status checked_shape(const la_shape& s) { return check_shape(s); }
la_status checked_device() { return check_device(); }
la_status checked_ptr(const void* p, const char* what) { return check_ptr(p, what); }
la_status failed(la_status st, const char* msg) { return fail(st, "%s", msg); }
void clear_detail() { t_detail.clear(); }

}  // namespace la

using namespace la;

namespace {

// The two backward sweeps and the reverse scan between them; segS holds the
// exclusive prefix state of every segment.
static la_status causal_bwd_sweeps(const void* q, const void* k, const void* v, const void* dout, void* dq, void* dk,
                                   void* dv, const la_shape& s, const Plan& p, const float* segS, char* base,
                                   const WsLayout& w, cudaStream_t st) {
    float* segR = reinterpret_cast<float*>(base + w.seg_states2);
    float* den_g = reinterpret_cast<float*>(base + w.den_g);
    if (p.tc) {
        LA_TRY(cuda_status(tc_bwd_forward_sweep(q, k, v, dout, dq, segS, segR, den_g, s, p, st),
                           "backward forward sweep"));
        LA_TRY(cuda_status(scan_segments(segR, nullptr, s, p, SCAN_EXCLUSIVE_SUFFIX, st), "reverse scan"));
        LA_TRY(cuda_status(tc_bwd_reverse_sweep(q, k, v, dout, dk, dv, segR, den_g, s, p, st),
                           "backward reverse sweep"));
    } else {
        LA_TRY(cuda_status(simt_bwd_forward_sweep(q, k, v, dout, dq, segS, segR, den_g, s, p, st),
                           "backward forward sweep"));
        LA_TRY(cuda_status(scan_segments(segR, nullptr, s, p, SCAN_EXCLUSIVE_SUFFIX, st), "reverse scan"));
        LA_TRY(cuda_status(simt_bwd_reverse_sweep(q, k, v, dout, dk, dv, segR, den_g, s, p, st),
                           "backward reverse sweep"));
    }
    return LA_OK;
}

static la_status check_bwd_args(const void* q, const void* k, const void* v, const void* dout, const void* dq,
                                const void* dk, const void* dv) {
    LA_TRY(check_device());
    LA_TRY(check_ptr(q, "q"));
    LA_TRY(check_ptr(k, "k"));
    LA_TRY(check_ptr(v, "v"));
    LA_TRY(check_ptr(dout, "dout"));
    LA_TRY(check_ptr(dq, "dq"));
    LA_TRY(check_ptr(dk, "dk"));
    LA_TRY(check_ptr(dv, "dv"));
    return LA_OK;
}

// The causal forward.  one_launch selects the single-kernel form (segment sums, chained scan
// and outputs in one launch) where the tensor-core path runs; otherwise the segment sums, the
// scan and the output pass are three launches, which measure faster at every size timed (the
// chained scan's look-back reads the earlier segments' records one L2 round trip at a time
// whenever their inclusive prefixes are not yet published, as in a first wave).
static la_status causal_fwd_impl(const void* q, const void* k, const void* v, void* o, float* S_out, float* z_out,
                                 la_shape s, void* ws, size_t ws_bytes, la_stream_t stream,
                                 bool one_launch = false, bool withhold_first = false) {
    t_detail.clear();
    LA_TRY(check_shape(s));
    if (empty(s)) {
        if (!S_out || s.B == 0 || s.H == 0) return LA_OK;
        // no position: the state after it is zero
        LA_TRY(check_device());
        LA_TRY(check_ptr(S_out, "S"));
        LA_TRY(check_ptr(z_out, "z"));
        cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
        const size_t BH = (size_t)s.B * s.H;
        LA_TRY(cuda_status(cudaMemsetAsync(S_out, 0, BH * s.Dk * s.Dv * sizeof(float), st), "state clear"));
        LA_TRY(cuda_status(cudaMemsetAsync(z_out, 0, BH * s.Dk * sizeof(float), st), "state clear"));
        return LA_OK;
    }
    LA_TRY(check_device());
    LA_TRY(check_ptr(q, "q"));
    LA_TRY(check_ptr(k, "k"));
    LA_TRY(check_ptr(v, "v"));
    LA_TRY(check_ptr(o, "o"));
    if (S_out) {
        LA_TRY(check_ptr(S_out, "S"));
        LA_TRY(check_ptr(z_out, "z"));
    }
    const Plan p = make_plan(s, LA_OP_CAUSAL_FWD);
    const WsLayout w = make_ws_layout(s, LA_OP_CAUSAL_FWD, p);
    LA_TRY(check_ws(ws, ws_bytes, w.bytes));
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    char* base = static_cast<char*>(ws);
    float* seg = reinterpret_cast<float*>(base + w.seg_states);
    if (p.tc && one_launch) {  // one kernel: segment sums, chained scan and outputs (after a memset of its flags)
        LA_TRY(cuda_status(tc_causal_fwd_fused(q, k, v, o, seg, reinterpret_cast<float*>(base + w.agg),
                                               reinterpret_cast<unsigned*>(base + w.flags), S_out, z_out, s, p, st,
                                               withhold_first),
                           "causal forward"));
        return LA_OK;
    }
    const size_t seg_bytes = (size_t)s.B * s.H * p.P * plan_state_elems(p) * sizeof(float);
    if (p.P > 1 || S_out) {
        if (p.tc)
            LA_TRY(cuda_status(tc_causal_fwd(nullptr, k, v, nullptr, seg, s, p, false, st), "segment sums"));
        else
            LA_TRY(cuda_status(simt_segment_sums(k, v, seg, s, p, st), "segment sums"));
        if (S_out)
            LA_TRY(cuda_status(scan_segments_final_state(seg, S_out, z_out, s, p, st), "segment scan"));
        else
            LA_TRY(cuda_status(scan_segments(seg, nullptr, s, p, SCAN_EXCLUSIVE_PREFIX, st), "segment scan"));
    } else {
        LA_TRY(cuda_status(cudaMemsetAsync(seg, 0, seg_bytes, st), "state clear"));
    }
    if (p.tc)
        LA_TRY(cuda_status(tc_causal_fwd(q, k, v, o, seg, s, p, true, st), "causal forward"));
    else
        LA_TRY(cuda_status(simt_causal_fwd_out(q, k, v, o, seg, s, p, st), "causal forward"));
    return LA_OK;
}

}  // namespace

extern "C" {

size_t la_workspace_bytes(int op, la_shape s) {
    if (op < LA_OP_NONCAUSAL_FWD || op > LA_OP_RETENTION_FWD) return 0;
    if (check_shape(s) != LA_OK || empty(s)) return 0;
    const Plan p = make_plan(s, op);
    return make_ws_layout(s, op, p).bytes;
}

la_status la_noncausal_fwd(const void* q, const void* k, const void* v, void* o, la_shape s, void* ws,
                           size_t ws_bytes, la_stream_t stream) {
    t_detail.clear();
    LA_TRY(check_shape(s));
    if (empty(s)) return LA_OK;
    LA_TRY(check_device());
    LA_TRY(check_ptr(q, "q"));
    LA_TRY(check_ptr(k, "k"));
    LA_TRY(check_ptr(v, "v"));
    LA_TRY(check_ptr(o, "o"));
    const Plan p = make_plan(s, LA_OP_NONCAUSAL_FWD);
    const WsLayout w = make_ws_layout(s, LA_OP_NONCAUSAL_FWD, p);
    LA_TRY(check_ws(ws, ws_bytes, w.bytes));
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    float* seg = reinterpret_cast<float*>(static_cast<char*>(ws) + w.seg_states);
    float* tot = reinterpret_cast<float*>(static_cast<char*>(ws) + w.totals);
    if (p.tc) {  // padded records in, [BH][Dk*Dv + Dk] totals out
        LA_TRY(cuda_status(tc_causal_fwd(nullptr, k, v, nullptr, seg, s, p, false, st), "noncausal segment sums"));
        LA_TRY(cuda_status(scan_segments_unpadded_totals(seg, tot, s, p, st), "noncausal totals"));
    } else {
        LA_TRY(cuda_status(simt_segment_sums(k, v, seg, s, p, st), "noncausal segment sums"));
        LA_TRY(cuda_status(scan_segments(seg, tot, s, p, SCAN_TOTAL, st), "noncausal totals"));
    }
    if (p.tc)
        LA_TRY(cuda_status(tc_noncausal_apply(q, o, tot, s, p, st), "noncausal apply"));
    else
        LA_TRY(cuda_status(simt_noncausal_apply(q, o, tot, s, st), "noncausal apply"));
    return LA_OK;
}

// The causal forward; with S_out / z_out also the state after position N.

la_status la_causal_fwd(const void* q, const void* k, const void* v, void* o, la_shape s, void* ws, size_t ws_bytes,
                        la_stream_t stream) {
    return causal_fwd_impl(q, k, v, o, nullptr, nullptr, s, ws, ws_bytes, stream);
}

la_status la_causal_fwd_fused(const void* q, const void* k, const void* v, void* o, la_shape s, void* ws,
                              size_t ws_bytes, la_stream_t stream) {
    return causal_fwd_impl(q, k, v, o, nullptr, nullptr, s, ws, ws_bytes, stream, true);
}

la_status la_causal_fwd_with_state(const void* q, const void* k, const void* v, void* o, float* S, float* z,
                                   la_shape s, void* ws, size_t ws_bytes, la_stream_t stream) {
    if (!S || !z) {
        t_detail.clear();
        return fail(LA_ERR_INVALID_ARG, "S and z are required");
    }
    return causal_fwd_impl(q, k, v, o, S, z, s, ws, ws_bytes, stream);
}

la_status la_selftest_lookback_timeout(const void* q, const void* k, const void* v, void* o, la_shape s, void* ws,
                                       size_t ws_bytes, la_stream_t stream) {
    t_detail.clear();
    LA_TRY(check_shape(s));
    const Plan p = make_plan(s, LA_OP_CAUSAL_FWD);
    if (empty(s) || !p.tc || p.P < 2)
        return fail(LA_ERR_INVALID_ARG, "the look-back self-test needs a tensor-core shape with two or more segments "
                                        "(bf16, Dk = Dv = 64 or 128; this one has %d)", empty(s) ? 0 : p.P);
    return causal_fwd_impl(q, k, v, o, nullptr, nullptr, s, ws, ws_bytes, stream, true, true);
}

la_status la_causal_bwd(const void* q, const void* k, const void* v, const void* dout, void* dq, void* dk, void* dv,
                        la_shape s, void* ws, size_t ws_bytes, la_stream_t stream) {
    t_detail.clear();
    LA_TRY(check_shape(s));
    if (empty(s)) return LA_OK;
    LA_TRY(check_bwd_args(q, k, v, dout, dq, dk, dv));
    const Plan p = make_plan(s, LA_OP_CAUSAL_BWD);
    const WsLayout w = make_ws_layout(s, LA_OP_CAUSAL_BWD, p);
    LA_TRY(check_ws(ws, ws_bytes, w.bytes));
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    char* base = static_cast<char*>(ws);
    float* segS = reinterpret_cast<float*>(base + w.seg_states);
    const size_t seg_bytes = (size_t)s.B * s.H * p.P * plan_state_elems(p) * sizeof(float);
    if (p.P > 1) {
        if (p.tc)
            LA_TRY(cuda_status(tc_causal_fwd(nullptr, k, v, nullptr, segS, s, p, false, st), "segment sums"));
        else
            LA_TRY(cuda_status(simt_segment_sums(k, v, segS, s, p, st), "segment sums"));
        LA_TRY(cuda_status(scan_segments(segS, nullptr, s, p, SCAN_EXCLUSIVE_PREFIX, st), "segment scan"));
    } else {
        LA_TRY(cuda_status(cudaMemsetAsync(segS, 0, seg_bytes, st), "state clear"));
    }
    return causal_bwd_sweeps(q, k, v, dout, dq, dk, dv, s, p, segS, base, w, st);
}

la_status la_causal_bwd_after_fwd(const void* q, const void* k, const void* v, const void* dout, void* dq, void* dk,
                                  void* dv, la_shape s, const void* fwd_ws, size_t fwd_ws_bytes, void* ws,
                                  size_t ws_bytes, la_stream_t stream) {
    t_detail.clear();
    LA_TRY(check_shape(s));
    if (empty(s)) return LA_OK;
    LA_TRY(check_bwd_args(q, k, v, dout, dq, dk, dv));
    const Plan p = make_plan(s, LA_OP_CAUSAL_BWD);
    const Plan pf = make_plan(s, LA_OP_CAUSAL_FWD);
    if (pf.P != p.P || pf.C != p.C)  // the forward's segments are the backward's (same planner)
        return fail(LA_ERR_UNSUPPORTED, "forward and backward segmentations differ (P %d vs %d)", pf.P, p.P);
    const WsLayout wf = make_ws_layout(s, LA_OP_CAUSAL_FWD, pf);
    if (fwd_ws_bytes < wf.bytes)
        return fail(LA_ERR_WORKSPACE, "forward workspace of %zu bytes, the forward needs %zu", fwd_ws_bytes, wf.bytes);
    LA_TRY(check_ptr(fwd_ws, "fwd_ws"));
    const WsLayout w = make_ws_layout(s, LA_OP_CAUSAL_BWD, p);
    LA_TRY(check_ws(ws, ws_bytes, w.bytes));
    const float* segS = reinterpret_cast<const float*>(static_cast<const char*>(fwd_ws) + wf.seg_states);
    return causal_bwd_sweeps(q, k, v, dout, dq, dk, dv, s, p, segS, static_cast<char*>(ws), w,
                             reinterpret_cast<cudaStream_t>(stream));
}

la_status la_noncausal_bwd(const void* q, const void* k, const void* v, const void* dout, void* dq, void* dk, void* dv,
                           la_shape s, void* ws, size_t ws_bytes, la_stream_t stream) {
    t_detail.clear();
    LA_TRY(check_shape(s));
    if (empty(s)) return LA_OK;
    LA_TRY(check_bwd_args(q, k, v, dout, dq, dk, dv));
    const Plan p = make_plan(s, LA_OP_NONCAUSAL_BWD);
    const WsLayout w = make_ws_layout(s, LA_OP_NONCAUSAL_BWD, p);
    LA_TRY(check_ws(ws, ws_bytes, w.bytes));
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    char* base = static_cast<char*>(ws);
    float* seg = reinterpret_cast<float*>(base + w.seg_states);
    float* segR = reinterpret_cast<float*>(base + w.seg_states2);
    float* den_g = reinterpret_cast<float*>(base + w.den_g);
    float* totS = reinterpret_cast<float*>(base + w.totals);
    float* totR = reinterpret_cast<float*>(base + w.totals2);
    if (p.tc) {  // padded (S, z) and (R, r) records throughout; phi(K) split hi + lo in the sums
        LA_TRY(cuda_status(tc_causal_fwd(nullptr, k, v, nullptr, seg, s, p, false, st, true),
                           "noncausal segment sums"));
        LA_TRY(cuda_status(scan_segments(seg, totS, s, p, SCAN_TOTAL, st), "noncausal totals"));
        LA_TRY(cuda_status(tc_noncausal_bwd_query(q, dout, dq, totS, segR, s, p, st),
                           "noncausal backward, query pass"));
        LA_TRY(cuda_status(scan_segments(segR, totR, s, p, SCAN_TOTAL, st), "noncausal reverse totals"));
        LA_TRY(cuda_status(tc_noncausal_bwd_key(k, v, dk, dv, totR, s, p, st), "noncausal backward, key pass"));
        return LA_OK;
    }
    LA_TRY(cuda_status(simt_segment_sums(k, v, seg, s, p, st), "noncausal segment sums"));
    LA_TRY(cuda_status(scan_segments(seg, totS, s, p, SCAN_TOTAL, st), "noncausal totals"));
    LA_TRY(cuda_status(simt_bwd_forward_sweep(q, k, v, dout, dq, totS, segR, den_g, s, p, st, false),
                       "noncausal backward, query pass"));
    LA_TRY(cuda_status(scan_segments(segR, totR, s, p, SCAN_TOTAL, st), "noncausal reverse totals"));
    LA_TRY(cuda_status(simt_bwd_reverse_sweep(q, k, v, dout, dk, dv, totR, den_g, s, p, st, false),
                       "noncausal backward, key pass"));
    return LA_OK;
}

la_status la_recurrent_step(const void* q, const void* k, const void* v, float* S, float* z, void* out, la_shape s,
                            la_stream_t stream) {
    t_detail.clear();
    la_shape s1 = s;
    s1.N = 1;  // N is ignored by the step
    LA_TRY(check_shape(s1));
    if (empty(s1)) return LA_OK;
    LA_TRY(check_device());
    LA_TRY(check_ptr(q, "q"));
    LA_TRY(check_ptr(k, "k"));
    LA_TRY(check_ptr(v, "v"));
    LA_TRY(check_ptr(S, "S"));
    LA_TRY(check_ptr(z, "z"));
    LA_TRY(check_ptr(out, "out"));
    LA_TRY(cuda_status(la::recurrent_step(q, k, v, S, z, out, s1, reinterpret_cast<cudaStream_t>(stream)),
                       "recurrent step"));
    return LA_OK;
}

la_status la_retention_fwd(const void* q, const void* k, const void* v, const float* gamma, void* o, float* S,
                           la_shape s, void* ws, size_t ws_bytes, la_stream_t stream) {
    t_detail.clear();
    LA_TRY(check_shape(s));
    if (s.B == 0 || s.H == 0) return LA_OK;
    LA_TRY(check_device());
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (s.N == 0) {  // no position: the state after it is zero
        if (!S) return LA_OK;
        LA_TRY(check_ptr(S, "S"));
        LA_TRY(cuda_status(cudaMemsetAsync(S, 0, (size_t)s.B * s.H * s.Dk * s.Dv * sizeof(float), st), "state clear"));
        return LA_OK;
    }
    LA_TRY(check_ptr(q, "q"));
    LA_TRY(check_ptr(k, "k"));
    LA_TRY(check_ptr(v, "v"));
    LA_TRY(check_ptr(o, "o"));
    LA_TRY(check_ptr(gamma, "gamma", 4));
    if (S) LA_TRY(check_ptr(S, "S"));
    const Plan p = make_plan(s, LA_OP_RETENTION_FWD);
    const WsLayout w = make_ws_layout(s, LA_OP_RETENTION_FWD, p);
    LA_TRY(check_ws(ws, ws_bytes, w.bytes));
    float* seg = reinterpret_cast<float*>(static_cast<char*>(ws) + w.seg_states);
    if (p.P > 1 || S) {
        if (p.tc)
            LA_TRY(cuda_status(tc_retention_fwd(nullptr, k, v, gamma, nullptr, seg, s, p, false, st),
                               "retention segment sums"));
        else
            LA_TRY(cuda_status(retention_segment_sums(k, v, gamma, seg, s, p, st), "retention segment sums"));
        LA_TRY(cuda_status(retention_scan(seg, S, gamma, s, p, st), "retention segment scan"));
    } else {
        const size_t seg_bytes = (size_t)s.B * s.H * p.sk * p.sv * sizeof(float);
        LA_TRY(cuda_status(cudaMemsetAsync(seg, 0, seg_bytes, st), "state clear"));
    }
    if (p.tc)
        LA_TRY(cuda_status(tc_retention_fwd(q, k, v, gamma, o, seg, s, p, true, st), "retention forward"));
    else
        LA_TRY(cuda_status(retention_out(q, k, v, gamma, o, seg, s, p, st), "retention forward"));
    return LA_OK;
}

la_status la_retention_step(const void* q, const void* k, const void* v, const float* gamma, float* S, void* out,
                            la_shape s, la_stream_t stream) {
    t_detail.clear();
    la_shape s1 = s;
    s1.N = 1;  // N is ignored by the step
    LA_TRY(check_shape(s1));
    if (empty(s1)) return LA_OK;
    LA_TRY(check_device());
    LA_TRY(check_ptr(q, "q"));
    LA_TRY(check_ptr(k, "k"));
    LA_TRY(check_ptr(v, "v"));
    LA_TRY(check_ptr(gamma, "gamma", 4));
    LA_TRY(check_ptr(S, "S"));
    LA_TRY(check_ptr(out, "out"));
    LA_TRY(cuda_status(la::retention_step(q, k, v, gamma, S, out, s1, reinterpret_cast<cudaStream_t>(stream)),
                       "retention step"));
    return LA_OK;
}

la_status la_last_error(void) {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_error_word, sizeof(int)) != cudaSuccess)
        return fail(LA_ERR_CUDA, "cannot read the device error word");
#ifdef LA_DEBUG
    if (v == LA_ERR_BOUNDS) {
        unsigned site = 0;
        if (cudaMemcpyFromSymbol(&site, g_debug_site, sizeof(site)) == cudaSuccess) {
            static const char* const kFiles[] = {"api.cu", "decode.cu", "host_step.cu", "noalloc.cu", "retention.cu",
                                                 "selftest.cu", "simt_kernels.cu", "tc_apply.cu", "tc_bwd.cu",
                                                 "tc_fwd.cu", "tc_noncausal_bwd.cu", "tc_retention.cu",
                                                 "la_internal.cuh", "simt_common.cuh", "tc_common.cuh", "sm100.cuh"};
            const char* file = "unknown file";
            for (const char* f : kFiles)
                if (dbg::file_tag(f) == (site >> 16)) file = f;
            fail(LA_ERR_BOUNDS, "index check failed at %s:%u", file, site & 0xFFFFu);
        }
    }
#endif
    return static_cast<la_status>(v);
}

la_status la_clear_error(void) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_error_word, &zero, sizeof(int)) != cudaSuccess)
        return fail(LA_ERR_CUDA, "cannot clear the device error word");
#ifdef LA_DEBUG
    const unsigned zs = 0;
    if (cudaMemcpyToSymbol(g_debug_site, &zs, sizeof(zs)) != cudaSuccess)
        return fail(LA_ERR_CUDA, "cannot clear the device error site");
#endif
    return LA_OK;
}

const char* la_status_string(la_status st) {
    switch (st) {
        case LA_OK: return "LA_OK";
        case LA_ERR_INVALID_ARG: return "LA_ERR_INVALID_ARG: invalid argument";
        case LA_ERR_UNSUPPORTED: return "LA_ERR_UNSUPPORTED: unsupported size or device";
        case LA_ERR_WORKSPACE: return "LA_ERR_WORKSPACE: workspace missing or too small";
        case LA_ERR_CUDA: return "LA_ERR_CUDA: CUDA runtime or launch failure";
        case LA_ERR_TIMEOUT: return "LA_ERR_TIMEOUT: a bounded device wait ran out";
        case LA_ERR_BOUNDS: return "LA_ERR_BOUNDS: a device-side index check of the debug build failed";
    }
    return "unknown la_status";
}

const char* la_error_detail(void) { return t_detail.c_str(); }

#ifdef LA_DEBUG
const char* la_version(void) { return "0.1.1-debug"; }
#else
const char* la_version(void) { return "0.1.1"; }
#endif

la_status la_timing_enable(int on) {
    std::lock_guard<std::mutex> g(g_t_mu);
    g_timing = on != 0;
    return LA_OK;
}

la_status la_timing_reset(void) {
    std::lock_guard<std::mutex> g(g_t_mu);
    drain_locked();
    g_totals.clear();
    return LA_OK;
}

int la_timing_read(la_kernel_time* out, int max) {
    std::lock_guard<std::mutex> g(g_t_mu);
    drain_locked();
    const int n = (int)g_totals.size();
    for (int i = 0; i < n && i < max && out; ++i) out[i] = {g_totals[i].name, g_totals[i].launches, g_totals[i].ms};
    return n;
}

}  // extern "C"
