// la_internal.cuh -- definitions shared by the libla translation units.
//
// Work decomposition used by every chunked kernel.  A head's N positions are
// cut into chunks of C positions (the last one may be short and is masked);
// consecutive chunks are grouped into P segments of `cps` chunks.  One CTA owns
// one (segment, head) pair and walks its chunks in order, carrying the state
// (S, z) chunk to chunk on chip.  The states that cross segment boundaries are
// produced by a per-segment reduction kernel and an exclusive scan over the P
// segments (the prefix-sum structure of the causal form: "Transformers은 RNN이다"
// digest, Insights / Prefix-sum 병렬성; itwiki 계산 형태 비교, chunked row).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "la.h"

namespace la {

// Elements of one (S, z) state record in the workspace: Dk*Dv for S then Dk for z.
inline __host__ __device__ size_t state_elems(int Dk, int Dv) { return (size_t)Dk * Dv + Dk; }

struct Plan {
    int C;        // chunk length (positions)
    int nchunks;  // ceil(N / C)
    int P;        // segments per head
    int cps;      // chunks per segment
    bool tc;      // tensor-core (tcgen05) kernels, else CUDA-core kernels
    int sk, sv;   // dimensions of the state records (Dk, Dv; 128 on the tensor-core path, which
                  // pads a 64-wide head to 128 on chip)
};
inline size_t plan_state_elems(const Plan& p) { return state_elems(p.sk, p.sv); }

// Byte offsets of the workspace regions of one call (all 256-byte aligned).
struct WsLayout {
    size_t seg_states;   // [BH][P][E] fp32: per-segment S/z sums, then scanned in place
    size_t seg_states2;  // [BH][P][E] fp32: backward reverse-state sums (R, r)
    size_t totals;       // [BH][E] fp32: non-causal totals (S, z)
    size_t totals2;      // [BH][E] fp32: non-causal backward totals (R, r)
    size_t den_g;        // [BH][N][2] fp32: backward per-position den and g
    size_t agg;          // [BH][P][E] fp32: the one-launch causal forward's per-segment own sums
    size_t flags;        // [BH][P] + 1 uint32: their publication flags and the ticket counter
    size_t bytes;        // total
};

Plan make_plan(const la_shape& s, int op);
WsLayout make_ws_layout(const la_shape& s, int op, const Plan& p);

// ------------------------------------------------------------------ device helpers
template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// 2^x with the ex2.approx instruction (relative error about 2^-22).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// phi(x) = elu(x) + 1 (alpha = 1): x + 1 for x > 0, exp(x) = 2^(x log2 e) for x <= 0.
// Branch-free and select-free: max(x, 0) + 2^(min(x, 0) log2 e) is x + 2^0 for
// x > 0 and 0 + e^x otherwise.
__device__ __forceinline__ float phi_f(float x) {
    return fmaxf(x, 0.f) + ex2_approx(fminf(x, 0.f) * 1.4426950408889634f);
}
// phi'(x) = 1 for x > 0, exp(x) otherwise; equal to min(1, phi(x)).
__device__ __forceinline__ float dphi_from_phi(float p) { return fminf(p, 1.f); }

// ------------------------------------------------------------------ debug-build index checks
// LA_DCHECK(cond) is `true` in the regular build (the condition is not even
// evaluated).  In the debug build (compiled with -DLA_DEBUG and relocatable
// device code, so every translation unit sees the one sticky error word) it
// evaluates the condition; if it is false it records LA_ERR_BOUNDS in the
// sticky word and the site (a 16-bit tag of the source file's name and the
// line) in g_debug_site, both first-failure-wins, and yields false so that the
// caller skips the access.  Nothing traps.
namespace dbg {
constexpr uint32_t file_tag(const char* path) {  // FNV-1a of the base name, 16 bits
    const char* b = path;
    for (const char* c = path; *c; ++c)
        if (*c == '/') b = c + 1;
    uint32_t h = 2166136261u;
    for (; *b; ++b) h = (h ^ (uint32_t)(unsigned char)*b) * 16777619u;
    return (h ^ (h >> 16)) & 0xFFFFu;
}
template <uint32_t V> struct Const { static constexpr uint32_t value = V; };
}  // namespace dbg

#ifdef LA_DEBUG
extern __device__ int g_error_word;
extern __device__ unsigned int g_debug_site;
namespace dbg {
__device__ __forceinline__ bool check(bool ok, uint32_t tag, uint32_t line) {
    if (!ok) {
        atomicCAS(&g_error_word, 0, (int)LA_ERR_BOUNDS);
        atomicCAS(&g_debug_site, 0u, (tag << 16) | (line & 0xFFFFu));
    }
    return ok;
}
}  // namespace dbg
#define LA_DCHECK(cond) (::la::dbg::check((cond), ::la::dbg::Const<::la::dbg::file_tag(__FILE__)>::value, __LINE__))
#else
namespace dbg {
__host__ __device__ constexpr bool pass() { return true; }
}  // namespace dbg
#define LA_DCHECK(cond) (::la::dbg::pass())
#endif

// ------------------------------------------------------------------ programmatic dependent launch
// Kernels launched with launch_pdl may be scheduled while the previous kernel in
// the stream finishes its last blocks.  Each such kernel calls pdl_enter() after its
// prologue (barrier init, TMEM allocation, tensor-map prefetch) and before any
// global-memory access: it waits until the previous grid has completed and its
// writes are visible, and lets the next kernel be scheduled (which happens once
// every block of this grid has reached this point, so a waiting dependent block
// never holds an SM that a block of this grid still needs).
__device__ __forceinline__ void pdl_enter() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// ------------------------------------------------------------------ launch bookkeeping
// Every launch goes through launch_begin/launch_end so the optional per-kernel
// timing (la_timing_enable) can bracket it with events on the launch stream.
void launch_begin(const char* name, cudaStream_t st);
cudaError_t launch_end(const char* name, cudaStream_t st);

// Device address of the sticky error word (set once per device).
int* device_error_word();

// ------------------------------------------------------------------ host launchers
// CUDA-core (SIMT) kernels, any dtype, Dk/Dv multiples of 16 up to 128.
cudaError_t simt_segment_sums(const void* k, const void* v, float* seg, const la_shape& s, const Plan& p,
                              cudaStream_t st);
cudaError_t scan_segments(float* seg, float* totals, const la_shape& s, const Plan& p, int mode,
                          cudaStream_t st);
// The sum over all segments as [BH][Dk*Dv + Dk] records without padding (seg unchanged).
cudaError_t scan_segments_unpadded_totals(float* seg, float* totals, const la_shape& s, const Plan& p,
                                          cudaStream_t st);
// Exclusive prefix in place, and the sum over all segments (the state after
// position N) split into S_out [BH][Dk][Dv] and z_out [BH][Dk].
cudaError_t scan_segments_final_state(float* seg, float* S_out, float* z_out, const la_shape& s, const Plan& p,
                                      cudaStream_t st);
cudaError_t simt_causal_fwd_out(const void* q, const void* k, const void* v, void* o, const float* seg,
                                const la_shape& s, const Plan& p, cudaStream_t st);
cudaError_t simt_noncausal_apply(const void* q, void* o, const float* totals, const la_shape& s,
                                 cudaStream_t st);
cudaError_t simt_bwd_forward_sweep(const void* q, const void* k, const void* v, const void* dout,
                                   void* dq, const float* seg_S, float* seg_R, float* den_g,
                                   const la_shape& s, const Plan& p, cudaStream_t st, bool causal = true);
cudaError_t simt_bwd_reverse_sweep(const void* q, const void* k, const void* v, const void* dout,
                                   void* dk, void* dv, const float* seg_R, const float* den_g,
                                   const la_shape& s, const Plan& p, cudaStream_t st, bool causal = true);
cudaError_t recurrent_step(const void* q, const void* k, const void* v, float* S, float* z, void* out,
                           const la_shape& s, cudaStream_t st);

// Tensor-core (tcgen05) kernels: bf16, Dk = Dv = 128 (or 64, zero-padded to 128 on chip), C = 128.
// out_pass = false: per-segment sums (S, z) into seg; true: outputs from the scanned prefixes.
// split_k (sums only): phi(K) enters the sums as hi + lo bf16 parts (the non-causal gradient).
cudaError_t tc_causal_fwd(const void* q, const void* k, const void* v, void* o, float* seg, const la_shape& s,
                          const Plan& p, bool out_pass, cudaStream_t st, bool split_k = false);
// The causal forward in one kernel launch (after a memset of the flags): each CTA
// forms and publishes its segment's own sums, adds the earlier segments' in order
// (a chained scan with bounded waits), writes that exclusive prefix to seg and runs
// the output pass; with S_out / z_out also the state after position N.
// withhold_first (tests only): segment 0 of head 0 never publishes, so the later
// segments of that head time out with LA_ERR_TIMEOUT.
cudaError_t tc_causal_fwd_fused(const void* q, const void* k, const void* v, void* o, float* seg, float* agg,
                                unsigned* flags, float* S_out, float* z_out, const la_shape& s, const Plan& p,
                                cudaStream_t st, bool withhold_first = false);
cudaError_t tc_bwd_forward_sweep(const void* q, const void* k, const void* v, const void* dout, void* dq,
                                 const float* seg_S, float* seg_R, float* den_g, const la_shape& s, const Plan& p,
                                 cudaStream_t st);
cudaError_t tc_bwd_reverse_sweep(const void* q, const void* k, const void* v, const void* dout, void* dk, void* dv,
                                 const float* seg_R, const float* den_g, const la_shape& s, const Plan& p,
                                 cudaStream_t st);
// Retention (constant decay per head).  Segment records are sk*sv floats (S only,
// no z).  CUDA-core kernels for any dtype and head size; the scan serves both paths.
cudaError_t retention_segment_sums(const void* k, const void* v, const float* gamma, float* seg, const la_shape& s,
                                   const Plan& p, cudaStream_t st);
cudaError_t retention_scan(float* seg, float* S_out, const float* gamma, const la_shape& s, const Plan& p,
                           cudaStream_t st);
cudaError_t retention_out(const void* q, const void* k, const void* v, const float* gamma, void* o, const float* seg,
                          const la_shape& s, const Plan& p, cudaStream_t st);
// Tensor-core retention (bf16, Dk = Dv = 128 or 64, C = 128): out_pass = false forms
// the segments' local states in seg, true the outputs from the scanned prefixes.
cudaError_t tc_retention_fwd(const void* q, const void* k, const void* v, const float* gamma, void* o, float* seg,
                             const la_shape& s, const Plan& p, bool out_pass, cudaStream_t st);
cudaError_t retention_step(const void* q, const void* k, const void* v, const float* gamma, float* S, void* out,
                           const la_shape& s, cudaStream_t st);
// Tensor-core non-causal apply (bf16, Dk = Dv = 128 or 64): o from the head totals
// [BH][Dk*Dv + Dk] (unpadded S then z), over the chunks of Plan p.
cudaError_t tc_noncausal_apply(const void* q, void* o, const float* totals, const la_shape& s, const Plan& p,
                               cudaStream_t st);
// Tensor-core non-causal gradient (bf16, Dk = Dv = 128 or 64): the query pass writes dq
// and the segments' (R, r) sums (padded records) from the padded totals (S, z); the key
// pass writes dk, dv from the padded totals (R, r).
cudaError_t tc_noncausal_bwd_query(const void* q, const void* dout, void* dq, const float* totS, float* seg_R,
                                   const la_shape& s, const Plan& p, cudaStream_t st);
cudaError_t tc_noncausal_bwd_key(const void* k, const void* v, void* dk, void* dv, const float* totR,
                                 const la_shape& s, const Plan& p, cudaStream_t st);
bool tc_supported(const la_shape& s, int op);

enum ScanMode { SCAN_EXCLUSIVE_PREFIX = 0, SCAN_EXCLUSIVE_SUFFIX = 1, SCAN_TOTAL = 2 };

}  // namespace la
