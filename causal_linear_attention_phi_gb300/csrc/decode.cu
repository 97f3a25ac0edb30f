// decode.cu -- one recurrent step for every head:
//   S <- S + phi(k) v^T,  z <- z + phi(k),  out = phi(q)^T S / phi(q)^T z
// (state updated first, then read: the diagonal term j = i is included).
// "Transformers은 RNN이다" digest, 핵심 구성요소 4 (RNN view); velog review 3.6;
// itwiki 인과 마스킹과 순환형.
//
// The step is bound by memory traffic: S (fp32, Dk x Dv per head) is read and
// written once, everything else is O(Dk + Dv) per head.  One warp owns one head.
// S rows are moved as float4: a row of Dv floats is Dv/4 vectors, so a warp
// instruction covers (32 / (Dv/4)) consecutive rows when Dv < 128, i.e. one
// contiguous, fully coalesced span of S per instruction.  Each lane keeps its
// four v values and four partial numerators in registers; the partial
// numerators of lanes that share a column group are combined with shuffles.
#include "la_internal.cuh"

namespace la {
namespace {

constexpr int kWarpsPerBlock = 2;

template <typename T>
__device__ __forceinline__ float4 load4(const T* p);
template <>
__device__ __forceinline__ float4 load4<float>(const float* p) {
    return *reinterpret_cast<const float4*>(p);
}
template <>
__device__ __forceinline__ float4 load4<__nv_bfloat16>(const __nv_bfloat16* p) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(p);
    float2 a = __bfloat1622float2(h[0]), b = __bfloat1622float2(h[1]);
    return make_float4(a.x, a.y, b.x, b.y);
}

template <typename T>
__device__ __forceinline__ void store4(T* p, float4 x);
template <>
__device__ __forceinline__ void store4<float>(float* p, float4 x) {
    *reinterpret_cast<float4*>(p) = x;
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* p, float4 x) {
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(p);
    h[0] = __floats2bfloat162_rn(x.x, x.y);
    h[1] = __floats2bfloat162_rn(x.z, x.w);
}

template <typename T>
__global__ void __launch_bounds__(32 * kWarpsPerBlock)
recurrent_step_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                      float* __restrict__ S, float* __restrict__ z, T* __restrict__ out, int BH, int Dk, int Dv) {
    __shared__ float qk_s[kWarpsPerBlock][2][128];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.x * kWarpsPerBlock + warp;
    if (h >= BH) return;  // whole warp leaves together

    const T* qh = q + (size_t)h * Dk;
    const T* kh = k + (size_t)h * Dk;
    float* zh = z + (size_t)h * Dk;
    // phi(q), phi(k) into shared memory; z update and phi(q).z on the way
    float den = 0.f;
    for (int d = lane; d < Dk; d += 32) {
        const float qt = phi_f(to_f32(qh[d]));
        const float kt = phi_f(to_f32(kh[d]));
        qk_s[warp][0][d] = qt;
        qk_s[warp][1][d] = kt;
        const float zn = zh[d] + kt;
        zh[d] = zn;
        den = fmaf(qt, zn, den);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    __syncwarp();

    const int ncol4 = Dv >> 2;                    // float4 columns per row (4..32)
    const int cols = ncol4 < 32 ? ncol4 : 32;     // lanes across a row
    const int rows_per_iter = 32 / cols;          // rows covered by one warp instruction
    const int c4 = lane % cols, rsub = lane / cols;
    const int npass = ncol4 / cols;               // column passes (1 unless Dv > 128)
    float* Sh = S + (size_t)h * Dk * Dv;

    for (int pass = 0; pass < npass; ++pass) {
        const int col = (pass * cols + c4) * 4;
        const float4 vv = load4<T>(v + (size_t)h * Dv + col);
        float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
        for (int d = rsub; d < Dk; d += rows_per_iter) {
            float4* sp = reinterpret_cast<float4*>(Sh + (size_t)d * Dv + col);
            float4 s = *sp;
            const float kt = qk_s[warp][1][d], qt = qk_s[warp][0][d];
            s.x = fmaf(kt, vv.x, s.x);
            s.y = fmaf(kt, vv.y, s.y);
            s.z = fmaf(kt, vv.z, s.z);
            s.w = fmaf(kt, vv.w, s.w);
            *sp = s;
            num.x = fmaf(qt, s.x, num.x);
            num.y = fmaf(qt, s.y, num.y);
            num.z = fmaf(qt, s.z, num.z);
            num.w = fmaf(qt, s.w, num.w);
        }
        // combine lanes with the same column group (they differ in the row bits)
        for (int o = cols; o < 32; o <<= 1) {
            num.x += __shfl_xor_sync(0xffffffffu, num.x, o);
            num.y += __shfl_xor_sync(0xffffffffu, num.y, o);
            num.z += __shfl_xor_sync(0xffffffffu, num.z, o);
            num.w += __shfl_xor_sync(0xffffffffu, num.w, o);
        }
        if (rsub == 0) {
            const float inv = 1.f / den;
            store4<T>(out + (size_t)h * Dv + col, make_float4(num.x * inv, num.y * inv, num.z * inv, num.w * inv));
        }
    }
}

// Fast path for heads with Dk, Dv <= 64: one warp per head, every global load
// of the step issued before any arithmetic (one memory round trip), S held in
// registers as float4s.  Lane layout for S: COLS = Dv/4 lanes across a row,
// RPI = 32/COLS rows per warp instruction, ROWS = Dk/RPI rows per lane.  q, k
// and z are read once, element d by lane d % 32 (coalesced); phi is applied
// there once and the value of row d reaches the lanes that update row d by a
// shuffle.  Launched with programmatic stream serialization: the grid may be
// scheduled while the previous kernel in the stream drains, and it waits
// (griddepcontrol.wait) before touching any global memory, so the stream
// order seen by memory is unchanged.
template <typename T, int DK, int DV>
__global__ void __launch_bounds__(32 * kWarpsPerBlock)
recurrent_step_small_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                            float* __restrict__ S, float* __restrict__ z, T* __restrict__ out, int BH) {
    constexpr int COLS = DV / 4;
    constexpr int RPI = 32 / COLS;
    constexpr int ROWS = DK / RPI;
    constexpr int ZPL = (DK + 31) / 32;  // q, k, z entries per lane
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.x * kWarpsPerBlock + warp;
    if (h >= BH) return;
    const int c4 = lane % COLS, rsub = lane / COLS;
    const int col = c4 * 4;
    float* Sh = S + (size_t)h * DK * DV;
    // ---- all loads first
    float4 s[ROWS];
#pragma unroll
    for (int x = 0; x < ROWS; ++x)
        s[x] = *reinterpret_cast<const float4*>(Sh + (size_t)(rsub + RPI * x) * DV + col);
    const float4 vv = load4<T>(v + (size_t)h * DV + col);
    float zq[ZPL], zk[ZPL], zz[ZPL];
#pragma unroll
    for (int y = 0; y < ZPL; ++y) {
        const int d = lane + 32 * y;
        const bool in = d < DK;
        zz[y] = in ? z[(size_t)h * DK + d] : 0.f;
        zk[y] = in ? to_f32(k[(size_t)h * DK + d]) : 0.f;
        zq[y] = in ? to_f32(q[(size_t)h * DK + d]) : 0.f;
    }
    // ---- phi once per element, z update and phi(q).z
    float den = 0.f;
#pragma unroll
    for (int y = 0; y < ZPL; ++y) {
        const int d = lane + 32 * y;
        zk[y] = phi_f(zk[y]);
        zq[y] = phi_f(zq[y]);
        if (d < DK) {
            const float zn = zz[y] + zk[y];
            z[(size_t)h * DK + d] = zn;
            den = fmaf(zq[y], zn, den);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    // ---- S update and phi(q)^T S; row d's phi(k), phi(q) come from lane d % 32
    float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int x = 0; x < ROWS; ++x) {
        const int d = rsub + RPI * x;
        float a = __shfl_sync(0xffffffffu, zk[0], d & 31), b = __shfl_sync(0xffffffffu, zq[0], d & 31);
        if (ZPL > 1) {
            const float a1 = __shfl_sync(0xffffffffu, zk[ZPL - 1], d & 31);
            const float b1 = __shfl_sync(0xffffffffu, zq[ZPL - 1], d & 31);
            if (d >= 32) {
                a = a1;
                b = b1;
            }
        }
        float4 t = s[x];
        t.x = fmaf(a, vv.x, t.x);
        t.y = fmaf(a, vv.y, t.y);
        t.z = fmaf(a, vv.z, t.z);
        t.w = fmaf(a, vv.w, t.w);
        *reinterpret_cast<float4*>(Sh + (size_t)d * DV + col) = t;
        num.x = fmaf(b, t.x, num.x);
        num.y = fmaf(b, t.y, num.y);
        num.z = fmaf(b, t.z, num.z);
        num.w = fmaf(b, t.w, num.w);
    }
#pragma unroll
    for (int o = COLS; o < 32; o <<= 1) {
        num.x += __shfl_xor_sync(0xffffffffu, num.x, o);
        num.y += __shfl_xor_sync(0xffffffffu, num.y, o);
        num.z += __shfl_xor_sync(0xffffffffu, num.z, o);
        num.w += __shfl_xor_sync(0xffffffffu, num.w, o);
    }
    if (rsub == 0) {
        const float inv = 1.f / den;
        store4<T>(out + (size_t)h * DV + col, make_float4(num.x * inv, num.y * inv, num.z * inv, num.w * inv));
    }
}

template <typename T, int DK, int DV>
cudaError_t launch_small(const void* q, const void* k, const void* v, float* S, float* z, void* out, int BH,
                         cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((BH + kWarpsPerBlock - 1) / kWarpsPerBlock));
    cfg.blockDim = dim3(32 * kWarpsPerBlock);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, recurrent_step_small_kernel<T, DK, DV>, (const T*)q, (const T*)k, (const T*)v, S,
                              z, (T*)out, BH);
}

template <typename T>
cudaError_t dispatch_small(const void* q, const void* k, const void* v, float* S, float* z, void* out, int BH,
                           int Dk, int Dv, cudaStream_t st, bool* handled) {
    *handled = true;
#define LA_SMALL(a, b) \
    if (Dk == a && Dv == b) return launch_small<T, a, b>(q, k, v, S, z, out, BH, st);
    LA_SMALL(16, 16) LA_SMALL(16, 32) LA_SMALL(16, 64) LA_SMALL(32, 16) LA_SMALL(32, 32) LA_SMALL(32, 64)
    LA_SMALL(64, 16) LA_SMALL(64, 32) LA_SMALL(64, 64)
#undef LA_SMALL
    *handled = false;
    return cudaSuccess;
}

}  // namespace

cudaError_t recurrent_step(const void* q, const void* k, const void* v, float* S, float* z, void* out,
                           const la_shape& s, cudaStream_t st) {
    const int BH = s.B * s.H;
    bool handled = false;
    cudaError_t e;
    launch_begin("recurrent_step", st);
    if (s.dtype == LA_BF16)
        e = dispatch_small<__nv_bfloat16>(q, k, v, S, z, out, BH, s.Dk, s.Dv, st, &handled);
    else
        e = dispatch_small<float>(q, k, v, S, z, out, BH, s.Dk, s.Dv, st, &handled);
    if (handled) {
        cudaError_t e2 = launch_end("recurrent_step", st);
        return e != cudaSuccess ? e : e2;
    }
    const unsigned blocks = (unsigned)((BH + kWarpsPerBlock - 1) / kWarpsPerBlock);
    if (s.dtype == LA_BF16)
        recurrent_step_kernel<__nv_bfloat16><<<blocks, 32 * kWarpsPerBlock, 0, st>>>(
            (const __nv_bfloat16*)q, (const __nv_bfloat16*)k, (const __nv_bfloat16*)v, S, z, (__nv_bfloat16*)out, BH,
            s.Dk, s.Dv);
    else
        recurrent_step_kernel<float><<<blocks, 32 * kWarpsPerBlock, 0, st>>>(
            (const float*)q, (const float*)k, (const float*)v, S, z, (float*)out, BH, s.Dk, s.Dv);
    return launch_end("recurrent_step", st);
}

}  // namespace la
