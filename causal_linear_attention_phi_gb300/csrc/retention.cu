// retention.cu -- causal linear attention with a constant decay per head
// (RetNet's retention, itwiki 선형 어텐션, 발전: 감쇠, 게이트, 델타 규칙):
//   S_t = gamma S_(t-1) + k_t v_t^T,   o_t = S_t^T q_t,
// with the identity feature map and no normaliser.  gamma = 1 is the plain
// causal product tril(Q K^T) V; gamma = 0 keeps only o_t = (q_t . k_t) v_t.
//
// Chunked form.  For a chunk of n positions starting at c0 (a, b = 0..n-1
// inside it) and S_in the state after position c0 - 1:
//   o_(c0+a) = gamma^(a+1) q_a^T S_in + sum_(b<=a) gamma^(a-b) (q_a . k_b) v_b
//   S_out    = gamma^n S_in + sum_b gamma^(n-1-b) k_b v_b^T
// The first term is the carried state seen a+1 steps later; the second is the
// chunk's own causal product with a decay mask.  Segments of `cps` chunks give
// independent CTAs: each segment's local state (started from zero) is summed
// by one kernel, an exclusive scan R_(p+1) = gamma^(L_p) R_p + seg_p (L_p the
// segment's length in positions) forms the state entering every segment, and
// the output kernel walks the segment's chunks from that state.
//
// Powers gamma^m are formed by square-and-multiply in fp64 and rounded once to
// fp32 (0^0 = 1, so gamma = 0 needs no special case); each CTA keeps a table of
// gamma^0 .. gamma^C in shared memory.  Accumulation is fp32 throughout.
#include "simt_common.cuh"

namespace la {
namespace {

using namespace simt;

// g^m for m >= 0 by binary exponentiation (square-and-multiply).
__device__ __forceinline__ double pow_int(double g, int m) {
    double r = 1.0, b = g;
    while (m > 0) {
        if (m & 1) r *= b;
        b *= b;
        m >>= 1;
    }
    return r;
}

__device__ __forceinline__ void fill_powers(float* pw, float g) {
    for (int t = threadIdx.x; t <= kC; t += kThreads) pw[t] = (float)pow_int((double)g, t);
}

// ---------------------------------------------------------------- segment sums
// seg[bh][p] = the state after the segment's last position when the segment
// starts from S = 0:  sum over its positions j of gamma^(L_end - 1 - j) k_j v_j^T.
template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
retention_sums_kernel(const T* __restrict__ k, const T* __restrict__ v, const float* __restrict__ gamma,
                      float* __restrict__ seg, int H, int N, int Dk, int Dv, int nchunks, int cps, int P) {
    extern __shared__ __align__(16) char smem_raw[];
    Smem sm{smem_raw};
    const int ldk = Dk + 1, ldv = Dv + 1;
    float* ks = sm.take((size_t)kC * ldk);
    float* vs = sm.take((size_t)kC * ldv);
    float* pw = sm.take(kC + 1);
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int nA = Dk / 16, nB = Dv / 16;
    const int p = blockIdx.x;
    const size_t bh = blockIdx.y;
    const T* kh = k + bh * N * Dk;
    const T* vh = v + bh * N * Dv;
    fill_powers(pw, gamma[bh % H]);

    float s[kMaxT][kMaxT];
#pragma unroll
    for (int a = 0; a < kMaxT; ++a)
#pragma unroll
        for (int j = 0; j < kMaxT; ++j) s[a][j] = 0.f;

    const int cbeg = p * cps, cend = min(nchunks, cbeg + cps);

    LA_DCHECK(p < (int)gridDim.x && cbeg < cend && cend <= nchunks && (long long)nchunks * kC < (long long)N + kC);
    for (int c = cbeg; c < cend; ++c) {
        const int c0 = c * kC, n = min(kC, N - c0);
        LA_DCHECK(c0 >= 0 && n >= 1 && c0 + n <= N && blockIdx.y < gridDim.y);
        __syncthreads();
        load_tile(ks, ldk, kh, c0, n, Dk, false);
        load_tile(vs, ldv, vh, c0, n, Dv, false);
        __syncthreads();
        const float gn = pw[n];
#pragma unroll
        for (int a = 0; a < kMaxT; ++a)
#pragma unroll
            for (int j = 0; j < kMaxT; ++j) s[a][j] *= gn;
        for (int b = 0; b < n; ++b) {
            const float w = pw[n - 1 - b];
            float kd[kMaxT], vm[kMaxT];
#pragma unroll
            for (int a = 0; a < kMaxT; ++a) kd[a] = (a < nA) ? w * ks[b * ldk + ty + 16 * a] : 0.f;
#pragma unroll
            for (int j = 0; j < kMaxT; ++j) vm[j] = (j < nB) ? vs[b * ldv + tx + 16 * j] : 0.f;
#pragma unroll
            for (int a = 0; a < kMaxT; ++a)
#pragma unroll
                for (int j = 0; j < kMaxT; ++j) s[a][j] = fmaf(kd[a], vm[j], s[a][j]);
        }
    }
    float* out = seg + (bh * P + p) * (size_t)Dk * Dv;  // unpadded records on this path
#pragma unroll
    for (int a = 0; a < kMaxT; ++a)
#pragma unroll
        for (int j = 0; j < kMaxT; ++j)
            if (a < nA && j < nB) out[(size_t)(ty + 16 * a) * Dv + tx + 16 * j] = s[a][j];
}

// ---------------------------------------------------------------- decayed scan over segments
// In place: seg[bh][p] <- R_p with R_0 = 0 and R_(p+1) = gamma^(L_p) R_p + seg[bh][p].
// A record is an sk x sv state (sk = Dk, sv = Dv, or 128 x 128 on the padded
// tensor-core path).  With S_out, R_P (the state after position N) is written
// to S_out[bh] as Dk x Dv.  Each thread owns four consecutive elements of every
// record (E = sk * sv).
constexpr int kScanBatch = 24;  // covers the segment counts the planner picks for the long workloads (19)

__global__ void retention_scan_kernel(float* __restrict__ seg, float* __restrict__ S_out,
                                      const float* __restrict__ gamma, int H, int N, int P, int seg_len, size_t E,
                                      int sv, int Dk, int Dv) {
    pdl_enter();  // launched with programmatic dependent launch
    const size_t bh = blockIdx.y;
    // the segment decays, once per block (fp64 square-and-multiply is slow; every thread needs them)
    __shared__ float decay[2];
    if (threadIdx.x == 0) {
        const double g = gamma[bh % H];
        decay[0] = (float)pow_int(g, seg_len);
        decay[1] = (float)pow_int(g, N - (P - 1) * seg_len);
    }
    __syncthreads();
    const float d_full = decay[0], d_last = decay[1];
    const size_t e4 = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
    if (e4 >= E) return;
    float* base = seg + bh * P * E + e4;
    float4 run = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int b0 = 0; b0 < P; b0 += kScanBatch) {
        const int nb = min(kScanBatch, P - b0);
        float4 t[kScanBatch];
#pragma unroll
        for (int j = 0; j < kScanBatch; ++j)
            if (j < nb) t[j] = *reinterpret_cast<const float4*>(base + (size_t)(b0 + j) * E);
#pragma unroll
        for (int j = 0; j < kScanBatch; ++j) {
            if (j < nb) {
                const int p = b0 + j;
                *reinterpret_cast<float4*>(base + (size_t)p * E) = run;
                const float d = p == P - 1 ? d_last : d_full;
                run.x = fmaf(d, run.x, t[j].x);
                run.y = fmaf(d, run.y, t[j].y);
                run.z = fmaf(d, run.z, t[j].z);
                run.w = fmaf(d, run.w, t[j].w);
            }
        }
    }
    if (S_out) {
        const int d = (int)(e4 / sv), m = (int)(e4 % sv);
        if (d < Dk && m < Dv) *reinterpret_cast<float4*>(S_out + bh * Dk * Dv + (size_t)d * Dv + m) = run;
    }
}

// ---------------------------------------------------------------- outputs
// Per chunk: A = tril(Q_c K_c^T) with A[a][b] scaled by gamma^(a-b);
// o_a = sum_b A[a][b] v_b + gamma^(a+1) q_a^T S; then the state update.
template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
retention_out_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                     const float* __restrict__ gamma, T* __restrict__ o, const float* __restrict__ seg, int H, int N,
                     int Dk, int Dv, int nchunks, int cps, int P) {
    extern __shared__ __align__(16) char smem_raw[];
    Smem sm{smem_raw};
    const int ldk = Dk + 1, ldv = Dv + 1, lds = Dv + 1;
    float* qs = sm.take((size_t)kC * ldk);
    float* ks = sm.take((size_t)kC * ldk);
    float* vs = sm.take((size_t)kC * ldv);
    float* A = sm.take((size_t)kC * kC);
    float* Ss = sm.take((size_t)Dk * lds);
    float* pw = sm.take(kC + 1);
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int nA = Dk / 16, nB = Dv / 16;
    const int p = blockIdx.x;
    const size_t bh = blockIdx.y;
    const T* qh = q + bh * N * Dk;
    const T* kh = k + bh * N * Dk;
    const T* vh = v + bh * N * Dv;
    T* oh = o + bh * N * Dv;
    const float* init = seg + (bh * P + p) * (size_t)Dk * Dv;
    fill_powers(pw, gamma[bh % H]);

    float s[kMaxT][kMaxT];
#pragma unroll
    for (int a = 0; a < kMaxT; ++a)
#pragma unroll
        for (int j = 0; j < kMaxT; ++j) {
            float x = 0.f;
            if (a < nA && j < nB) {
                x = init[(size_t)(ty + 16 * a) * Dv + tx + 16 * j];
                Ss[(ty + 16 * a) * lds + tx + 16 * j] = x;
            }
            s[a][j] = x;
        }

    const int cbeg = p * cps, cend = min(nchunks, cbeg + cps);

    LA_DCHECK(p < (int)gridDim.x && cbeg < cend && cend <= nchunks && (long long)nchunks * kC < (long long)N + kC);
    for (int c = cbeg; c < cend; ++c) {
        const int c0 = c * kC, n = min(kC, N - c0);
        LA_DCHECK(c0 >= 0 && n >= 1 && c0 + n <= N && blockIdx.y < gridDim.y);
        __syncthreads();
        load_tile(qs, ldk, qh, c0, n, Dk, false);
        load_tile(ks, ldk, kh, c0, n, Dk, false);
        load_tile(vs, ldv, vh, c0, n, Dv, false);
        __syncthreads();
        // A = tril(Q K^T) with the decay mask
#pragma unroll
        for (int i = 0; i < kC / 16; ++i)
#pragma unroll
            for (int j = 0; j < kC / 16; ++j) {
                const int a = ty + 16 * i, b = tx + 16 * j;
                float acc = 0.f;
                for (int d = 0; d < Dk; ++d) acc = fmaf(qs[a * ldk + d], ks[b * ldk + d], acc);
                A[a * kC + b] = (b <= a) ? acc * pw[b <= a ? a - b : 0] : 0.f;
            }
        __syncthreads();
#pragma unroll 1
        for (int i = 0; i < kC / 16; ++i) {
            const int a = ty + 16 * i;
            if (a >= n) break;
            float intra[kMaxT], carry[kMaxT];
#pragma unroll
            for (int j = 0; j < kMaxT; ++j) intra[j] = carry[j] = 0.f;
            for (int b = 0; b <= a; ++b) {
                const float w = A[a * kC + b];
#pragma unroll
                for (int j = 0; j < kMaxT; ++j)
                    if (j < nB) intra[j] = fmaf(w, vs[b * ldv + tx + 16 * j], intra[j]);
            }
            for (int d = 0; d < Dk; ++d) {
                const float qd = qs[a * ldk + d];
#pragma unroll
                for (int j = 0; j < kMaxT; ++j)
                    if (j < nB) carry[j] = fmaf(qd, Ss[d * lds + tx + 16 * j], carry[j]);
            }
            const float ga = pw[a + 1];
#pragma unroll
            for (int j = 0; j < kMaxT; ++j)
                if (j < nB) oh[(size_t)(c0 + a) * Dv + tx + 16 * j] = from_f32<T>(fmaf(ga, carry[j], intra[j]));
        }
        __syncthreads();
        // S <- gamma^n S + sum_b gamma^(n-1-b) k_b v_b^T
        const float gn = pw[n];
#pragma unroll
        for (int a = 0; a < kMaxT; ++a)
#pragma unroll
            for (int j = 0; j < kMaxT; ++j) s[a][j] *= gn;
        for (int b = 0; b < n; ++b) {
            const float w = pw[n - 1 - b];
            float kd[kMaxT], vm[kMaxT];
#pragma unroll
            for (int a = 0; a < kMaxT; ++a) kd[a] = (a < nA) ? w * ks[b * ldk + ty + 16 * a] : 0.f;
#pragma unroll
            for (int j = 0; j < kMaxT; ++j) vm[j] = (j < nB) ? vs[b * ldv + tx + 16 * j] : 0.f;
#pragma unroll
            for (int a = 0; a < kMaxT; ++a)
#pragma unroll
                for (int j = 0; j < kMaxT; ++j) s[a][j] = fmaf(kd[a], vm[j], s[a][j]);
        }
#pragma unroll
        for (int a = 0; a < kMaxT; ++a)
#pragma unroll
            for (int j = 0; j < kMaxT; ++j)
                if (a < nA && j < nB) Ss[(ty + 16 * a) * lds + tx + 16 * j] = s[a][j];
    }
}

// ---------------------------------------------------------------- one decode step
// S <- gamma S + k v^T, out = S^T q, one warp per head.  S rows move as float4
// (Dv / 4 lanes across a row, 32 / (Dv / 4) rows per warp instruction); lanes
// that share a column group combine their partial outputs with shuffles.
constexpr int kStepWarps = 2;

template <typename T>
__global__ void __launch_bounds__(32 * kStepWarps)
retention_step_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                      const float* __restrict__ gamma, float* __restrict__ S, T* __restrict__ out, int BH, int H,
                      int Dk, int Dv) {
    __shared__ float qk_s[kStepWarps][2][128];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.x * kStepWarps + warp;
    if (h >= BH) return;  // whole warp leaves together
    const float g = gamma[h % H];
    for (int d = lane; d < Dk; d += 32) {
        qk_s[warp][0][d] = to_f32(q[(size_t)h * Dk + d]);
        qk_s[warp][1][d] = to_f32(k[(size_t)h * Dk + d]);
    }
    __syncwarp();
    const int ncol4 = Dv >> 2;  // 4..32
    const int rows_per_iter = 32 / ncol4;
    const int c4 = lane % ncol4, rsub = lane / ncol4;
    const int col = c4 * 4;
    float* Sh = S + (size_t)h * Dk * Dv;
    const T* vh = v + (size_t)h * Dv + col;
    float4 vv;
    vv.x = to_f32(vh[0]);
    vv.y = to_f32(vh[1]);
    vv.z = to_f32(vh[2]);
    vv.w = to_f32(vh[3]);
    float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
    for (int d = rsub; d < Dk; d += rows_per_iter) {
        float4* sp = reinterpret_cast<float4*>(Sh + (size_t)d * Dv + col);
        float4 s = *sp;
        const float kt = qk_s[warp][1][d], qt = qk_s[warp][0][d];
        s.x = fmaf(kt, vv.x, g * s.x);
        s.y = fmaf(kt, vv.y, g * s.y);
        s.z = fmaf(kt, vv.z, g * s.z);
        s.w = fmaf(kt, vv.w, g * s.w);
        *sp = s;
        num.x = fmaf(qt, s.x, num.x);
        num.y = fmaf(qt, s.y, num.y);
        num.z = fmaf(qt, s.z, num.z);
        num.w = fmaf(qt, s.w, num.w);
    }
    for (int o = ncol4; o < 32; o <<= 1) {
        num.x += __shfl_xor_sync(0xffffffffu, num.x, o);
        num.y += __shfl_xor_sync(0xffffffffu, num.y, o);
        num.z += __shfl_xor_sync(0xffffffffu, num.z, o);
        num.w += __shfl_xor_sync(0xffffffffu, num.w, o);
    }
    if (rsub == 0) {
        T* oh = out + (size_t)h * Dv + col;
        oh[0] = from_f32<T>(num.x);
        oh[1] = from_f32<T>(num.y);
        oh[2] = from_f32<T>(num.z);
        oh[3] = from_f32<T>(num.w);
    }
}

// Four consecutive elements as one vector access (16 bytes of fp32, 8 of bf16).
__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 ld4(const __nv_bfloat16* p) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(p);
    const float2 a = __bfloat1622float2(h[0]), b = __bfloat1622float2(h[1]);
    return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ void st4(float* p, float4 x) { *reinterpret_cast<float4*>(p) = x; }
__device__ __forceinline__ void st4(__nv_bfloat16* p, float4 x) {
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(p);
    h[0] = __floats2bfloat162_rn(x.x, x.y);
    h[1] = __floats2bfloat162_rn(x.z, x.w);
}

// Heads with Dk, Dv <= 64: one warp per head with S held in registers as float4s
// (COLS = Dv/4 lanes across a row, RPI = 32/COLS rows per instruction, ROWS = Dk/RPI
// rows per lane), every global load of the step issued before any arithmetic (one
// memory round trip), q and k read once per element (lane d % 32) and handed to the
// lanes of row d by a shuffle.  Launched with programmatic stream serialization: the
// grid may be scheduled while the previous kernel in the stream drains and waits
// (griddepcontrol.wait) before its first global access, so the order memory sees is
// the stream's.
template <typename T, int DK, int DV>
__global__ void __launch_bounds__(32 * kStepWarps)
retention_step_small_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                            const float* __restrict__ gamma, float* __restrict__ S, T* __restrict__ out, int BH,
                            int H) {
    constexpr int COLS = DV / 4;
    constexpr int RPI = 32 / COLS;
    constexpr int ROWS = DK / RPI;
    constexpr int QPL = (DK + 31) / 32;  // q, k entries per lane
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.x * kStepWarps + warp;
    if (h >= BH) return;
    const int c4 = lane % COLS, rsub = lane / COLS;
    const int col = c4 * 4;
    float* Sh = S + (size_t)h * DK * DV;
    float4 st[ROWS];
#pragma unroll
    for (int x = 0; x < ROWS; ++x)
        st[x] = *reinterpret_cast<const float4*>(Sh + (size_t)(rsub + RPI * x) * DV + col);
    const float4 vv = ld4(v + (size_t)h * DV + col);
    float qa[QPL], ka[QPL];
#pragma unroll
    for (int y = 0; y < QPL; ++y) {
        const int d = lane + 32 * y;
        qa[y] = d < DK ? to_f32(q[(size_t)h * DK + d]) : 0.f;
        ka[y] = d < DK ? to_f32(k[(size_t)h * DK + d]) : 0.f;
    }
    const float g = gamma[h % H];
    float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int x = 0; x < ROWS; ++x) {
        const int d = rsub + RPI * x;
        float kd = __shfl_sync(0xffffffffu, ka[0], d & 31), qd = __shfl_sync(0xffffffffu, qa[0], d & 31);
        if (QPL > 1) {
            const float k1 = __shfl_sync(0xffffffffu, ka[QPL - 1], d & 31);
            const float q1 = __shfl_sync(0xffffffffu, qa[QPL - 1], d & 31);
            if (d >= 32) {
                kd = k1;
                qd = q1;
            }
        }
        float4 t = st[x];
        t.x = fmaf(kd, vv.x, g * t.x);
        t.y = fmaf(kd, vv.y, g * t.y);
        t.z = fmaf(kd, vv.z, g * t.z);
        t.w = fmaf(kd, vv.w, g * t.w);
        *reinterpret_cast<float4*>(Sh + (size_t)d * DV + col) = t;
        num.x = fmaf(qd, t.x, num.x);
        num.y = fmaf(qd, t.y, num.y);
        num.z = fmaf(qd, t.z, num.z);
        num.w = fmaf(qd, t.w, num.w);
    }
#pragma unroll
    for (int o = COLS; o < 32; o <<= 1) {
        num.x += __shfl_xor_sync(0xffffffffu, num.x, o);
        num.y += __shfl_xor_sync(0xffffffffu, num.y, o);
        num.z += __shfl_xor_sync(0xffffffffu, num.z, o);
        num.w += __shfl_xor_sync(0xffffffffu, num.w, o);
    }
    if (rsub == 0) st4(out + (size_t)h * DV + col, num);
}

template <typename T, int DK, int DV>
cudaError_t launch_step_small(const void* q, const void* k, const void* v, const float* gamma, float* S, void* out,
                              int BH, int H, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((BH + kStepWarps - 1) / kStepWarps));
    cfg.blockDim = dim3(32 * kStepWarps);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, retention_step_small_kernel<T, DK, DV>, (const T*)q, (const T*)k, (const T*)v,
                              gamma, S, (T*)out, BH, H);
}

// The small-head fast path for (Dk, Dv) in {16, 32, 64}^2; *handled = false otherwise.
template <typename T>
cudaError_t step_small(const void* q, const void* k, const void* v, const float* gamma, float* S, void* out, int BH,
                       int H, int Dk, int Dv, cudaStream_t st, bool* handled) {
    *handled = true;
#define LA_RET_SMALL(a, b) \
    if (Dk == a && Dv == b) return launch_step_small<T, a, b>(q, k, v, gamma, S, out, BH, H, st);
    LA_RET_SMALL(16, 16) LA_RET_SMALL(16, 32) LA_RET_SMALL(16, 64) LA_RET_SMALL(32, 16) LA_RET_SMALL(32, 32)
    LA_RET_SMALL(32, 64) LA_RET_SMALL(64, 16) LA_RET_SMALL(64, 32) LA_RET_SMALL(64, 64)
#undef LA_RET_SMALL
    *handled = false;
    return cudaSuccess;
}

size_t smem_bytes_sums(int Dk, int Dv) {
    return smem_floats((size_t)kC * (Dk + 1)) + smem_floats((size_t)kC * (Dv + 1)) + smem_floats(kC + 1);
}
size_t smem_bytes_out(int Dk, int Dv) {
    return smem_floats((size_t)kC * (Dk + 1)) * 2 + smem_floats((size_t)kC * (Dv + 1)) + smem_floats((size_t)kC * kC) +
           smem_floats((size_t)Dk * (Dv + 1)) + smem_floats(kC + 1);
}

}  // namespace

cudaError_t retention_segment_sums(const void* k, const void* v, const float* gamma, float* seg, const la_shape& s,
                                   const Plan& p, cudaStream_t st) {
    const size_t smem = smem_bytes_sums(s.Dk, s.Dv);
    const dim3 grid(p.P, s.B * s.H);
    cudaError_t err = cudaSuccess;
    auto run = [&](auto tag) {
        using T = decltype(tag);
        auto kern = retention_sums_kernel<T>;
        if ((err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
            return;
        launch_begin("retention_segment_sums", st);
        kern<<<grid, kThreads, smem, st>>>((const T*)k, (const T*)v, gamma, seg, s.H, s.N, s.Dk, s.Dv, p.nchunks,
                                           p.cps, p.P);
        err = launch_end("retention_segment_sums", st);
    };
    if (s.dtype == LA_BF16)
        run(__nv_bfloat16{});
    else
        run(float{});
    return err;
}

cudaError_t retention_scan(float* seg, float* S_out, const float* gamma, const la_shape& s, const Plan& p,
                           cudaStream_t st) {
    const size_t E = (size_t)p.sk * p.sv;  // a multiple of 256 for the supported head sizes
    const dim3 grid((unsigned)((E / 4 + 127) / 128), s.B * s.H);
    launch_begin("retention_scan", st);
    const cudaError_t le = launch_pdl(retention_scan_kernel, grid, dim3(128), 0, st, seg, S_out, gamma, s.H, s.N, p.P,
                                      p.cps * p.C, E, p.sv, s.Dk, s.Dv);
    const cudaError_t le2 = launch_end("retention_scan", st);
    return le != cudaSuccess ? le : le2;
}

cudaError_t retention_out(const void* q, const void* k, const void* v, const float* gamma, void* o, const float* seg,
                          const la_shape& s, const Plan& p, cudaStream_t st) {
    const size_t smem = smem_bytes_out(s.Dk, s.Dv);
    const dim3 grid(p.P, s.B * s.H);
    cudaError_t err = cudaSuccess;
    auto run = [&](auto tag) {
        using T = decltype(tag);
        auto kern = retention_out_kernel<T>;
        if ((err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
            return;
        launch_begin("retention_out", st);
        kern<<<grid, kThreads, smem, st>>>((const T*)q, (const T*)k, (const T*)v, gamma, (T*)o, seg, s.H, s.N, s.Dk,
                                           s.Dv, p.nchunks, p.cps, p.P);
        err = launch_end("retention_out", st);
    };
    if (s.dtype == LA_BF16)
        run(__nv_bfloat16{});
    else
        run(float{});
    return err;
}

cudaError_t retention_step(const void* q, const void* k, const void* v, const float* gamma, float* S, void* out,
                           const la_shape& s, cudaStream_t st) {
    const int BH = s.B * s.H;
    const unsigned blocks = (unsigned)((BH + kStepWarps - 1) / kStepWarps);
    launch_begin("retention_step", st);
    bool handled = false;
    cudaError_t e = s.dtype == LA_BF16
                        ? step_small<__nv_bfloat16>(q, k, v, gamma, S, out, BH, s.H, s.Dk, s.Dv, st, &handled)
                        : step_small<float>(q, k, v, gamma, S, out, BH, s.H, s.Dk, s.Dv, st, &handled);
    if (handled) {
        const cudaError_t e2 = launch_end("retention_step", st);
        return e != cudaSuccess ? e : e2;
    }
    if (s.dtype == LA_BF16)
        retention_step_kernel<__nv_bfloat16><<<blocks, 32 * kStepWarps, 0, st>>>(
            (const __nv_bfloat16*)q, (const __nv_bfloat16*)k, (const __nv_bfloat16*)v, gamma, S,
            (__nv_bfloat16*)out, BH, s.H, s.Dk, s.Dv);
    else
        retention_step_kernel<float><<<blocks, 32 * kStepWarps, 0, st>>>((const float*)q, (const float*)k,
                                                                         (const float*)v, gamma, S, (float*)out, BH,
                                                                         s.H, s.Dk, s.Dv);
    return launch_end("retention_step", st);
}

}  // namespace la
