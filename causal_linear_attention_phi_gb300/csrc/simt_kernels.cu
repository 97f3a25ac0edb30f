// simt_kernels.cu -- CUDA-core (FFMA) kernels of the chunked causal form, the
// non-causal form and the segment scan.  These serve fp32 inputs (where tf32
// tensor cores cannot meet a 1e-4 relative bound) and every head size the
// tcgen05 kernels do not cover.  Accumulation is fp32 throughout.
//
// Thread layout: 256 threads viewed as a 16 x 16 grid (ty = tid / 16,
// tx = tid % 16).  Register tiles are strided by 16 (row ty + 16*i, column
// tx + 16*j) so that shared-memory reads across a warp hit distinct banks or
// broadcast.  Tiles hold fp32 values with phi already applied ("fused into the
// tile load"); rows past the end of the sequence hold zeros.
#include <mutex>

#include "simt_common.cuh"

namespace la {
namespace {

using namespace simt;

// ---------------------------------------------------------------- segment sums
// seg[bh][p] = ( sum over the segment of phi(k_j) v_j^T , sum of phi(k_j) ).
template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
segment_sums_kernel(const T* __restrict__ k, const T* __restrict__ v, float* __restrict__ seg, int N, int Dk,
                    int Dv, int nchunks, int cps, int P) {
    extern __shared__ __align__(16) char smem_raw[];
    Smem sm{smem_raw};
    const int ldk = Dk + 1, ldv = Dv + 1;
    float* ks = sm.take((size_t)kC * ldk);
    float* vs = sm.take((size_t)kC * ldv);
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int nA = Dk / 16, nB = Dv / 16;
    const int p = blockIdx.x;
    const size_t bh = blockIdx.y;
    const T* kh = k + bh * N * Dk;
    const T* vh = v + bh * N * Dv;

    float s[kMaxT][kMaxT];
#pragma unroll
    for (int a = 0; a < kMaxT; ++a)
#pragma unroll
        for (int j = 0; j < kMaxT; ++j) s[a][j] = 0.f;
    float zacc = 0.f;

    const int cbeg = p * cps, cend = min(nchunks, cbeg + cps);

    LA_DCHECK(p < (int)gridDim.x && cbeg < cend && cend <= nchunks && (long long)nchunks * kC < (long long)N + kC);
    for (int c = cbeg; c < cend; ++c) {
        const int c0 = c * kC, n = min(kC, N - c0);
        LA_DCHECK(c0 >= 0 && n >= 1 && c0 + n <= N && blockIdx.y < gridDim.y);
        __syncthreads();
        load_tile(ks, ldk, kh, c0, n, Dk, true);
        load_tile(vs, ldv, vh, c0, n, Dv, false);
        __syncthreads();
        for (int b = 0; b < n; ++b) {
            float kd[kMaxT], vm[kMaxT];
#pragma unroll
            for (int a = 0; a < kMaxT; ++a) kd[a] = (a < nA) ? ks[b * ldk + ty + 16 * a] : 0.f;
#pragma unroll
            for (int j = 0; j < kMaxT; ++j) vm[j] = (j < nB) ? vs[b * ldv + tx + 16 * j] : 0.f;
#pragma unroll
            for (int a = 0; a < kMaxT; ++a)
#pragma unroll
                for (int j = 0; j < kMaxT; ++j) s[a][j] = fmaf(kd[a], vm[j], s[a][j]);
        }
        if (tid < Dk)
            for (int b = 0; b < n; ++b) zacc += ks[b * ldk + tid];
    }
    float* out = seg + (bh * P + p) * state_elems(Dk, Dv);
#pragma unroll
    for (int a = 0; a < kMaxT; ++a)
#pragma unroll
        for (int j = 0; j < kMaxT; ++j)
            if (a < nA && j < nB) out[(size_t)(ty + 16 * a) * Dv + tx + 16 * j] = s[a][j];
    if (tid < Dk) out[(size_t)Dk * Dv + tid] = zacc;
}

// ---------------------------------------------------------------- scan over segments
// mode 0: exclusive prefix over p (in place); 1: exclusive suffix (in place);
// 2: totals only (seg unchanged).  With totS, the sum over p of each record is
// also written.  A record is an sk x sv state (row length sv) followed by sk z
// entries; of these, rows < Dk and columns < Dv of the state go to
// totS + bh * sS (row length Dv) and z entries < Dk to totz + bh * sz (sk = Dk,
// sv = Dv except on the padded tensor-core path).  Each thread owns four
// consecutive elements (one float4, inside one row) of every segment record and
// walks the P records in batches whose loads are all issued before any of them
// is used.
constexpr int kScanBatch = 24;  // covers the segment counts the planner picks for the long workloads (19)

__global__ void scan_kernel(float* __restrict__ seg, float* __restrict__ totS, float* __restrict__ totz, size_t sS,
                            size_t sz, int P, size_t E, int sk, int sv, int Dk, int Dv, int mode) {
    pdl_enter();  // launched with programmatic dependent launch: the records are visible from here on
    const size_t e4 = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
    if (e4 >= E) return;
    const size_t bh = blockIdx.y;
    if (!LA_DCHECK((E & 3) == 0 && (sv & 3) == 0 && e4 + 3 < E && P >= 1)) return;
    float* base = seg + bh * P * E + e4;
    float4 run = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int b0 = 0; b0 < P; b0 += kScanBatch) {
        const int nb = min(kScanBatch, P - b0);
        float4 t[kScanBatch];
#pragma unroll
        for (int j = 0; j < kScanBatch; ++j) {
            if (j < nb) {
                const int p = mode == SCAN_EXCLUSIVE_SUFFIX ? P - 1 - (b0 + j) : b0 + j;
                t[j] = *reinterpret_cast<const float4*>(base + (size_t)p * E);
            }
        }
#pragma unroll
        for (int j = 0; j < kScanBatch; ++j) {
            if (j < nb) {
                const int p = mode == SCAN_EXCLUSIVE_SUFFIX ? P - 1 - (b0 + j) : b0 + j;
                if (mode != SCAN_TOTAL) *reinterpret_cast<float4*>(base + (size_t)p * E) = run;
                run.x += t[j].x;
                run.y += t[j].y;
                run.z += t[j].z;
                run.w += t[j].w;
            }
        }
    }
    if (totS) {
        const size_t SkSv = (size_t)sk * sv;
        if (e4 < SkSv) {
            const int d = (int)(e4 / sv), m = (int)(e4 % sv);
            if (d < Dk && m < Dv) *reinterpret_cast<float4*>(totS + bh * sS + (size_t)d * Dv + m) = run;
        } else if (e4 - SkSv < (size_t)Dk) {
            *reinterpret_cast<float4*>(totz + bh * sz + (e4 - SkSv)) = run;
        }
    }
}

// ---------------------------------------------------------------- causal forward
// Per chunk: A = tril(phi(Q_c) phi(K_c)^T); o = (A V_c + phi(Q_c) S) / (A 1 + phi(Q_c) z);
// then S += phi(K_c)^T V_c, z += phi(K_c)^T 1.  S, z enter from the scanned prefix.
template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
causal_fwd_out_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v, T* __restrict__ o,
                      const float* __restrict__ seg, int N, int Dk, int Dv, int nchunks, int cps, int P) {
    extern __shared__ __align__(16) char smem_raw[];
    Smem sm{smem_raw};
    const int ldk = Dk + 1, ldv = Dv + 1, lds = Dv + 1;
    float* qs = sm.take((size_t)kC * ldk);
    float* ks = sm.take((size_t)kC * ldk);
    float* vs = sm.take((size_t)kC * ldv);
    float* A = sm.take((size_t)kC * kC);
    float* Ss = sm.take((size_t)Dk * lds);
    float* zs = sm.take((size_t)Dk);
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int nA = Dk / 16, nB = Dv / 16;
    const int p = blockIdx.x;
    const size_t bh = blockIdx.y;
    const T* qh = q + bh * N * Dk;
    const T* kh = k + bh * N * Dk;
    const T* vh = v + bh * N * Dv;
    T* oh = o + bh * N * Dv;
    const float* init = seg + (bh * P + p) * state_elems(Dk, Dv);

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
    float zreg = 0.f;
    if (tid < Dk) {
        zreg = init[(size_t)Dk * Dv + tid];
        zs[tid] = zreg;
    }

    const int cbeg = p * cps, cend = min(nchunks, cbeg + cps);

    LA_DCHECK(p < (int)gridDim.x && cbeg < cend && cend <= nchunks && (long long)nchunks * kC < (long long)N + kC);
    for (int c = cbeg; c < cend; ++c) {
        const int c0 = c * kC, n = min(kC, N - c0);
        LA_DCHECK(c0 >= 0 && n >= 1 && c0 + n <= N && blockIdx.y < gridDim.y);
        __syncthreads();
        load_tile(qs, ldk, qh, c0, n, Dk, true);
        load_tile(ks, ldk, kh, c0, n, Dk, true);
        load_tile(vs, ldv, vh, c0, n, Dv, false);
        __syncthreads();
        // A = tril(Q~ K~^T)
#pragma unroll
        for (int i = 0; i < kC / 16; ++i)
#pragma unroll
            for (int j = 0; j < kC / 16; ++j) {
                const int a = ty + 16 * i, b = tx + 16 * j;
                float acc = 0.f;
                for (int d = 0; d < Dk; ++d) acc = fmaf(qs[a * ldk + d], ks[b * ldk + d], acc);
                A[a * kC + b] = (b <= a) ? acc : 0.f;
            }
        __syncthreads();
        // outputs
#pragma unroll 1
        for (int i = 0; i < kC / 16; ++i) {
            const int a = ty + 16 * i;
            float num[kMaxT];
#pragma unroll
            for (int j = 0; j < kMaxT; ++j) num[j] = 0.f;
            float den = 0.f;
            for (int b = 0; b <= a; ++b) {
                const float w = A[a * kC + b];
                den += w;
#pragma unroll
                for (int j = 0; j < kMaxT; ++j)
                    if (j < nB) num[j] = fmaf(w, vs[b * ldv + tx + 16 * j], num[j]);
            }
            for (int d = 0; d < Dk; ++d) {
                const float qd = qs[a * ldk + d];
                den = fmaf(qd, zs[d], den);
#pragma unroll
                for (int j = 0; j < kMaxT; ++j)
                    if (j < nB) num[j] = fmaf(qd, Ss[d * lds + tx + 16 * j], num[j]);
            }
            if (a < n) {
#pragma unroll
                for (int j = 0; j < kMaxT; ++j)
                    if (j < nB) oh[(size_t)(c0 + a) * Dv + tx + 16 * j] = from_f32<T>(num[j] / den);
            }
        }
        __syncthreads();
        // state update
        for (int b = 0; b < n; ++b) {
            float kd[kMaxT], vm[kMaxT];
#pragma unroll
            for (int a = 0; a < kMaxT; ++a) kd[a] = (a < nA) ? ks[b * ldk + ty + 16 * a] : 0.f;
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
        if (tid < Dk) {
            for (int b = 0; b < n; ++b) zreg += ks[b * ldk + tid];
            zs[tid] = zreg;
        }
    }
}

// ---------------------------------------------------------------- non-causal apply
// o_i = phi(q_i)^T S / phi(q_i)^T z with the head's total (S, z).
template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
noncausal_apply_kernel(const T* __restrict__ q, T* __restrict__ o, const float* __restrict__ totals, int N, int Dk,
                       int Dv) {
    extern __shared__ __align__(16) char smem_raw[];
    Smem sm{smem_raw};
    const int ldk = Dk + 1;
    float* qs = sm.take((size_t)kC * ldk);
    float* Ss = sm.take((size_t)Dk * Dv);
    float* zs = sm.take((size_t)Dk);
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int nB = Dv / 16;
    const size_t bh = blockIdx.y;
    const float* tot = totals + bh * state_elems(Dk, Dv);
    for (int e = tid; e < Dk * Dv; e += kThreads) Ss[e] = tot[e];
    if (tid < Dk) zs[tid] = tot[(size_t)Dk * Dv + tid];
    const int c0 = blockIdx.x * kC, n = min(kC, N - c0);
    LA_DCHECK(c0 >= 0 && n >= 1 && c0 + n <= N && blockIdx.y < gridDim.y);
    load_tile(qs, ldk, q + bh * N * Dk, c0, n, Dk, true);
    __syncthreads();
    for (int i = 0; i < kC / 16; ++i) {
        const int a = ty + 16 * i;
        if (a >= n) break;
        float num[kMaxT];
#pragma unroll
        for (int j = 0; j < kMaxT; ++j) num[j] = 0.f;
        float den = 0.f;
        for (int d = 0; d < Dk; ++d) {
            const float qd = qs[a * ldk + d];
            den = fmaf(qd, zs[d], den);
#pragma unroll
            for (int j = 0; j < kMaxT; ++j)
                if (j < nB) num[j] = fmaf(qd, Ss[d * Dv + tx + 16 * j], num[j]);
        }
#pragma unroll
        for (int j = 0; j < kMaxT; ++j)
            if (j < nB) o[(bh * N + c0 + a) * Dv + tx + 16 * j] = from_f32<T>(num[j] / den);
    }
}

// ---------------------------------------------------------------- backward, forward sweep
// Recomputes den_i and o_i chunk by chunk from the carried (S, z), derives
// P_i = dout_i / den_i and g_i = -(dout_i . o_i) / den_i, writes
// dq = (P S^T + g z^T + D K~) * phi'(q) with D = tril(P V^T + g 1^T), stores
// (den, g) per position, and sums the segment's reverse-state contributions
// (sum phi(q_i) P_i^T, sum g_i phi(q_i)) into seg_R.
template <typename T, bool kCausal>
__global__ void __launch_bounds__(kThreads, 1)
bwd_forward_sweep_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                         const T* __restrict__ dout, T* __restrict__ dq, const float* __restrict__ seg_S,
                         float* __restrict__ seg_R, float* __restrict__ den_g, int N, int Dk, int Dv, int nchunks,
                         int cps, int P) {
    extern __shared__ __align__(16) char smem_raw[];
    Smem sm{smem_raw};
    const int ldk = Dk + 1, ldv = Dv + 1, lds = Dv + 1;
    float* qs = sm.take((size_t)kC * ldk);
    float* ks = sm.take((size_t)kC * ldk);
    float* vs = sm.take((size_t)kC * ldv);
    float* ps = sm.take((size_t)kC * ldv);
    float* AD = sm.take((size_t)kC * kC);
    float* Ss = sm.take((size_t)Dk * lds);
    float* zs = sm.take((size_t)Dk);
    float* gs = sm.take((size_t)kC);
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int nA = Dk / 16, nB = Dv / 16;
    const int p = blockIdx.x;
    const size_t bh = blockIdx.y;
    const T* qh = q + bh * N * Dk;
    const T* kh = k + bh * N * Dk;
    const T* vh = v + bh * N * Dv;
    const T* doh = dout + bh * N * Dv;
    T* dqh = dq + bh * N * Dk;
    float* dgh = den_g + bh * N * 2;
    const size_t E = state_elems(Dk, Dv);
    // causal: the segment's exclusive prefix state; non-causal: the total over the head (fixed)
    const float* init = kCausal ? seg_S + (bh * P + p) * E : seg_S + bh * E;

    float s[kMaxT][kMaxT], r[kMaxT][kMaxT];
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
            r[a][j] = 0.f;
        }
    float zreg = 0.f, rz = 0.f;
    if (tid < Dk) {
        zreg = init[(size_t)Dk * Dv + tid];
        zs[tid] = zreg;
    }

    const int cbeg = p * cps, cend = min(nchunks, cbeg + cps);

    LA_DCHECK(p < (int)gridDim.x && cbeg < cend && cend <= nchunks && (long long)nchunks * kC < (long long)N + kC);
    for (int c = cbeg; c < cend; ++c) {
        const int c0 = c * kC, n = min(kC, N - c0);
        LA_DCHECK(c0 >= 0 && n >= 1 && c0 + n <= N && blockIdx.y < gridDim.y);
        __syncthreads();
        load_tile(qs, ldk, qh, c0, n, Dk, true);
        load_tile(ks, ldk, kh, c0, n, Dk, true);
        load_tile(vs, ldv, vh, c0, n, Dv, false);
        load_tile(ps, ldv, doh, c0, n, Dv, false);
        __syncthreads();
        if (kCausal) {
#pragma unroll
            for (int i = 0; i < kC / 16; ++i)
#pragma unroll
                for (int j = 0; j < kC / 16; ++j) {
                    const int a = ty + 16 * i, b = tx + 16 * j;
                    float acc = 0.f;
                    for (int d = 0; d < Dk; ++d) acc = fmaf(qs[a * ldk + d], ks[b * ldk + d], acc);
                    AD[a * kC + b] = (b <= a) ? acc : 0.f;
                }
        }
        __syncthreads();
        // den, o -> g and P (P overwrites dout in place: each thread touches only its own entries)
#pragma unroll 1
        for (int i = 0; i < kC / 16; ++i) {
            const int a = ty + 16 * i;
            float num[kMaxT];
#pragma unroll
            for (int j = 0; j < kMaxT; ++j) num[j] = 0.f;
            float den = 0.f;
            for (int b = 0; kCausal && b <= a; ++b) {
                const float w = AD[a * kC + b];
                den += w;
#pragma unroll
                for (int j = 0; j < kMaxT; ++j)
                    if (j < nB) num[j] = fmaf(w, vs[b * ldv + tx + 16 * j], num[j]);
            }
            for (int d = 0; d < Dk; ++d) {
                const float qd = qs[a * ldk + d];
                den = fmaf(qd, zs[d], den);
#pragma unroll
                for (int j = 0; j < kMaxT; ++j)
                    if (j < nB) num[j] = fmaf(qd, Ss[d * lds + tx + 16 * j], num[j]);
            }
            const bool valid = a < n;
            if (!valid) den = 1.f;  // masked rows: dout is 0 there, so P = 0 and g = 0
            float dot = 0.f;
#pragma unroll
            for (int j = 0; j < kMaxT; ++j)
                if (j < nB) dot = fmaf(ps[a * ldv + tx + 16 * j], num[j], dot);
            dot += __shfl_xor_sync(0xffffffffu, dot, 1);
            dot += __shfl_xor_sync(0xffffffffu, dot, 2);
            dot += __shfl_xor_sync(0xffffffffu, dot, 4);
            dot += __shfl_xor_sync(0xffffffffu, dot, 8);
            const float inv = 1.f / den;
            const float g = -dot * inv * inv;
#pragma unroll
            for (int j = 0; j < kMaxT; ++j)
                if (j < nB) ps[a * ldv + tx + 16 * j] *= inv;
            if (tx == 0) {
                gs[a] = g;
                if (valid) {
                    dgh[(size_t)(c0 + a) * 2 + 0] = den;
                    dgh[(size_t)(c0 + a) * 2 + 1] = g;
                }
            }
        }
        __syncthreads();
        // D = tril(P V^T + g 1^T), masked to valid columns
        if (kCausal) {
#pragma unroll
            for (int i = 0; i < kC / 16; ++i)
#pragma unroll
                for (int j = 0; j < kC / 16; ++j) {
                    const int a = ty + 16 * i, b = tx + 16 * j;
                    float acc = 0.f;
                    for (int m = 0; m < Dv; ++m) acc = fmaf(ps[a * ldv + m], vs[b * ldv + m], acc);
                    AD[a * kC + b] = (b <= a && b < n) ? acc + gs[a] : 0.f;
                }
        }
        __syncthreads();
        // dq = (P S^T + g z^T + D K~) * phi'(q)  (no D K~ term without the mask: S, z are totals)
#pragma unroll 1
        for (int i = 0; i < kC / 16; ++i) {
            const int a = ty + 16 * i;
            float acc[kMaxT];
#pragma unroll
            for (int j = 0; j < kMaxT; ++j) acc[j] = (j < nA) ? gs[a] * zs[tx + 16 * j] : 0.f;
            for (int m = 0; m < Dv; ++m) {
                const float pm = ps[a * ldv + m];
#pragma unroll
                for (int j = 0; j < kMaxT; ++j)
                    if (j < nA) acc[j] = fmaf(pm, Ss[(tx + 16 * j) * lds + m], acc[j]);
            }
            for (int b = 0; kCausal && b <= a; ++b) {
                const float w = AD[a * kC + b];
#pragma unroll
                for (int j = 0; j < kMaxT; ++j)
                    if (j < nA) acc[j] = fmaf(w, ks[b * ldk + tx + 16 * j], acc[j]);
            }
            if (a < n) {
#pragma unroll
                for (int j = 0; j < kMaxT; ++j)
                    if (j < nA) {
                        const int d = tx + 16 * j;
                        dqh[(size_t)(c0 + a) * Dk + d] = from_f32<T>(acc[j] * dphi_from_phi(qs[a * ldk + d]));
                    }
            }
        }
        // segment reverse-state sums: R += Q~^T P, r += Q~^T g
        for (int a = 0; a < n; ++a) {
            float qd[kMaxT], pm[kMaxT];
#pragma unroll
            for (int x = 0; x < kMaxT; ++x) qd[x] = (x < nA) ? qs[a * ldk + ty + 16 * x] : 0.f;
#pragma unroll
            for (int j = 0; j < kMaxT; ++j) pm[j] = (j < nB) ? ps[a * ldv + tx + 16 * j] : 0.f;
#pragma unroll
            for (int x = 0; x < kMaxT; ++x)
#pragma unroll
                for (int j = 0; j < kMaxT; ++j) r[x][j] = fmaf(qd[x], pm[j], r[x][j]);
        }
        if (tid < Dk)
            for (int a = 0; a < n; ++a) rz = fmaf(gs[a], qs[a * ldk + tid], rz);
        __syncthreads();
        if (kCausal) {  // without the mask the state is the total: no update
            // forward state update
            for (int b = 0; b < n; ++b) {
                float kd[kMaxT], vm[kMaxT];
#pragma unroll
                for (int x = 0; x < kMaxT; ++x) kd[x] = (x < nA) ? ks[b * ldk + ty + 16 * x] : 0.f;
#pragma unroll
                for (int j = 0; j < kMaxT; ++j) vm[j] = (j < nB) ? vs[b * ldv + tx + 16 * j] : 0.f;
#pragma unroll
                for (int x = 0; x < kMaxT; ++x)
#pragma unroll
                    for (int j = 0; j < kMaxT; ++j) s[x][j] = fmaf(kd[x], vm[j], s[x][j]);
            }
#pragma unroll
            for (int x = 0; x < kMaxT; ++x)
#pragma unroll
                for (int j = 0; j < kMaxT; ++j)
                    if (x < nA && j < nB) Ss[(ty + 16 * x) * lds + tx + 16 * j] = s[x][j];
            if (tid < Dk) {
                for (int b = 0; b < n; ++b) zreg += ks[b * ldk + tid];
                zs[tid] = zreg;
            }
        }
    }
    float* out = seg_R + (bh * P + p) * E;
#pragma unroll
    for (int x = 0; x < kMaxT; ++x)
#pragma unroll
        for (int j = 0; j < kMaxT; ++j)
            if (x < nA && j < nB) out[(size_t)(ty + 16 * x) * Dv + tx + 16 * j] = r[x][j];
    if (tid < Dk) out[(size_t)Dk * Dv + tid] = rz;
}

// ---------------------------------------------------------------- backward, reverse sweep
// Chunks of the segment in reverse order, R_next / r_next carried from the
// scanned suffix:  dk = (V R_next^T + 1 r_next^T + D^T Q~) * phi'(k),
// dv = K~ R_next + A^T P, then R_next += Q~^T P, r_next += Q~^T g.
template <typename T, bool kCausal>
__global__ void __launch_bounds__(kThreads, 1)
bwd_reverse_sweep_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                         const T* __restrict__ dout, T* __restrict__ dk, T* __restrict__ dv,
                         const float* __restrict__ seg_R, const float* __restrict__ den_g, int N, int Dk, int Dv,
                         int nchunks, int cps, int P) {
    extern __shared__ __align__(16) char smem_raw[];
    Smem sm{smem_raw};
    const int ldk = Dk + 1, ldv = Dv + 1, lds = Dv + 1;
    float* qs = sm.take((size_t)kC * ldk);
    float* ks = sm.take((size_t)kC * ldk);
    float* vs = sm.take((size_t)kC * ldv);
    float* ps = sm.take((size_t)kC * ldv);
    float* AD = sm.take((size_t)kC * kC);
    float* Rs = sm.take((size_t)Dk * lds);
    float* rs = sm.take((size_t)Dk);
    float* gs = sm.take((size_t)kC);
    float* dens = sm.take((size_t)kC);
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int nA = Dk / 16, nB = Dv / 16;
    const int p = blockIdx.x;
    const size_t bh = blockIdx.y;
    const T* qh = q + bh * N * Dk;
    const T* kh = k + bh * N * Dk;
    const T* vh = v + bh * N * Dv;
    const T* doh = dout + bh * N * Dv;
    T* dkh = dk + bh * N * Dk;
    T* dvh = dv + bh * N * Dv;
    const float* dgh = den_g + bh * N * 2;
    const size_t E = state_elems(Dk, Dv);
    // causal: the segment's exclusive suffix; non-causal: the total over the head (fixed)
    const float* init = kCausal ? seg_R + (bh * P + p) * E : seg_R + bh * E;

    float r[kMaxT][kMaxT];
#pragma unroll
    for (int a = 0; a < kMaxT; ++a)
#pragma unroll
        for (int j = 0; j < kMaxT; ++j) {
            float x = 0.f;
            if (a < nA && j < nB) {
                x = init[(size_t)(ty + 16 * a) * Dv + tx + 16 * j];
                Rs[(ty + 16 * a) * lds + tx + 16 * j] = x;
            }
            r[a][j] = x;
        }
    float rz = 0.f;
    if (tid < Dk) {
        rz = init[(size_t)Dk * Dv + tid];
        rs[tid] = rz;
    }

    const int cbeg = p * cps, cend = min(nchunks, cbeg + cps);

    LA_DCHECK(p < (int)gridDim.x && cbeg < cend && cend <= nchunks && (long long)nchunks * kC < (long long)N + kC);
    for (int c = cend - 1; c >= cbeg; --c) {
        const int c0 = c * kC, n = min(kC, N - c0);
        LA_DCHECK(c0 >= 0 && n >= 1 && c0 + n <= N && blockIdx.y < gridDim.y);
        __syncthreads();
        if (tid < kC) {
            const bool valid = tid < n;
            dens[tid] = valid ? dgh[(size_t)(c0 + tid) * 2 + 0] : 1.f;
            gs[tid] = valid ? dgh[(size_t)(c0 + tid) * 2 + 1] : 0.f;
        }
        load_tile(qs, ldk, qh, c0, n, Dk, true);
        load_tile(ks, ldk, kh, c0, n, Dk, true);
        load_tile(vs, ldv, vh, c0, n, Dv, false);
        load_tile(ps, ldv, doh, c0, n, Dv, false);
        __syncthreads();
        for (int idx = tid; idx < kC * Dv; idx += kThreads) {
            const int a = idx / Dv, m = idx - a * Dv;
            ps[a * ldv + m] /= dens[a];
        }
        __syncthreads();
        // D = tril(P V^T + g 1^T), masked to valid columns
        if (kCausal) {
#pragma unroll
            for (int i = 0; i < kC / 16; ++i)
#pragma unroll
                for (int j = 0; j < kC / 16; ++j) {
                    const int a = ty + 16 * i, b = tx + 16 * j;
                    float acc = 0.f;
                    for (int m = 0; m < Dv; ++m) acc = fmaf(ps[a * ldv + m], vs[b * ldv + m], acc);
                    AD[a * kC + b] = (b <= a && b < n) ? acc + gs[a] : 0.f;
                }
        }
        __syncthreads();
        // dk = (V R^T + r + D^T Q~) * phi'(k)  (no D^T Q~ term without the mask: R, r are totals)
#pragma unroll 1
        for (int i = 0; i < kC / 16; ++i) {
            const int b = ty + 16 * i;
            float acc[kMaxT];
#pragma unroll
            for (int j = 0; j < kMaxT; ++j) acc[j] = (j < nA) ? rs[tx + 16 * j] : 0.f;
            for (int m = 0; m < Dv; ++m) {
                const float vm = vs[b * ldv + m];
#pragma unroll
                for (int j = 0; j < kMaxT; ++j)
                    if (j < nA) acc[j] = fmaf(vm, Rs[(tx + 16 * j) * lds + m], acc[j]);
            }
            for (int a = b; kCausal && a < kC; ++a) {
                const float w = AD[a * kC + b];
#pragma unroll
                for (int j = 0; j < kMaxT; ++j)
                    if (j < nA) acc[j] = fmaf(w, qs[a * ldk + tx + 16 * j], acc[j]);
            }
            if (b < n) {
#pragma unroll
                for (int j = 0; j < kMaxT; ++j)
                    if (j < nA) {
                        const int d = tx + 16 * j;
                        dkh[(size_t)(c0 + b) * Dk + d] = from_f32<T>(acc[j] * dphi_from_phi(ks[b * ldk + d]));
                    }
            }
        }
        __syncthreads();
        // A = tril(Q~ K~^T)
        if (kCausal) {
#pragma unroll
            for (int i = 0; i < kC / 16; ++i)
#pragma unroll
                for (int j = 0; j < kC / 16; ++j) {
                    const int a = ty + 16 * i, b = tx + 16 * j;
                    float acc = 0.f;
                    for (int d = 0; d < Dk; ++d) acc = fmaf(qs[a * ldk + d], ks[b * ldk + d], acc);
                    AD[a * kC + b] = (b <= a) ? acc : 0.f;
                }
        }
        __syncthreads();
        // dv = K~ R + A^T P
#pragma unroll 1
        for (int i = 0; i < kC / 16; ++i) {
            const int b = ty + 16 * i;
            float acc[kMaxT];
#pragma unroll
            for (int j = 0; j < kMaxT; ++j) acc[j] = 0.f;
            for (int d = 0; d < Dk; ++d) {
                const float kd = ks[b * ldk + d];
#pragma unroll
                for (int j = 0; j < kMaxT; ++j)
                    if (j < nB) acc[j] = fmaf(kd, Rs[d * lds + tx + 16 * j], acc[j]);
            }
            for (int a = b; kCausal && a < kC; ++a) {
                const float w = AD[a * kC + b];
#pragma unroll
                for (int j = 0; j < kMaxT; ++j)
                    if (j < nB) acc[j] = fmaf(w, ps[a * ldv + tx + 16 * j], acc[j]);
            }
            if (b < n) {
#pragma unroll
                for (int j = 0; j < kMaxT; ++j)
                    if (j < nB) dvh[(size_t)(c0 + b) * Dv + tx + 16 * j] = from_f32<T>(acc[j]);
            }
        }
        __syncthreads();
        if (kCausal) {  // without the mask R, r are the totals: no update
            // R += Q~^T P, r += Q~^T g
            for (int a = 0; a < n; ++a) {
                float qd[kMaxT], pm[kMaxT];
#pragma unroll
                for (int x = 0; x < kMaxT; ++x) qd[x] = (x < nA) ? qs[a * ldk + ty + 16 * x] : 0.f;
#pragma unroll
                for (int j = 0; j < kMaxT; ++j) pm[j] = (j < nB) ? ps[a * ldv + tx + 16 * j] : 0.f;
#pragma unroll
                for (int x = 0; x < kMaxT; ++x)
#pragma unroll
                    for (int j = 0; j < kMaxT; ++j) r[x][j] = fmaf(qd[x], pm[j], r[x][j]);
            }
#pragma unroll
            for (int x = 0; x < kMaxT; ++x)
#pragma unroll
                for (int j = 0; j < kMaxT; ++j)
                    if (x < nA && j < nB) Rs[(ty + 16 * x) * lds + tx + 16 * j] = r[x][j];
            if (tid < Dk) {
                for (int a = 0; a < n; ++a) rz = fmaf(gs[a], qs[a * ldk + tid], rz);
                rs[tid] = rz;
            }
        }
    }
}

// ---------------------------------------------------------------- host side
size_t smem_floats_fwd(int Dk, int Dv) {
    auto r = [](size_t n) { return ((n * 4 + 15) / 16) * 16; };
    return r((size_t)kC * (Dk + 1)) * 2 + r((size_t)kC * (Dv + 1)) + r((size_t)kC * kC) + r((size_t)Dk * (Dv + 1)) +
           r(Dk);
}
size_t smem_bytes_sums(int Dk, int Dv) {
    auto r = [](size_t n) { return ((n * 4 + 15) / 16) * 16; };
    return r((size_t)kC * (Dk + 1)) + r((size_t)kC * (Dv + 1));
}
size_t smem_bytes_apply(int Dk, int Dv) {
    auto r = [](size_t n) { return ((n * 4 + 15) / 16) * 16; };
    return r((size_t)kC * (Dk + 1)) + r((size_t)Dk * Dv) + r(Dk);
}
size_t smem_bytes_bwd(int Dk, int Dv) {
    auto r = [](size_t n) { return ((n * 4 + 15) / 16) * 16; };
    return r((size_t)kC * (Dk + 1)) * 2 + r((size_t)kC * (Dv + 1)) * 2 + r((size_t)kC * kC) +
           r((size_t)Dk * (Dv + 1)) + r(Dk) + r(kC) * 2;
}

template <typename K>
cudaError_t allow_smem(K kernel, size_t bytes) {
    // Opt in to large dynamic shared memory (the attribute is per kernel and idempotent).
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

#define LA_DISPATCH_DTYPE(dt, T, ...)                 \
    do {                                              \
        if ((dt) == LA_BF16) {                        \
            using T = __nv_bfloat16;                  \
            __VA_ARGS__;                              \
        } else {                                      \
            using T = float;                          \
            __VA_ARGS__;                              \
        }                                             \
    } while (0)

cudaError_t simt_segment_sums(const void* k, const void* v, float* seg, const la_shape& s, const Plan& p,
                              cudaStream_t st) {
    const size_t smem = smem_bytes_sums(s.Dk, s.Dv);
    dim3 grid(p.P, s.B * s.H);
    cudaError_t err = cudaSuccess;
    LA_DISPATCH_DTYPE(s.dtype, T, {
        auto kern = segment_sums_kernel<T>;
        if ((err = allow_smem(kern, smem)) != cudaSuccess) return err;
        launch_begin("simt_segment_sums", st);
        kern<<<grid, kThreads, smem, st>>>((const T*)k, (const T*)v, seg, s.N, s.Dk, s.Dv, p.nchunks, p.cps, p.P);
        err = launch_end("simt_segment_sums", st);
    });
    return err;
}

// totals: [BH][E] records (the non-causal path, whose records are unpadded).
cudaError_t scan_segments(float* seg, float* totals, const la_shape& s, const Plan& p, int mode, cudaStream_t st) {
    const size_t E = plan_state_elems(p);  // a multiple of 16 for the supported head sizes
    const size_t SkSv = (size_t)p.sk * p.sv;
    dim3 grid((unsigned)((E / 4 + 127) / 128), s.B * s.H);
    launch_begin("scan_segments", st);
    const cudaError_t e = launch_pdl(scan_kernel, grid, dim3(128), 0, st, seg, totals,
                                     totals ? totals + SkSv : (float*)nullptr, E, E, p.P, E, p.sk, p.sv, p.sk, p.sv,
                                     mode);
    const cudaError_t e2 = launch_end("scan_segments", st);
    return e != cudaSuccess ? e : e2;
}

cudaError_t scan_segments_unpadded_totals(float* seg, float* totals, const la_shape& s, const Plan& p,
                                          cudaStream_t st) {
    const size_t E = plan_state_elems(p), Eu = state_elems(s.Dk, s.Dv);
    dim3 grid((unsigned)((E / 4 + 127) / 128), s.B * s.H);
    launch_begin("scan_segments", st);
    scan_kernel<<<grid, 128, 0, st>>>(seg, totals, totals + (size_t)s.Dk * s.Dv, Eu, Eu, p.P, E, p.sk, p.sv, s.Dk,
                                      s.Dv, SCAN_TOTAL);
    return launch_end("scan_segments", st);
}

cudaError_t scan_segments_final_state(float* seg, float* S_out, float* z_out, const la_shape& s, const Plan& p,
                                      cudaStream_t st) {
    const size_t E = plan_state_elems(p);
    dim3 grid((unsigned)((E / 4 + 127) / 128), s.B * s.H);
    launch_begin("scan_segments", st);
    scan_kernel<<<grid, 128, 0, st>>>(seg, S_out, z_out, (size_t)s.Dk * s.Dv, (size_t)s.Dk, p.P, E, p.sk, p.sv, s.Dk,
                                      s.Dv, SCAN_EXCLUSIVE_PREFIX);
    return launch_end("scan_segments", st);
}

cudaError_t simt_causal_fwd_out(const void* q, const void* k, const void* v, void* o, const float* seg,
                                const la_shape& s, const Plan& p, cudaStream_t st) {
    const size_t smem = smem_floats_fwd(s.Dk, s.Dv);
    dim3 grid(p.P, s.B * s.H);
    cudaError_t err = cudaSuccess;
    LA_DISPATCH_DTYPE(s.dtype, T, {
        auto kern = causal_fwd_out_kernel<T>;
        if ((err = allow_smem(kern, smem)) != cudaSuccess) return err;
        launch_begin("simt_causal_fwd_out", st);
        kern<<<grid, kThreads, smem, st>>>((const T*)q, (const T*)k, (const T*)v, (T*)o, seg, s.N, s.Dk, s.Dv,
                                           p.nchunks, p.cps, p.P);
        err = launch_end("simt_causal_fwd_out", st);
    });
    return err;
}

cudaError_t simt_noncausal_apply(const void* q, void* o, const float* totals, const la_shape& s, cudaStream_t st) {
    const size_t smem = smem_bytes_apply(s.Dk, s.Dv);
    dim3 grid((s.N + kC - 1) / kC, s.B * s.H);
    cudaError_t err = cudaSuccess;
    LA_DISPATCH_DTYPE(s.dtype, T, {
        auto kern = noncausal_apply_kernel<T>;
        if ((err = allow_smem(kern, smem)) != cudaSuccess) return err;
        launch_begin("simt_noncausal_apply", st);
        kern<<<grid, kThreads, smem, st>>>((const T*)q, (T*)o, totals, s.N, s.Dk, s.Dv);
        err = launch_end("simt_noncausal_apply", st);
    });
    return err;
}

cudaError_t simt_bwd_forward_sweep(const void* q, const void* k, const void* v, const void* dout, void* dq,
                                   const float* seg_S, float* seg_R, float* den_g, const la_shape& s, const Plan& p,
                                   cudaStream_t st, bool causal) {
    const size_t smem = smem_bytes_bwd(s.Dk, s.Dv);
    dim3 grid(p.P, s.B * s.H);
    cudaError_t err = cudaSuccess;
    LA_DISPATCH_DTYPE(s.dtype, T, {
        auto kern = causal ? bwd_forward_sweep_kernel<T, true> : bwd_forward_sweep_kernel<T, false>;
        if ((err = allow_smem(kern, smem)) != cudaSuccess) return err;
        launch_begin(causal ? "simt_bwd_forward_sweep" : "simt_noncausal_bwd_query", st);
        kern<<<grid, kThreads, smem, st>>>((const T*)q, (const T*)k, (const T*)v, (const T*)dout, (T*)dq, seg_S,
                                           seg_R, den_g, s.N, s.Dk, s.Dv, p.nchunks, p.cps, p.P);
        err = launch_end(causal ? "simt_bwd_forward_sweep" : "simt_noncausal_bwd_query", st);
    });
    return err;
}

cudaError_t simt_bwd_reverse_sweep(const void* q, const void* k, const void* v, const void* dout, void* dk, void* dv,
                                   const float* seg_R, const float* den_g, const la_shape& s, const Plan& p,
                                   cudaStream_t st, bool causal) {
    const size_t smem = smem_bytes_bwd(s.Dk, s.Dv) + 256;
    dim3 grid(p.P, s.B * s.H);
    cudaError_t err = cudaSuccess;
    LA_DISPATCH_DTYPE(s.dtype, T, {
        auto kern = causal ? bwd_reverse_sweep_kernel<T, true> : bwd_reverse_sweep_kernel<T, false>;
        if ((err = allow_smem(kern, smem)) != cudaSuccess) return err;
        launch_begin(causal ? "simt_bwd_reverse_sweep" : "simt_noncausal_bwd_key", st);
        kern<<<grid, kThreads, smem, st>>>((const T*)q, (const T*)k, (const T*)v, (const T*)dout, (T*)dk, (T*)dv,
                                           seg_R, den_g, s.N, s.Dk, s.Dv, p.nchunks, p.cps, p.P);
        err = launch_end(causal ? "simt_bwd_reverse_sweep" : "simt_noncausal_bwd_key", st);
    });
    return err;
}

}  // namespace la
