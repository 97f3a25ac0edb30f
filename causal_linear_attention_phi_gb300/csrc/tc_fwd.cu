// tc_fwd.cu -- tensor-core (tcgen05 / TMEM / TMA) kernels of the chunked causal
// forward for bf16 inputs with Dk = Dv = 128 and chunks of C = 128 positions.
//
// Per chunk c of a segment ("선형 어텐션" (itwiki), 계산 형태 비교: matrix
// products inside a chunk, the state passed between chunks):
//   QK   = phi(Q_c) phi(K_c)^T                      tcgen05, TMEM fp32 (128 x 128)
//   A    = tril(QK)  -> bf16, written back to TMEM   compute warpgroup
//   O    = phi(Q_c) S_prev + A V_c                   tcgen05, TMEM fp32 (128 x 128)
//   den  = phi(Q_c) z_prev + A 1                     CUDA cores, fp32
//   o    = O / den -> bf16 -> global                 compute warpgroup
//   S   += phi(K_c)^T V_c,  z += phi(K_c)^T 1         tcgen05 (S in TMEM), CUDA cores (z)
// S_prev enters the O product as a bf16 copy in shared memory, refreshed from
// the fp32 TMEM state after every chunk.  phi is applied in place to the
// TMA-staged Q and K tiles (fused into the tile load).
//
// The same kernel with kOut = false only accumulates the segment's sums
// (S, z) for the segment scan.
//
// Roles (192 threads): warp 0 issues TMA loads, warp 1 owns TMEM and issues
// tcgen05.mma, warps 2-5 (a warpgroup) transform tiles, mask A, refresh S_prev
// and write outputs.  Warp w of the warpgroup reads TMEM lanes 32*(w%4)...
// Every wait is bounded: on timeout the kernel records LA_ERR_TIMEOUT in the
// sticky error word and all roles leave their loops.
#include <cudaTypedefs.h>

#include <mutex>

#include "la_internal.cuh"
#include "sm100.cuh"

namespace la {
namespace {
using namespace sm100;

constexpr int kC = 128;          // chunk length
constexpr int kD = 128;          // Dk = Dv
constexpr int kTileBytes = 32768;   // 128 rows x 128 bf16, as two 64-column swizzled blocks
constexpr int kBlockBytes = 16384;  // one 64-column block (128 rows x 128 B)
constexpr int kThreads = 192;

// TMEM column map (512 columns allocated)
constexpr uint32_t kTmS = 0, kTmQK = 128, kTmO = 256, kTmA = 384;

struct __align__(8) Barriers {
    uint64_t q_full, q_empty;
    uint64_t kv_full[2], kv_empty[2];
    uint64_t qk_ready[2], sb_ready, a_ready;  // qk_ready per K/V stage: its producer may run one chunk ahead
    uint64_t qk_done, o_done, s_done;
    uint64_t final_mma;
};

struct SmemLayout {
    // offsets from the 1024-aligned base
    static constexpr int Q = 0;
    static constexpr int K0 = Q + kTileBytes;
    static constexpr int K1 = K0 + kTileBytes;
    static constexpr int V0 = K1 + kTileBytes;
    static constexpr int V1 = V0 + kTileBytes;
    static constexpr int Sb = V1 + kTileBytes;
    static constexpr int zsh = Sb + kTileBytes;       // float[128]: z before the current chunk
    static constexpr int zchunk = zsh + 512;          // float[128]: this chunk's sum of phi(k)
    static constexpr int bars = zchunk + 512;
    static constexpr int tmem_slot = bars + 256;
    static constexpr int total = tmem_slot + 16;
};
constexpr size_t kSmemBytes = SmemLayout::total + 1024;  // + alignment slack

__device__ __forceinline__ bool wg_all(bool v) {
    // barrier over the 128-thread compute warpgroup (id 1) that also ANDs a predicate
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ void wg_sync() { named_barrier(1, 128); }

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Apply phi in place to a 128 x 128 bf16 tile (two swizzled 64-column blocks),
// zeroing rows >= n.  With `zpart`, also accumulate the per-column sums of the
// rounded phi values.  Thread t (0..127) touches 16-byte vectors t + 128 j:
// block j / 8, row ((t >> 3) + 16 j) & 127, physical chunk t & 7, whose
// logical chunk (columns 8*lc .. 8*lc + 7 of the block) is (t & 7) ^ (row & 7).
template <bool kZ>
__device__ __forceinline__ void phi_tile(uint8_t* tile, int t, int n, float (&zp)[2][8]) {
#pragma unroll 4
    for (int j = 0; j < 16; ++j) {
        const int blk = j >> 3;
        const int row = ((t >> 3) + 16 * j) & 127;
        uint4* p = reinterpret_cast<uint4*>(tile + blk * kBlockBytes + row * 128 + (t & 7) * 16);
        uint4 w = *p;
        uint32_t* u = reinterpret_cast<uint32_t*>(&w);
        const bool valid = row < n;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            float a = valid ? phi_f(bf_lo(u[e])) : 0.f;
            float b = valid ? phi_f(bf_hi(u[e])) : 0.f;
            u[e] = pack_bf16x2(a, b);
            if (kZ) {
                zp[blk][2 * e] += bf_lo(u[e]);
                zp[blk][2 * e + 1] += bf_hi(u[e]);
            }
        }
        *p = w;
    }
}

template <bool kOut>
__global__ void __launch_bounds__(kThreads, 1)
tc_causal_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, __nv_bfloat16* __restrict__ o,
                     float* __restrict__ seg, int N, int nchunks, int cps, int P, int* err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = base + SmemLayout::Q;
    uint8_t* sK[2] = {base + SmemLayout::K0, base + SmemLayout::K1};
    uint8_t* sV[2] = {base + SmemLayout::V0, base + SmemLayout::V1};
    uint8_t* sSb = base + SmemLayout::Sb;
    float* zsh = reinterpret_cast<float*>(base + SmemLayout::zsh);
    float* zchunk = reinterpret_cast<float*>(base + SmemLayout::zchunk);
    Barriers* bar = reinterpret_cast<Barriers*>(base + SmemLayout::bars);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + SmemLayout::tmem_slot);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int p = blockIdx.x, bh = blockIdx.y;
    const int cbeg = p * cps, cend = min(nchunks, cbeg + cps), nloc = cend - cbeg;
    const size_t E = state_elems(kD, kD);
    float* segp = seg + ((size_t)bh * P + p) * E;

    if (tid == 0) {
        mbar_init(&bar->q_full, 1);
        mbar_init(&bar->q_empty, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bar->kv_full[s], 1);
            mbar_init(&bar->kv_empty[s], 1);
        }
        mbar_init(&bar->qk_ready[0], 1);
        mbar_init(&bar->qk_ready[1], 1);
        mbar_init(&bar->sb_ready, 1);
        mbar_init(&bar->a_ready, 1);
        mbar_init(&bar->qk_done, 1);
        mbar_init(&bar->o_done, 1);
        mbar_init(&bar->s_done, 1);
        mbar_init(&bar->final_mma, 1);
        fence_mbar_init();
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        if (kOut) tma_prefetch_desc(&tm_q);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int armed_kv[2] = {-1, -1}, armed_q = -1;
            bool ok = true;
            for (int i = 0; i < nloc && ok; ++i) {
                const int s = i & 1, t0 = (cbeg + i) * kC;
                ok = mbar_wait(&bar->kv_empty[s], ((i >> 1) & 1) ^ 1, err, LA_ERR_TIMEOUT);
                if (!ok) break;
                mbar_arrive_expect_tx(&bar->kv_full[s], 2 * kTileBytes);
                tma_load_3d(sK[s], &tm_k, 0, t0, bh, &bar->kv_full[s]);
                tma_load_3d(sK[s] + kBlockBytes, &tm_k, 64, t0, bh, &bar->kv_full[s]);
                tma_load_3d(sV[s], &tm_v, 0, t0, bh, &bar->kv_full[s]);
                tma_load_3d(sV[s] + kBlockBytes, &tm_v, 64, t0, bh, &bar->kv_full[s]);
                armed_kv[s] = i;
                if (kOut) {
                    ok = mbar_wait(&bar->q_empty, (i & 1) ^ 1, err, LA_ERR_TIMEOUT);
                    if (!ok) break;
                    mbar_arrive_expect_tx(&bar->q_full, kTileBytes);
                    tma_load_3d(sQ, &tm_q, 0, t0, bh, &bar->q_full);
                    tma_load_3d(sQ + kBlockBytes, &tm_q, 64, t0, bh, &bar->q_full);
                    armed_q = i;
                }
            }
            // never leave with copies in flight: wait for the last armed phase of each buffer
            for (int s = 0; s < 2; ++s)
                if (armed_kv[s] >= 0) mbar_wait(&bar->kv_full[s], (armed_kv[s] >> 1) & 1, err, LA_ERR_TIMEOUT);
            if (armed_q >= 0) mbar_wait(&bar->q_full, armed_q & 1, err, LA_ERR_TIMEOUT);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t id_qk = idesc_bf16_f32(128, 128, 0, 0);
            constexpr uint32_t id_kmn = idesc_bf16_f32(128, 128, 0, 1);
            constexpr uint32_t id_mnmn = idesc_bf16_f32(128, 128, 1, 1);
            const uint32_t q_addr = smem_u32(sQ), sb_addr = smem_u32(sSb);
            bool ok = true;
            for (int i = 0; i < nloc && ok; ++i) {
                const int s = i & 1;
                const uint32_t k_addr = smem_u32(sK[s]), v_addr = smem_u32(sV[s]);
                if (!(ok = mbar_wait(&bar->qk_ready[s], (i >> 1) & 1, err, LA_ERR_TIMEOUT))) break;
                tc_fence_after();
                if (kOut) {
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t off = (kk >> 2) * kBlockBytes + (kk & 3) * 32;
                        mma_ss(tmem + kTmQK, smem_desc_sw128(q_addr + off, 16, 1024),
                               smem_desc_sw128(k_addr + off, 16, 1024), id_qk, kk > 0);
                    }
                    mma_commit(&bar->qk_done);
                    if (!(ok = mbar_wait(&bar->sb_ready, i & 1, err, LA_ERR_TIMEOUT))) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t off = (kk >> 2) * kBlockBytes + (kk & 3) * 32;
                        mma_ss(tmem + kTmO, smem_desc_sw128(q_addr + off, 16, 1024),
                               smem_desc_sw128(sb_addr + kk * 2048, kBlockBytes, 1024), id_kmn, kk > 0);
                    }
                    mma_commit(&bar->q_empty);
                    if (!(ok = mbar_wait(&bar->a_ready, i & 1, err, LA_ERR_TIMEOUT))) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_ts(tmem + kTmO, tmem + kTmA + 8 * kk,
                               smem_desc_sw128(v_addr + kk * 2048, kBlockBytes, 1024), id_kmn, 1);
                    mma_commit(&bar->o_done);
                }
                // S += phi(K)^T V  (K tile read as an MN-major A operand)
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ss(tmem + kTmS, smem_desc_sw128(k_addr + kk * 2048, kBlockBytes, 1024),
                           smem_desc_sw128(v_addr + kk * 2048, kBlockBytes, 1024), id_mnmn,
                           (kOut || i > 0 || kk > 0) ? 1u : 0u);
                mma_commit(&bar->s_done);
                mma_commit(&bar->kv_empty[s]);
            }
            // drain: every MMA this thread issued has completed before TMEM is released
            mma_commit(&bar->final_mma);
            mbar_wait(&bar->final_mma, 0, err, LA_ERR_TIMEOUT);
        }
    } else {
        // ------------------------------------------------------------ compute warpgroup
        const int t = tid - 64;                       // 0..127
        const int r = 32 * (warp & 3) + lane;         // TMEM lane / tile row owned by this thread
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        // initial state: S_prev from the scanned segment prefix (kOut), z likewise
        if (kOut) {
            const float* pre = segp + (size_t)r * kD;
#pragma unroll
            for (int cb = 0; cb < 4; ++cb) {
                uint32_t w[32];
#pragma unroll
                for (int x = 0; x < 32; ++x) w[x] = __float_as_uint(pre[32 * cb + x]);
                tmem_st32(tmem + lane_base + kTmS + 32 * cb, w);
            }
            tmem_st_wait();
            zsh[r] = segp[(size_t)kD * kD + r];
        } else {
            zsh[r] = 0.f;
        }
        zchunk[r] = 0.f;
        tc_fence_before();
        bool ok = wg_all(true);
        for (int i = 0; i < nloc && ok; ++i) {
            const int s = i & 1;
            const int c0 = (cbeg + i) * kC, n = min(kC, N - c0);
            // (a) phi on the K (and Q) tiles, z partial sums
            ok = mbar_wait(&bar->kv_full[s], (i >> 1) & 1, err, LA_ERR_TIMEOUT);
            if (kOut) ok = ok && mbar_wait(&bar->q_full, i & 1, err, LA_ERR_TIMEOUT);
            if (!wg_all(ok)) { ok = false; break; }
            float zp[2][8];
#pragma unroll
            for (int b = 0; b < 2; ++b)
#pragma unroll
                for (int e = 0; e < 8; ++e) zp[b][e] = 0.f;
            phi_tile<true>(sK[s], t, n, zp);
            {
                const int lc = (t & 7) ^ ((t >> 3) & 7);
#pragma unroll
                for (int b = 0; b < 2; ++b)
#pragma unroll
                    for (int e = 0; e < 8; ++e) atomicAdd(&zchunk[64 * b + 8 * lc + e], zp[b][e]);
            }
            float den_inter = 0.f;
            if (kOut) {
                float dummy[2][8];
                phi_tile<false>(sQ, t, kC, dummy);
            }
            fence_proxy_async_smem();
            wg_sync();
            if (t == 0) mbar_arrive(&bar->qk_ready[s]);
            if (kOut) {
                // den_inter = phi(q_r) . z_prev from this thread's Q row
#pragma unroll
                for (int b = 0; b < 2; ++b)
#pragma unroll
                    for (int lc = 0; lc < 8; ++lc) {
                        const uint4 w = *reinterpret_cast<const uint4*>(sQ + b * kBlockBytes + r * 128 +
                                                                        ((lc ^ (r & 7)) * 16));
                        const uint32_t* u = reinterpret_cast<const uint32_t*>(&w);
                        const float* zz = zsh + 64 * b + 8 * lc;
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            den_inter += bf_lo(u[e]) * zz[2 * e] + bf_hi(u[e]) * zz[2 * e + 1];
                    }
                // (b) S_prev -> bf16 B operand (MN-major: row = dk = r, 64-wide dv blocks)
                if (i > 0) {
                    ok = mbar_wait(&bar->s_done, (i - 1) & 1, err, LA_ERR_TIMEOUT);
                    if (!wg_all(ok)) { ok = false; break; }
                    tc_fence_after();
                }
#pragma unroll
                for (int cb = 0; cb < 4; ++cb) {
                    uint32_t w[32];
                    tmem_ld32(tmem + lane_base + kTmS + 32 * cb, w);
                    tmem_ld_wait();
                    // columns 32cb .. 32cb+31 = dv; block cb/2, logical chunks 4*(cb&1) .. +3
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const int lc = 4 * (cb & 1) + q4;
                        uint4 v4;
                        v4.x = pack_bf16x2(__uint_as_float(w[8 * q4 + 0]), __uint_as_float(w[8 * q4 + 1]));
                        v4.y = pack_bf16x2(__uint_as_float(w[8 * q4 + 2]), __uint_as_float(w[8 * q4 + 3]));
                        v4.z = pack_bf16x2(__uint_as_float(w[8 * q4 + 4]), __uint_as_float(w[8 * q4 + 5]));
                        v4.w = pack_bf16x2(__uint_as_float(w[8 * q4 + 6]), __uint_as_float(w[8 * q4 + 7]));
                        *reinterpret_cast<uint4*>(sSb + (cb >> 1) * kBlockBytes + r * 128 + ((lc ^ (r & 7)) * 16)) =
                            v4;
                    }
                }
                tc_fence_before();
                fence_proxy_async_smem();
                wg_sync();
                if (t == 0) mbar_arrive(&bar->sb_ready);
                // (c) A = tril(QK) -> bf16 into TMEM; row sums for den
                ok = mbar_wait(&bar->qk_done, i & 1, err, LA_ERR_TIMEOUT);
                if (!wg_all(ok)) { ok = false; break; }
                tc_fence_after();
                float rs = 0.f;
#pragma unroll
                for (int cb = 0; cb < 4; ++cb) {
                    uint32_t w[32];
                    tmem_ld32(tmem + lane_base + kTmQK + 32 * cb, w);
                    tmem_ld_wait();
                    uint32_t pk[16];
#pragma unroll
                    for (int x = 0; x < 16; ++x) {
                        const int j0 = 32 * cb + 2 * x;
                        const float a0 = (j0 <= r) ? __uint_as_float(w[2 * x]) : 0.f;
                        const float a1 = (j0 + 1 <= r) ? __uint_as_float(w[2 * x + 1]) : 0.f;
                        pk[x] = pack_bf16x2(a0, a1);
                        rs += bf_lo(pk[x]) + bf_hi(pk[x]);
                    }
                    tmem_st16(tmem + lane_base + kTmA + 16 * cb, pk);
                }
                tmem_st_wait();
                tc_fence_before();
                wg_sync();
                if (t == 0) mbar_arrive(&bar->a_ready);
                // (d) o = O / den
                ok = mbar_wait(&bar->o_done, i & 1, err, LA_ERR_TIMEOUT);
                if (!wg_all(ok)) { ok = false; break; }
                tc_fence_after();
                const float inv = 1.f / (rs + den_inter);
                __nv_bfloat16* orow = o + ((size_t)bh * N + c0 + r) * kD;
#pragma unroll
                for (int cb = 0; cb < 4; ++cb) {
                    uint32_t w[32];
                    tmem_ld32(tmem + lane_base + kTmO + 32 * cb, w);
                    tmem_ld_wait();
                    if (r < n) {
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            uint4 v4;
                            v4.x = pack_bf16x2(__uint_as_float(w[8 * q4 + 0]) * inv, __uint_as_float(w[8 * q4 + 1]) * inv);
                            v4.y = pack_bf16x2(__uint_as_float(w[8 * q4 + 2]) * inv, __uint_as_float(w[8 * q4 + 3]) * inv);
                            v4.z = pack_bf16x2(__uint_as_float(w[8 * q4 + 4]) * inv, __uint_as_float(w[8 * q4 + 5]) * inv);
                            v4.w = pack_bf16x2(__uint_as_float(w[8 * q4 + 6]) * inv, __uint_as_float(w[8 * q4 + 7]) * inv);
                            *reinterpret_cast<uint4*>(orow + 32 * cb + 8 * q4) = v4;
                        }
                    }
                }
                tc_fence_before();
            }
            // z_prev += this chunk's sums (after every thread has used z_prev)
            wg_sync();
            zsh[r] += zchunk[r];
            zchunk[r] = 0.f;
            wg_sync();
        }
        if (!kOut && ok && nloc > 0) {
            // segment sums out: S from TMEM (row r = dk), z from shared memory.  The
            // MMA thread's single-use drain barrier marks the last S update done.
            ok = mbar_wait(&bar->final_mma, 0, err, LA_ERR_TIMEOUT);
            if (wg_all(ok)) {
                tc_fence_after();
                float* out = segp + (size_t)r * kD;
#pragma unroll
                for (int cb = 0; cb < 4; ++cb) {
                    uint32_t w[32];
                    tmem_ld32(tmem + lane_base + kTmS + 32 * cb, w);
                    tmem_ld_wait();
#pragma unroll
                    for (int x = 0; x < 32; x += 4)
                        *reinterpret_cast<float4*>(out + 32 * cb + x) =
                            make_float4(__uint_as_float(w[x]), __uint_as_float(w[x + 1]), __uint_as_float(w[x + 2]),
                                        __uint_as_float(w[x + 3]));
                }
                segp[(size_t)kD * kD + r] = zsh[r];
            }
        }
        tc_fence_before();
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

}  // namespace

// A [BH][N][128] bf16 tensor as a 3-D TMA map with 64 x 128 x 1 boxes and the
// 128-byte swizzle; rows past N inside a head read as zeros.
bool make_tmap_bf16_rows(CUtensorMap* map, const void* ptr, int BH, int N, int D, int box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)N, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)D * 2 * (cuuint64_t)N};
    cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t tc_causal_fwd(const void* q, const void* k, const void* v, void* o, float* seg, const la_shape& s,
                          const Plan& p, bool out_pass, cudaStream_t st) {
    const int BH = s.B * s.H;
    CUtensorMap tq, tk, tv;
    if (!make_tmap_bf16_rows(&tk, k, BH, s.N, kD, kC) || !make_tmap_bf16_rows(&tv, v, BH, s.N, kD, kC) ||
        !make_tmap_bf16_rows(&tq, q ? q : k, BH, s.N, kD, kC))
        return cudaErrorInvalidValue;
    int* err = device_error_word();
    dim3 grid(p.P, BH);
    cudaError_t e;
    if (out_pass) {
        auto kern = tc_causal_fwd_kernel<true>;
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes)) !=
            cudaSuccess)
            return e;
        launch_begin("tc_causal_fwd_out", st);
        kern<<<grid, kThreads, kSmemBytes, st>>>(tq, tk, tv, (__nv_bfloat16*)o, seg, s.N, p.nchunks, p.cps, p.P, err);
        return launch_end("tc_causal_fwd_out", st);
    }
    auto kern = tc_causal_fwd_kernel<false>;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes)) != cudaSuccess)
        return e;
    launch_begin("tc_segment_sums", st);
    kern<<<grid, kThreads, kSmemBytes, st>>>(tq, tk, tv, nullptr, seg, s.N, p.nchunks, p.cps, p.P, err);
    return launch_end("tc_segment_sums", st);
}

}  // namespace la
