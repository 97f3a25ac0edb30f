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
// Roles (320 threads): warp 0 issues TMA loads, warp 1 owns TMEM and issues
// tcgen05.mma, warps 2-9 (two warpgroups) transform tiles, mask A, refresh
// S_prev and write outputs.  Warp w reads TMEM lanes 32*(w%4) ..
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
constexpr int kThreads = 320;  // warp 0 TMA, warp 1 MMA, warps 2-9 compute

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
    static constexpr int K0 = Q + kTileBytes;       // K stages 0, 1
    static constexpr int V0 = K0 + 2 * kTileBytes;  // V stages 0, 1
    static constexpr int Sb = V0 + 2 * kTileBytes;
    static constexpr int zsh = Sb + kTileBytes;     // float[128]
    static constexpr int zpart = zsh + 512;         // float[2][128]
    static constexpr int rpart = zpart + 1024;      // float[2][128]
    static constexpr int dpart = rpart + 1024;      // float[2][128]
    static constexpr int bars = dpart + 1024;
    static constexpr int tmem_slot = bars + 256;
    static constexpr int total = tmem_slot + 16;
};
constexpr size_t kSmemBytes = SmemLayout::total + 1024;  // + alignment slack

// The compute group is two warpgroups (warps 2-9, 256 threads).  Warp w reads
// TMEM lanes 32*(w%4) .. +31 (row r of a 128-row tile); warps 2-5 take columns
// 0-63 of their rows and warps 6-9 columns 64-127, so each row is split
// between two threads whose partial row reductions meet in shared memory.
constexpr int kComputeThreads = 256;

__device__ __forceinline__ bool cg_all(bool v) {
    // barrier over the compute group (named barrier 1) that also ANDs a predicate
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, 256, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ void cg_sync() { named_barrier(1, kComputeThreads); }

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Byte offset of logical 16-byte chunk lc (0..15) of `row` in a swizzled tile.
__device__ __forceinline__ int chunk_off(int row, int lc) {
    return (lc >> 3) * kBlockBytes + row * 128 + (((lc & 7) ^ (row & 7)) << 4);
}

// phi in place on a staged 128 x 128 bf16 tile, rows >= n set to exactly 0.
// Compute thread ct (0..255) handles vectors ct + 256 j, j < 8: block j / 4,
// row ((ct >> 3) + 32 j) & 127, physical chunk ct & 7 (an elementwise map
// ignores the swizzle, which only permutes chunks within a row).
__device__ __forceinline__ void phi_tile(uint8_t* tile, int ct, int n) {
#pragma unroll 4
    for (int j = 0; j < 8; ++j) {
        const int row = ((ct >> 3) + 32 * j) & 127;
        uint4* p = reinterpret_cast<uint4*>(tile + (j >> 2) * kBlockBytes + row * 128 + (ct & 7) * 16);
        uint4 w = *p;
        uint32_t* u = reinterpret_cast<uint32_t*>(&w);
        const bool valid = row < n;
#pragma unroll
        for (int e = 0; e < 4; ++e) u[e] = valid ? pack_bf16x2(phi_f(bf_lo(u[e])), phi_f(bf_hi(u[e]))) : 0u;
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
    uint8_t* sSb = base + SmemLayout::Sb;
    float* zsh = reinterpret_cast<float*>(base + SmemLayout::zsh);       // [128] z before the chunk
    float* zpart = reinterpret_cast<float*>(base + SmemLayout::zpart);   // [2][128] this chunk's column sums
    float* rpart = reinterpret_cast<float*>(base + SmemLayout::rpart);   // [2][128] row partials of A 1
    float* dpart = reinterpret_cast<float*>(base + SmemLayout::dpart);   // [2][128] row partials of phi(q).z
    Barriers* bar = reinterpret_cast<Barriers*>(base + SmemLayout::bars);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + SmemLayout::tmem_slot);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int p = blockIdx.x, bh = blockIdx.y;
    const int cbeg = p * cps, cend = min(nchunks, cbeg + cps), nloc = cend - cbeg;
    const size_t E = state_elems(kD, kD);
    float* segp = seg + ((size_t)bh * P + p) * E;
    // K and V stage s live at K0 + s * kTileBytes and V0 + s * kTileBytes
    auto sK = [&](int s) { return base + SmemLayout::K0 + s * kTileBytes; };
    auto sV = [&](int s) { return base + SmemLayout::V0 + s * kTileBytes; };

    if (tid == 0) {
        uint64_t* b = reinterpret_cast<uint64_t*>(bar);
        for (int x = 0; x < (int)(sizeof(Barriers) / 8); ++x) mbar_init(b + x, 1);
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
                tma_load_3d(sK(s), &tm_k, 0, t0, bh, &bar->kv_full[s]);
                tma_load_3d(sK(s) + kBlockBytes, &tm_k, 64, t0, bh, &bar->kv_full[s]);
                tma_load_3d(sV(s), &tm_v, 0, t0, bh, &bar->kv_full[s]);
                tma_load_3d(sV(s) + kBlockBytes, &tm_v, 64, t0, bh, &bar->kv_full[s]);
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
                const uint32_t k_addr = smem_u32(sK(s)), v_addr = smem_u32(sV(s));
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
        // ------------------------------------------------------------ compute group (256 threads)
        const int ct = tid - 64;                       // 0..255
        const int h = (warp - 2) >> 2;                 // column half of the rows this thread serves
        const int r = 32 * (warp & 3) + lane;          // TMEM lane / tile row
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        const int zc = ct & 127, zh = ct >> 7;         // column-sum assignment: column zc, rows of half zh
        if (ct < 128) zsh[ct] = kOut ? segp[(size_t)kD * kD + ct] : 0.f;
        if (kOut) {
            // S_prev from the scanned segment prefix: row r, this thread's 64 columns
            const float* pre = segp + (size_t)r * kD + 64 * h;
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) {
                uint32_t w[32];
#pragma unroll
                for (int x = 0; x < 32; ++x) w[x] = __float_as_uint(pre[32 * cb + x]);
                tmem_st32(tmem + lane_base + kTmS + 64 * h + 32 * cb, w);
            }
            tmem_st_wait();
        }
        tc_fence_before();
        bool ok = cg_all(true);
        for (int i = 0; i < nloc && ok; ++i) {
            const int s = i & 1;
            const int c0 = (cbeg + i) * kC, n = min(kC, N - c0);
            uint8_t* kt = sK(s);
            // (a) phi on the K (and Q) tiles
            bool w = mbar_wait(&bar->kv_full[s], (i >> 1) & 1, err, LA_ERR_TIMEOUT);
            if (kOut) w = w && mbar_wait(&bar->q_full, i & 1, err, LA_ERR_TIMEOUT);
            if (!cg_all(w)) { ok = false; break; }
            phi_tile(kt, ct, n);
            if (kOut) phi_tile(sQ, ct, n);
            fence_proxy_async_smem();
            cg_sync();
            if (ct == 0) mbar_arrive(&bar->qk_ready[s]);
            {
                // this chunk's column sums of phi(K), rows [64 zh, 64 zh + 64) of column zc
                float acc = 0.f;
                const int rend = min(64 * zh + 64, n);
                for (int row = 64 * zh; row < rend; ++row) {
                    const uint16_t hv =
                        *reinterpret_cast<const uint16_t*>(kt + chunk_off(row, zc >> 3) + ((zc & 7) << 1));
                    acc += __uint_as_float((uint32_t)hv << 16);
                }
                zpart[zh * 128 + zc] = acc;
            }
            if (kOut) {
                // den partial: phi(q_r) . z_prev over this thread's 64 columns
                float di = 0.f;
#pragma unroll
                for (int lc8 = 0; lc8 < 8; ++lc8) {
                    const int lc = 8 * h + lc8;
                    const uint4 qv = *reinterpret_cast<const uint4*>(sQ + chunk_off(r, lc));
                    const uint32_t* u = reinterpret_cast<const uint32_t*>(&qv);
                    const float* zz = zsh + 8 * lc;
#pragma unroll
                    for (int e = 0; e < 4; ++e) di += bf_lo(u[e]) * zz[2 * e] + bf_hi(u[e]) * zz[2 * e + 1];
                }
                dpart[h * 128 + r] = di;
                // (b) S_prev -> bf16 B operand (row = dk = r, this thread's 64 dv columns = block h)
                if (i > 0) {
                    if (!cg_all(mbar_wait(&bar->s_done, (i - 1) & 1, err, LA_ERR_TIMEOUT))) { ok = false; break; }
                    tc_fence_after();
                }
#pragma unroll
                for (int cb = 0; cb < 2; ++cb) {
                    uint32_t wv[32];
                    tmem_ld32(tmem + lane_base + kTmS + 64 * h + 32 * cb, wv);
                    tmem_ld_wait();
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint4 v4;
                        v4.x = pack_bf16x2(__uint_as_float(wv[8 * q4 + 0]), __uint_as_float(wv[8 * q4 + 1]));
                        v4.y = pack_bf16x2(__uint_as_float(wv[8 * q4 + 2]), __uint_as_float(wv[8 * q4 + 3]));
                        v4.z = pack_bf16x2(__uint_as_float(wv[8 * q4 + 4]), __uint_as_float(wv[8 * q4 + 5]));
                        v4.w = pack_bf16x2(__uint_as_float(wv[8 * q4 + 6]), __uint_as_float(wv[8 * q4 + 7]));
                        *reinterpret_cast<uint4*>(sSb + chunk_off(r, 8 * h + 4 * cb + q4)) = v4;
                    }
                }
                tc_fence_before();
                fence_proxy_async_smem();
                cg_sync();
                if (ct == 0) mbar_arrive(&bar->sb_ready);
                // (c) A = tril(QK^T) on keys [64 h, 64 h + 64) -> bf16 pairs into TMEM; row-sum partial
                if (!cg_all(mbar_wait(&bar->qk_done, i & 1, err, LA_ERR_TIMEOUT))) { ok = false; break; }
                tc_fence_after();
                float rs = 0.f;
#pragma unroll
                for (int cb = 0; cb < 2; ++cb) {
                    uint32_t wv[32], pk[16];
                    tmem_ld32(tmem + lane_base + kTmQK + 64 * h + 32 * cb, wv);
                    tmem_ld_wait();
#pragma unroll
                    for (int x = 0; x < 16; ++x) {
                        const int j0 = 64 * h + 32 * cb + 2 * x;
                        pk[x] = pack_bf16x2(j0 <= r ? __uint_as_float(wv[2 * x]) : 0.f,
                                            j0 + 1 <= r ? __uint_as_float(wv[2 * x + 1]) : 0.f);
                        rs += bf_lo(pk[x]) + bf_hi(pk[x]);
                    }
                    tmem_st16(tmem + lane_base + kTmA + 32 * h + 16 * cb, pk);
                }
                rpart[h * 128 + r] = rs;
                tmem_st_wait();
                tc_fence_before();
                cg_sync();
                if (ct == 0) mbar_arrive(&bar->a_ready);
                // (d) o = O / den on this thread's 64 columns
                if (!cg_all(mbar_wait(&bar->o_done, i & 1, err, LA_ERR_TIMEOUT))) { ok = false; break; }
                tc_fence_after();
                const float inv = 1.f / (rpart[r] + rpart[128 + r] + dpart[r] + dpart[128 + r]);
                __nv_bfloat16* orow = o + ((size_t)bh * N + c0 + r) * kD + 64 * h;
#pragma unroll
                for (int cb = 0; cb < 2; ++cb) {
                    uint32_t wv[32];
                    tmem_ld32(tmem + lane_base + kTmO + 64 * h + 32 * cb, wv);
                    tmem_ld_wait();
                    if (r < n) {
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            uint4 v4;
                            v4.x = pack_bf16x2(__uint_as_float(wv[8 * q4 + 0]) * inv, __uint_as_float(wv[8 * q4 + 1]) * inv);
                            v4.y = pack_bf16x2(__uint_as_float(wv[8 * q4 + 2]) * inv, __uint_as_float(wv[8 * q4 + 3]) * inv);
                            v4.z = pack_bf16x2(__uint_as_float(wv[8 * q4 + 4]) * inv, __uint_as_float(wv[8 * q4 + 5]) * inv);
                            v4.w = pack_bf16x2(__uint_as_float(wv[8 * q4 + 6]) * inv, __uint_as_float(wv[8 * q4 + 7]) * inv);
                            *reinterpret_cast<uint4*>(orow + 32 * cb + 8 * q4) = v4;
                        }
                    }
                }
                tc_fence_before();
            }
            // z_prev += this chunk's column sums (after every thread has used z_prev)
            cg_sync();
            if (ct < 128) zsh[ct] += zpart[ct] + zpart[128 + ct];
            cg_sync();
        }
        if (!kOut && ok && nloc > 0) {
            // segment sums out: S from TMEM (row r = dk, this thread's 64 columns), z from shared memory.
            // The MMA thread's single-use drain barrier marks the last S update done.
            if (cg_all(mbar_wait(&bar->final_mma, 0, err, LA_ERR_TIMEOUT))) {
                tc_fence_after();
                float* out = segp + (size_t)r * kD + 64 * h;
#pragma unroll
                for (int cb = 0; cb < 2; ++cb) {
                    uint32_t wv[32];
                    tmem_ld32(tmem + lane_base + kTmS + 64 * h + 32 * cb, wv);
                    tmem_ld_wait();
#pragma unroll
                    for (int x = 0; x < 32; x += 4)
                        *reinterpret_cast<float4*>(out + 32 * cb + x) =
                            make_float4(__uint_as_float(wv[x]), __uint_as_float(wv[x + 1]),
                                        __uint_as_float(wv[x + 2]), __uint_as_float(wv[x + 3]));
                }
                if (ct < 128) segp[(size_t)kD * kD + ct] = zsh[ct];
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
