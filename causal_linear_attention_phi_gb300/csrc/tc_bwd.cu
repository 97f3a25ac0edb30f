// tc_bwd.cu -- tensor-core (tcgen05 / TMEM / TMA) kernels of the causal
// backward for bf16 inputs with Dk = Dv = 128, chunks of 128 positions.
//
// The gradient is a cumulative sum ("[논문 리뷰] Transformers are RNNs ..."
// (velog review), 3.5 Gradient Computation): states are recomputed, never
// stored per position.  With den_i = phi(q_i)^T z_i, P_i = dO_i / den_i,
// g_i = -(dO_i . o_i) / den_i, per chunk c (A = tril(Q~ K~^T), D = tril(P V^T + g 1^T)):
//   dQ~ = P S_prev^T + g z_prev^T + D K~
//   dK~ = V R_next^T + 1 r_next^T + D^T Q~
//   dV  = K~ R_next + A^T P
// where R_next = sum over later positions of phi(q_i) P_i^T and r_next = sum g_i phi(q_i).
//
// Forward sweep kernel: chunks in order, S and the segment's R contribution in
// TMEM; recomputes num, den (as the forward does), derives P and g, writes dq
// and the per-position (den, g).
// Reverse sweep kernel: chunks in reverse order with R_next in TMEM; every
// product is taken with the keys as the M (TMEM lane) dimension so dk and dv
// come out row by row.
//
// Roles as in the forward kernel: warp 0 TMA, warp 1 TMEM owner and MMA
// issuer, warps 2-5 the compute warpgroup.  All waits are bounded.
#include "tc_common.cuh"

namespace la {
namespace {
using namespace sm100;
using namespace tc;

constexpr int kThreads = 192;

// ------------------------------------------------------------------ forward sweep
// TMEM: S [0,128) fp32 state; R [128,256) segment sum of phi(q) P^T;
// X [256,384): QK^T fp32 -> A bf16 in X[0,64) -> P V^T fp32 -> D as bf16 hi / lo in X[0,64) / X[64,128);
// Y [384,512): O = phi(Q) S_prev + A V (numerator) -> dQ~.
constexpr uint32_t kFS = 0, kFR = 128, kFX = 256, kFY = 384;

struct FwdSweepBars {
    uint64_t full, empty;
    uint64_t qk_ready, sb_ready, a_ready, p_ready, d_ready;
    uint64_t qk_done, o_done, s_done, pv_done, dq_done;
    uint64_t final_mma;
};

struct FwdSweepSmem {
    static constexpr int Q = 0, K = kTileBytes, V = 2 * kTileBytes, P = 3 * kTileBytes, Sb = 4 * kTileBytes;
    static constexpr int KLo = 5 * kTileBytes;   // low bf16 half of phi(K) (hi is the K tile)
    static constexpr int zsh = 6 * kTileBytes;   // float[128] z_prev
    static constexpr int rsh = zsh + 512;        // float[128] segment sum of g phi(q)
    static constexpr int gsh = rsh + 512;        // float[128] g of the chunk's rows
    static constexpr int bars = gsh + 512;
    static constexpr int tmem_slot = bars + 256;
    static constexpr int total = tmem_slot + 16;
};

__global__ void __launch_bounds__(kThreads, 1)
tc_bwd_forward_sweep_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                            __nv_bfloat16* __restrict__ dq, const float* __restrict__ seg_S,
                            float* __restrict__ seg_R, float* __restrict__ den_g, int N, int nchunks, int cps, int P,
                            int* err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = base + FwdSweepSmem::Q;
    uint8_t* sK = base + FwdSweepSmem::K;
    uint8_t* sV = base + FwdSweepSmem::V;
    uint8_t* sP = base + FwdSweepSmem::P;
    uint8_t* sSb = base + FwdSweepSmem::Sb;
    uint8_t* sKLo = base + FwdSweepSmem::KLo;
    float* zsh = reinterpret_cast<float*>(base + FwdSweepSmem::zsh);
    float* rsh = reinterpret_cast<float*>(base + FwdSweepSmem::rsh);
    float* gsh = reinterpret_cast<float*>(base + FwdSweepSmem::gsh);
    FwdSweepBars* bar = reinterpret_cast<FwdSweepBars*>(base + FwdSweepSmem::bars);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + FwdSweepSmem::tmem_slot);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int p = blockIdx.x, bh = blockIdx.y;
    const int cbeg = p * cps, cend = min(nchunks, cbeg + cps), nloc = cend - cbeg;
    const size_t E = state_elems(kD, kD);

    if (tid == 0) {
        uint64_t* b = reinterpret_cast<uint64_t*>(bar);
        for (int x = 0; x < (int)(sizeof(FwdSweepBars) / 8); ++x) mbar_init(b + x, 1);
        fence_mbar_init();
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_do);
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
        if (lane == 0) {
            int armed = -1;
            for (int i = 0; i < nloc; ++i) {
                const int t0 = (cbeg + i) * kC;
                if (!mbar_wait(&bar->empty, (i & 1) ^ 1, err, LA_ERR_TIMEOUT)) break;
                mbar_arrive_expect_tx(&bar->full, 4 * kTileBytes);
                tma_load_3d(sQ, &tm_q, 0, t0, bh, &bar->full);
                tma_load_3d(sQ + kBlockBytes, &tm_q, 64, t0, bh, &bar->full);
                tma_load_3d(sK, &tm_k, 0, t0, bh, &bar->full);
                tma_load_3d(sK + kBlockBytes, &tm_k, 64, t0, bh, &bar->full);
                tma_load_3d(sV, &tm_v, 0, t0, bh, &bar->full);
                tma_load_3d(sV + kBlockBytes, &tm_v, 64, t0, bh, &bar->full);
                tma_load_3d(sP, &tm_do, 0, t0, bh, &bar->full);
                tma_load_3d(sP + kBlockBytes, &tm_do, 64, t0, bh, &bar->full);
                armed = i;
            }
            if (armed >= 0) mbar_wait(&bar->full, armed & 1, err, LA_ERR_TIMEOUT);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t id_kk = idesc_bf16_f32(128, 128, 0, 0);
            constexpr uint32_t id_kmn = idesc_bf16_f32(128, 128, 0, 1);
            constexpr uint32_t id_mnmn = idesc_bf16_f32(128, 128, 1, 1);
            const uint32_t aQ = smem_u32(sQ), aK = smem_u32(sK), aV = smem_u32(sV), aP = smem_u32(sP),
                           aSb = smem_u32(sSb), aKLo = smem_u32(sKLo);
            for (int i = 0; i < nloc; ++i) {
                const uint32_t ph = i & 1;
                if (!mbar_wait(&bar->qk_ready, ph, err, LA_ERR_TIMEOUT)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // X = Q~ K~^T
                    mma_ss(tmem + kFX, desc_kmajor(aQ, kk), desc_kmajor(aK, kk), id_kk, kk > 0);
                mma_commit(&bar->qk_done);
                if (!mbar_wait(&bar->sb_ready, ph, err, LA_ERR_TIMEOUT)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // Y = Q~ S_prev
                    mma_ss(tmem + kFY, desc_kmajor(aQ, kk), desc_mnmajor(aSb, kk), id_kmn, kk > 0);
                if (!mbar_wait(&bar->a_ready, ph, err, LA_ERR_TIMEOUT)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // Y += A V
                    mma_ts(tmem + kFY, tmem + kFX + 8 * kk, desc_mnmajor(aV, kk), id_kmn, 1);
                mma_commit(&bar->o_done);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // S += K~^T V
                    mma_ss(tmem + kFS, desc_mnmajor(aK, kk), desc_mnmajor(aV, kk), id_mnmn, 1);
                mma_commit(&bar->s_done);
                if (!mbar_wait(&bar->p_ready, ph, err, LA_ERR_TIMEOUT)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // X = P V^T
                    mma_ss(tmem + kFX, desc_kmajor(aP, kk), desc_kmajor(aV, kk), id_kk, kk > 0);
                mma_commit(&bar->pv_done);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // R += Q~^T P
                    mma_ss(tmem + kFR, desc_mnmajor(aQ, kk), desc_mnmajor(aP, kk), id_mnmn, (i > 0 || kk > 0));
                if (!mbar_wait(&bar->d_ready, ph, err, LA_ERR_TIMEOUT)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // Y = P S_prev^T
                    mma_ss(tmem + kFY, desc_kmajor(aP, kk), desc_kmajor(aSb, kk), id_kk, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // Y += D K~ as D_hi K_hi + D_lo K_hi + D_hi K_lo
                    mma_ts(tmem + kFY, tmem + kFX + 8 * kk, desc_mnmajor(aK, kk), id_kmn, 1);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ts(tmem + kFY, tmem + kFX + 64 + 8 * kk, desc_mnmajor(aK, kk), id_kmn, 1);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ts(tmem + kFY, tmem + kFX + 8 * kk, desc_mnmajor(aKLo, kk), id_kmn, 1);
                mma_commit(&bar->dq_done);
            }
            mma_commit(&bar->final_mma);
            mbar_wait(&bar->final_mma, 0, err, LA_ERR_TIMEOUT);
        }
    } else {
        const int t = tid - 64;
        const int r = 32 * (warp & 3) + lane;
        const uint32_t lb = (uint32_t)(32 * (warp & 3)) << 16;
        const float* pre = seg_S + ((size_t)bh * P + p) * E;
        global_row_to_tmem(pre + (size_t)r * kD, tmem + lb + kFS);
        zsh[r] = pre[(size_t)kD * kD + r];
        rsh[r] = 0.f;
        tc_fence_before();
        bool ok = wg_all(true);
        float* dgh = den_g + (size_t)bh * N * 2;
        for (int i = 0; i < nloc && ok; ++i) {
            const uint32_t ph = i & 1;
            const int c0 = (cbeg + i) * kC, n = min(kC, N - c0);
            // (a) phi on the Q and K tiles; this chunk's column sums of phi(K); den_inter
            if (!wg_all(mbar_wait(&bar->full, ph, err, LA_ERR_TIMEOUT))) { ok = false; break; }
            phi_tile_split(sK, sKLo, t, n);
            phi_tile(sQ, t, n);
            fence_proxy_async_smem();
            wg_sync();
            if (t == 0) mbar_arrive(&bar->qk_ready);
            const float zc = column_sum(sK, t, n, nullptr);
            float den_inter = 0.f;
#pragma unroll 4
            for (int lc = 0; lc < 16; ++lc) {
                const uint4 w = *reinterpret_cast<const uint4*>(sQ + chunk_off(r, lc));
                const uint32_t* u = reinterpret_cast<const uint32_t*>(&w);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    den_inter += bf_lo(u[e]) * zsh[8 * lc + 2 * e] + bf_hi(u[e]) * zsh[8 * lc + 2 * e + 1];
            }
            // (b) S_prev -> bf16 copy (rows = dk)
            if (i > 0) {
                const bool w1 = mbar_wait(&bar->s_done, (i - 1) & 1, err, LA_ERR_TIMEOUT);
                const bool w2 = mbar_wait(&bar->dq_done, (i - 1) & 1, err, LA_ERR_TIMEOUT);
                if (!wg_all(w1 && w2)) { ok = false; break; }
                tc_fence_after();
            }
            tmem_row_to_tile(tmem + lb + kFS, sSb, r);
            tc_fence_before();
            fence_proxy_async_smem();
            wg_sync();
            if (t == 0) mbar_arrive(&bar->sb_ready);
            // (c) A = tril(QK^T) as bf16 pairs into X[0,64) (each thread overwrites only columns it has read)
            if (!wg_all(mbar_wait(&bar->qk_done, ph, err, LA_ERR_TIMEOUT))) { ok = false; break; }
            tc_fence_after();
            float rs = 0.f;
#pragma unroll
            for (int cb = 0; cb < 4; ++cb) {
                uint32_t w[32], pk[16];
                tmem_ld32(tmem + lb + kFX + 32 * cb, w);
                tmem_ld_wait();
#pragma unroll
                for (int x = 0; x < 16; ++x) {
                    const int j = 32 * cb + 2 * x;
                    pk[x] = pack_bf16x2(j <= r ? __uint_as_float(w[2 * x]) : 0.f,
                                        j + 1 <= r ? __uint_as_float(w[2 * x + 1]) : 0.f);
                    rs += bf_lo(pk[x]) + bf_hi(pk[x]);
                }
                tmem_st16(tmem + lb + kFX + 16 * cb, pk);
            }
            tmem_st_wait();
            tc_fence_before();
            wg_sync();
            if (t == 0) mbar_arrive(&bar->a_ready);
            // (d) den, g, P = dO / den (in place over dO), store (den, g)
            if (!wg_all(mbar_wait(&bar->o_done, ph, err, LA_ERR_TIMEOUT))) { ok = false; break; }
            tc_fence_after();
            const bool valid = r < n;
            const float den = valid ? rs + den_inter : 1.f;
            const float inv = 1.f / den;
            float dot = 0.f;
#pragma unroll
            for (int cb = 0; cb < 4; ++cb) {
                uint32_t w[32];
                tmem_ld32(tmem + lb + kFY + 32 * cb, w);
                tmem_ld_wait();
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint4* pp = reinterpret_cast<uint4*>(sP + chunk_off(r, 4 * cb + q4));
                    uint4 v4 = *pp;
                    uint32_t* u = reinterpret_cast<uint32_t*>(&v4);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        u[e] = pack_bf16x2(bf_lo(u[e]) * inv, bf_hi(u[e]) * inv);
                        dot += bf_lo(u[e]) * __uint_as_float(w[8 * q4 + 2 * e]) +
                               bf_hi(u[e]) * __uint_as_float(w[8 * q4 + 2 * e + 1]);
                    }
                    *pp = v4;
                }
            }
            // g = -P.o with the bf16 P the products use (o = num / den)
            const float g = valid ? -dot * inv : 0.f;
            gsh[r] = g;
            if (valid) {
                dgh[(size_t)(c0 + r) * 2 + 0] = den;
                dgh[(size_t)(c0 + r) * 2 + 1] = g;
            }
            fence_proxy_async_smem();
            tc_fence_before();
            wg_sync();
            if (t == 0) mbar_arrive(&bar->p_ready);
            rsh[t] += column_sum(sQ, t, n, gsh);  // segment sum of g phi(q)
            // (e) D = tril(P V^T + g) as a hi + lo pair of bf16 operands: D_hi in X[0,64),
            // D_lo in X[64,128).  PV block cb (columns 32cb..32cb+31) gives D_hi columns
            // 16cb.. and D_lo columns 64+16cb..; loading the blocks in the order 0, 2, 1, 3,
            // each before the writes that land on it, means every column a thread
            // overwrites has already been read by that thread.
            if (!wg_all(mbar_wait(&bar->pv_done, ph, err, LA_ERR_TIMEOUT))) { ok = false; break; }
            tc_fence_after();
            {
                uint32_t w0[32], w1[32];
                auto emit = [&](const uint32_t (&w)[32], int cb) {
                    uint32_t hi[16], lo[16];
#pragma unroll
                    for (int x = 0; x < 16; ++x) {
                        const int j = 32 * cb + 2 * x;
                        const float d0 = j <= r ? __uint_as_float(w[2 * x]) + g : 0.f;
                        const float d1 = j + 1 <= r ? __uint_as_float(w[2 * x + 1]) + g : 0.f;
                        hi[x] = pack_bf16x2(d0, d1);
                        lo[x] = pack_bf16x2(d0 - bf_lo(hi[x]), d1 - bf_hi(hi[x]));
                    }
                    tmem_st16(tmem + lb + kFX + 16 * cb, hi);
                    tmem_st16(tmem + lb + kFX + 64 + 16 * cb, lo);
                };
                tmem_ld32(tmem + lb + kFX + 0, w0);
                tmem_ld32(tmem + lb + kFX + 64, w1);
                tmem_ld_wait();
                emit(w0, 0);                       // writes 0-15, 64-79 (blocks 0, 2 read)
                tmem_ld32(tmem + lb + kFX + 32, w0);
                tmem_ld_wait();
                emit(w0, 1);                       // writes 16-31, 80-95 (block 1 read)
                tmem_ld32(tmem + lb + kFX + 96, w0);
                tmem_ld_wait();
                emit(w1, 2);                       // writes 32-47, 96-111 (block 3 read)
                emit(w0, 3);                       // writes 48-63, 112-127
            }
            tmem_st_wait();
            tc_fence_before();
            wg_sync();
            if (t == 0) mbar_arrive(&bar->d_ready);
            // (f) dq = (dQ~ + g z_prev) * phi'(q)
            if (!wg_all(mbar_wait(&bar->dq_done, ph, err, LA_ERR_TIMEOUT))) { ok = false; break; }
            tc_fence_after();
            __nv_bfloat16* drow = dq + ((size_t)bh * N + c0 + r) * kD;
#pragma unroll
            for (int cb = 0; cb < 4; ++cb) {
                uint32_t w[32];
                tmem_ld32(tmem + lb + kFY + 32 * cb, w);
                tmem_ld_wait();
                if (valid) {
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const uint4 qv = *reinterpret_cast<const uint4*>(sQ + chunk_off(r, 4 * cb + q4));
                        const uint32_t* qu = reinterpret_cast<const uint32_t*>(&qv);
                        uint4 o4;
                        uint32_t* ou = reinterpret_cast<uint32_t*>(&o4);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int d = 32 * cb + 8 * q4 + 2 * e;
                            const float a0 = (__uint_as_float(w[8 * q4 + 2 * e]) + g * zsh[d]) * dphi_from_phi(bf_lo(qu[e]));
                            const float a1 =
                                (__uint_as_float(w[8 * q4 + 2 * e + 1]) + g * zsh[d + 1]) * dphi_from_phi(bf_hi(qu[e]));
                            ou[e] = pack_bf16x2(a0, a1);
                        }
                        *reinterpret_cast<uint4*>(drow + 32 * cb + 8 * q4) = o4;
                    }
                }
            }
            tc_fence_before();
            wg_sync();
            zsh[t] += zc;
            wg_sync();
            if (t == 0) mbar_arrive(&bar->empty);
        }
        // segment sums of the reverse state out: R from TMEM, r from shared memory
        if (ok && nloc > 0 && wg_all(mbar_wait(&bar->final_mma, 0, err, LA_ERR_TIMEOUT))) {
            tc_fence_after();
            float* out = seg_R + ((size_t)bh * P + p) * E;
            tmem_row_to_global(tmem + lb + kFR, out + (size_t)r * kD);
            out[(size_t)kD * kD + t] = rsh[t];
        }
        tc_fence_before();
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------ reverse sweep
// TMEM: R [0,128) fp32 reverse state R_next; DK [128,256) and DV [256,384)
// accumulators (they first hold D^T and A^T in fp32); X [384,512): D^T bf16 in
// X[0,64), A^T bf16 in X[64,128).
constexpr uint32_t kRR = 0, kRDK = 128, kRDV = 256, kRX = 384;

struct RevSweepBars {
    uint64_t full, empty;
    uint64_t ready, rb_ready, masks_ready;
    uint64_t at_done, dt_done, dkv_done;
    uint64_t final_mma;
};

struct RevSweepSmem {
    static constexpr int Q = 0, K = kTileBytes, V = 2 * kTileBytes, P = 3 * kTileBytes, Rb = 4 * kTileBytes;
    static constexpr int rsh = 5 * kTileBytes;  // float[128] r_next
    static constexpr int gsh = rsh + 512;       // float[128] g of the chunk's rows
    static constexpr int ish = gsh + 512;       // float[128] 1/den of the chunk's rows
    static constexpr int bars = ish + 512;
    static constexpr int tmem_slot = bars + 256;
    static constexpr int total = tmem_slot + 16;
};

__global__ void __launch_bounds__(kThreads, 1)
tc_bwd_reverse_sweep_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                            __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dv,
                            const float* __restrict__ seg_R, const float* __restrict__ den_g, int N, int nchunks,
                            int cps, int P, int* err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = base + RevSweepSmem::Q;
    uint8_t* sK = base + RevSweepSmem::K;
    uint8_t* sV = base + RevSweepSmem::V;
    uint8_t* sP = base + RevSweepSmem::P;
    uint8_t* sRb = base + RevSweepSmem::Rb;
    float* rsh = reinterpret_cast<float*>(base + RevSweepSmem::rsh);
    float* gsh = reinterpret_cast<float*>(base + RevSweepSmem::gsh);
    float* ish = reinterpret_cast<float*>(base + RevSweepSmem::ish);
    RevSweepBars* bar = reinterpret_cast<RevSweepBars*>(base + RevSweepSmem::bars);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + RevSweepSmem::tmem_slot);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int p = blockIdx.x, bh = blockIdx.y;
    const int cbeg = p * cps, cend = min(nchunks, cbeg + cps), nloc = cend - cbeg;
    const size_t E = state_elems(kD, kD);

    if (tid == 0) {
        uint64_t* b = reinterpret_cast<uint64_t*>(bar);
        for (int x = 0; x < (int)(sizeof(RevSweepBars) / 8); ++x) mbar_init(b + x, 1);
        fence_mbar_init();
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_do);
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
        if (lane == 0) {
            int armed = -1;
            for (int i = 0; i < nloc; ++i) {
                const int t0 = (cend - 1 - i) * kC;
                if (!mbar_wait(&bar->empty, (i & 1) ^ 1, err, LA_ERR_TIMEOUT)) break;
                mbar_arrive_expect_tx(&bar->full, 4 * kTileBytes);
                tma_load_3d(sQ, &tm_q, 0, t0, bh, &bar->full);
                tma_load_3d(sQ + kBlockBytes, &tm_q, 64, t0, bh, &bar->full);
                tma_load_3d(sK, &tm_k, 0, t0, bh, &bar->full);
                tma_load_3d(sK + kBlockBytes, &tm_k, 64, t0, bh, &bar->full);
                tma_load_3d(sV, &tm_v, 0, t0, bh, &bar->full);
                tma_load_3d(sV + kBlockBytes, &tm_v, 64, t0, bh, &bar->full);
                tma_load_3d(sP, &tm_do, 0, t0, bh, &bar->full);
                tma_load_3d(sP + kBlockBytes, &tm_do, 64, t0, bh, &bar->full);
                armed = i;
            }
            if (armed >= 0) mbar_wait(&bar->full, armed & 1, err, LA_ERR_TIMEOUT);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t id_kk = idesc_bf16_f32(128, 128, 0, 0);
            constexpr uint32_t id_kmn = idesc_bf16_f32(128, 128, 0, 1);
            constexpr uint32_t id_mnmn = idesc_bf16_f32(128, 128, 1, 1);
            const uint32_t aQ = smem_u32(sQ), aK = smem_u32(sK), aV = smem_u32(sV), aP = smem_u32(sP),
                           aRb = smem_u32(sRb);
            for (int i = 0; i < nloc; ++i) {
                const uint32_t ph = i & 1;
                if (!mbar_wait(&bar->ready, ph, err, LA_ERR_TIMEOUT)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // DV region = A^T = K~ Q~^T (rows = keys)
                    mma_ss(tmem + kRDV, desc_kmajor(aK, kk), desc_kmajor(aQ, kk), id_kk, kk > 0);
                mma_commit(&bar->at_done);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // DK region = V P^T (rows = keys)
                    mma_ss(tmem + kRDK, desc_kmajor(aV, kk), desc_kmajor(aP, kk), id_kk, kk > 0);
                mma_commit(&bar->dt_done);
                if (!mbar_wait(&bar->rb_ready, ph, err, LA_ERR_TIMEOUT)) break;
                if (!mbar_wait(&bar->masks_ready, ph, err, LA_ERR_TIMEOUT)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // dK~ = V R_next^T
                    mma_ss(tmem + kRDK, desc_kmajor(aV, kk), desc_kmajor(aRb, kk), id_kk, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // dK~ += D^T Q~
                    mma_ts(tmem + kRDK, tmem + kRX + 8 * kk, desc_mnmajor(aQ, kk), id_kmn, 1);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // dV = K~ R_next
                    mma_ss(tmem + kRDV, desc_kmajor(aK, kk), desc_mnmajor(aRb, kk), id_kmn, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // dV += A^T P
                    mma_ts(tmem + kRDV, tmem + kRX + 64 + 8 * kk, desc_mnmajor(aP, kk), id_kmn, 1);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // R_next += Q~^T P
                    mma_ss(tmem + kRR, desc_mnmajor(aQ, kk), desc_mnmajor(aP, kk), id_mnmn, 1);
                mma_commit(&bar->dkv_done);
            }
            mma_commit(&bar->final_mma);
            mbar_wait(&bar->final_mma, 0, err, LA_ERR_TIMEOUT);
        }
    } else {
        const int t = tid - 64;
        const int r = 32 * (warp & 3) + lane;
        const uint32_t lb = (uint32_t)(32 * (warp & 3)) << 16;
        const float* suf = seg_R + ((size_t)bh * P + p) * E;
        global_row_to_tmem(suf + (size_t)r * kD, tmem + lb + kRR);
        rsh[r] = suf[(size_t)kD * kD + r];
        tc_fence_before();
        bool ok = wg_all(true);
        const float* dgh = den_g + (size_t)bh * N * 2;
        for (int i = 0; i < nloc && ok; ++i) {
            const uint32_t ph = i & 1;
            const int c0 = (cend - 1 - i) * kC, n = min(kC, N - c0);
            // (a) per-row 1/den and g; phi on Q and K; P = dO / den in place
            if (!wg_all(mbar_wait(&bar->full, ph, err, LA_ERR_TIMEOUT))) { ok = false; break; }
            {
                const bool valid = t < n;
                ish[t] = valid ? 1.f / dgh[(size_t)(c0 + t) * 2 + 0] : 0.f;
                gsh[t] = valid ? dgh[(size_t)(c0 + t) * 2 + 1] : 0.f;
            }
            wg_sync();
            phi_tile(sQ, t, n);
            phi_tile(sK, t, n);
            scale_rows_tile(sP, t, ish);
            fence_proxy_async_smem();
            wg_sync();
            if (t == 0) mbar_arrive(&bar->ready);
            const float rc = column_sum(sQ, t, n, gsh);  // this chunk's sum of g phi(q), column t
            // (b) R_next -> bf16 copy (rows = dk)
            if (i > 0) {
                if (!wg_all(mbar_wait(&bar->dkv_done, (i - 1) & 1, err, LA_ERR_TIMEOUT))) { ok = false; break; }
                tc_fence_after();
            }
            tmem_row_to_tile(tmem + lb + kRR, sRb, r);
            tc_fence_before();
            fence_proxy_async_smem();
            wg_sync();
            if (t == 0) mbar_arrive(&bar->rb_ready);
            // (c) masks: row r is key j = r; column x is query i = x; keep j <= i
            if (!wg_all(mbar_wait(&bar->at_done, ph, err, LA_ERR_TIMEOUT))) { ok = false; break; }
            tc_fence_after();
#pragma unroll
            for (int cb = 0; cb < 4; ++cb) {
                uint32_t w[32], pk[16];
                tmem_ld32(tmem + lb + kRDV + 32 * cb, w);
                tmem_ld_wait();
#pragma unroll
                for (int x = 0; x < 16; ++x) {
                    const int qi = 32 * cb + 2 * x;
                    pk[x] = pack_bf16x2(r <= qi ? __uint_as_float(w[2 * x]) : 0.f,
                                        r <= qi + 1 ? __uint_as_float(w[2 * x + 1]) : 0.f);
                }
                tmem_st16(tmem + lb + kRX + 64 + 16 * cb, pk);
            }
            if (!wg_all(mbar_wait(&bar->dt_done, ph, err, LA_ERR_TIMEOUT))) { ok = false; break; }
            tc_fence_after();
#pragma unroll
            for (int cb = 0; cb < 4; ++cb) {
                uint32_t w[32], pk[16];
                tmem_ld32(tmem + lb + kRDK + 32 * cb, w);
                tmem_ld_wait();
#pragma unroll
                for (int x = 0; x < 16; ++x) {
                    const int qi = 32 * cb + 2 * x;
                    pk[x] = pack_bf16x2(r <= qi ? __uint_as_float(w[2 * x]) + gsh[qi] : 0.f,
                                        r <= qi + 1 ? __uint_as_float(w[2 * x + 1]) + gsh[qi + 1] : 0.f);
                }
                tmem_st16(tmem + lb + kRX + 16 * cb, pk);
            }
            tmem_st_wait();
            tc_fence_before();
            wg_sync();
            if (t == 0) mbar_arrive(&bar->masks_ready);
            // (d) dk = (dK~ + r_next) * phi'(k), dv
            if (!wg_all(mbar_wait(&bar->dkv_done, ph, err, LA_ERR_TIMEOUT))) { ok = false; break; }
            tc_fence_after();
            const bool valid = r < n;
            __nv_bfloat16* dkrow = dk + ((size_t)bh * N + c0 + r) * kD;
            __nv_bfloat16* dvrow = dv + ((size_t)bh * N + c0 + r) * kD;
#pragma unroll
            for (int cb = 0; cb < 4; ++cb) {
                uint32_t w[32];
                tmem_ld32(tmem + lb + kRDK + 32 * cb, w);
                tmem_ld_wait();
                if (valid) {
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const uint4 kv = *reinterpret_cast<const uint4*>(sK + chunk_off(r, 4 * cb + q4));
                        const uint32_t* ku = reinterpret_cast<const uint32_t*>(&kv);
                        uint4 o4;
                        uint32_t* ou = reinterpret_cast<uint32_t*>(&o4);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int d = 32 * cb + 8 * q4 + 2 * e;
                            ou[e] = pack_bf16x2((__uint_as_float(w[8 * q4 + 2 * e]) + rsh[d]) * dphi_from_phi(bf_lo(ku[e])),
                                                (__uint_as_float(w[8 * q4 + 2 * e + 1]) + rsh[d + 1]) *
                                                    dphi_from_phi(bf_hi(ku[e])));
                        }
                        *reinterpret_cast<uint4*>(dkrow + 32 * cb + 8 * q4) = o4;
                    }
                }
            }
#pragma unroll
            for (int cb = 0; cb < 4; ++cb) {
                uint32_t w[32];
                tmem_ld32(tmem + lb + kRDV + 32 * cb, w);
                tmem_ld_wait();
                if (valid) {
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint4 o4;
                        o4.x = pack_bf16x2(__uint_as_float(w[8 * q4 + 0]), __uint_as_float(w[8 * q4 + 1]));
                        o4.y = pack_bf16x2(__uint_as_float(w[8 * q4 + 2]), __uint_as_float(w[8 * q4 + 3]));
                        o4.z = pack_bf16x2(__uint_as_float(w[8 * q4 + 4]), __uint_as_float(w[8 * q4 + 5]));
                        o4.w = pack_bf16x2(__uint_as_float(w[8 * q4 + 6]), __uint_as_float(w[8 * q4 + 7]));
                        *reinterpret_cast<uint4*>(dvrow + 32 * cb + 8 * q4) = o4;
                    }
                }
            }
            tc_fence_before();
            wg_sync();
            rsh[t] += rc;
            wg_sync();
            if (t == 0) mbar_arrive(&bar->empty);
        }
        tc_fence_before();
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

constexpr size_t kFwdSweepSmem = FwdSweepSmem::total + 1024;
constexpr size_t kRevSweepSmem = RevSweepSmem::total + 1024;

}  // namespace

cudaError_t tc_bwd_forward_sweep(const void* q, const void* k, const void* v, const void* dout, void* dq,
                                 const float* seg_S, float* seg_R, float* den_g, const la_shape& s, const Plan& p,
                                 cudaStream_t st) {
    const int BH = s.B * s.H;
    CUtensorMap tq, tk, tv, td;
    if (!make_tmap_bf16_rows(&tq, q, BH, s.N, kD, kC) || !make_tmap_bf16_rows(&tk, k, BH, s.N, kD, kC) ||
        !make_tmap_bf16_rows(&tv, v, BH, s.N, kD, kC) || !make_tmap_bf16_rows(&td, dout, BH, s.N, kD, kC))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(tc_bwd_forward_sweep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kFwdSweepSmem);
    if (e != cudaSuccess) return e;
    launch_begin("tc_bwd_forward_sweep", st);
    tc_bwd_forward_sweep_kernel<<<dim3(p.P, BH), kThreads, kFwdSweepSmem, st>>>(
        tq, tk, tv, td, (__nv_bfloat16*)dq, seg_S, seg_R, den_g, s.N, p.nchunks, p.cps, p.P, device_error_word());
    return launch_end("tc_bwd_forward_sweep", st);
}

cudaError_t tc_bwd_reverse_sweep(const void* q, const void* k, const void* v, const void* dout, void* dk, void* dv,
                                 const float* seg_R, const float* den_g, const la_shape& s, const Plan& p,
                                 cudaStream_t st) {
    const int BH = s.B * s.H;
    CUtensorMap tq, tk, tv, td;
    if (!make_tmap_bf16_rows(&tq, q, BH, s.N, kD, kC) || !make_tmap_bf16_rows(&tk, k, BH, s.N, kD, kC) ||
        !make_tmap_bf16_rows(&tv, v, BH, s.N, kD, kC) || !make_tmap_bf16_rows(&td, dout, BH, s.N, kD, kC))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(tc_bwd_reverse_sweep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kRevSweepSmem);
    if (e != cudaSuccess) return e;
    launch_begin("tc_bwd_reverse_sweep", st);
    tc_bwd_reverse_sweep_kernel<<<dim3(p.P, BH), kThreads, kRevSweepSmem, st>>>(
        tq, tk, tv, td, (__nv_bfloat16*)dk, (__nv_bfloat16*)dv, seg_R, den_g, s.N, p.nchunks, p.cps, p.P,
        device_error_word());
    return launch_end("tc_bwd_reverse_sweep", st);
}

}  // namespace la
