// tc_noncausal_bwd.cu -- tensor-core (tcgen05 / TMEM / TMA) kernels of the gradient
// of the non-causal form, for bf16 heads of 128 (or 64, padded on chip).
//
// With the head totals S = phi(K)^T V, z = phi(K)^T 1, den_i = phi(q_i)^T z,
// P_i = dO_i / den_i, g_i = -(P_i . num_i) / den_i (num_i = phi(q_i)^T S),
// R = sum_i phi(q_i) P_i^T and r = sum_i g_i phi(q_i) over all positions:
//   dq_i = (S P_i + g_i z) * phi'(q_i),  dk_j = (R v_j + r) * phi'(k_j),  dv_j = R^T phi(k_j)
// (the causal gradient's state algebra without the mask: velog review 3.2 and 3.5,
// digest 핵심 구성요소 2).  There is no intra-chunk term, so each pass is a few
// products per chunk against totals held in shared memory as bf16 operands:
//   query pass:  num = phi(Q) S -> P, g (den in fp32 from phi(q) . z) -> dQ~ = P S^T,
//                dq = (dQ~ + g z) * phi'(q); R += phi(Q)^T P and the column sums of
//                g phi(Q) per segment (summed over segments by the scan that follows)
//   key pass:    dK~ = V R^T, dV = phi(K) R; dk = (dK~ + r) * phi'(k)
// dq_i = sum_j phi(k_j) P_i . (v_j - o_i) is a small difference of large terms when
// phi(k) varies little, and here every row carries the whole sum: an error of relative
// size e in o_i (through num and den) or in S reaches dq at about e / (the spread of
// phi(k)).  So S (summed from phi(K) as hi + lo parts) enters as a hi + lo pair of
// bf16 operands, num = Q S_hi + Q S_lo and dQ~ = P S_hi^T + P S_lo^T, with g formed
// from the bf16 P the products use (single bf16 copies gave 2.1-2.6 % error in dq
// against a 2 % bound).  phi(Q) stays one bf16 copy: its rounding scales every key's
// weight w_ij alike, num and den see the same copy, and o_i barely moves.  Q is
// double-buffered (the next chunk's tile lands while this one is worked on) and dO is
// released apart from it, right after its last reads.  Roles (320 threads): warp 0
// TMA loads, warp 1 TMEM owner and MMA issuer, warps 2-9 the compute group (warp w:
// TMEM lanes 32 (w % 4) .. +31, i.e. row r of the chunk, column half (w - 2) / 4).
// Every wait is bounded.
#include <cudaTypedefs.h>

#include "tc_common.cuh"

namespace la {
namespace {
using namespace sm100;
using namespace tc;

constexpr int kThreads = 320;  // warp 0 TMA, warp 1 MMA, warps 2-9 compute
constexpr int kComputeThreads = 256;
using CG = Grp<kComputeThreads>;
constexpr size_t kE = (size_t)kD * kD + kD;  // a padded (R, r) or (S, z) record

// ------------------------------------------------------------------ query pass
// TMEM: Y [0,128) num, then dQ~; R [128,256) the segment's sum of phi(Q)^T P.
constexpr uint32_t kQY = 0, kQR = 128;

// full/empty pairs: the Q buffers (empty: the MMA's last read and the compute group's)
// and the dO tile (likewise).
struct QBars {
    uint64_t full_q[2], empty_q[2], full_p, empty_p;
    uint64_t q_ready, num_done, p_ready, dq_done, y_free;
    uint64_t final_mma;
};

struct QSmem {
    static constexpr int Q0 = 0, P = 2 * kTileBytes, Sb = 3 * kTileBytes;  // Q buffers 0, 1; Sb: bf16 S (hi), rows = dk
    static constexpr int SbLo = 4 * kTileBytes;  // bf16 S - hi
    static constexpr int Ob = 5 * kTileBytes;    // dq tile for the TMA store
    static constexpr int zsh = 6 * kTileBytes;  // float[128] z
    static constexpr int dpart = zsh + 512;     // float[2][128] phi(q) . z per column half
    static constexpr int tpart = dpart + 1024;  // float[2][128] P . num per column half
    static constexpr int gsh = tpart + 1024;    // float[128] g of the chunk's rows
    static constexpr int drpart = gsh + 512;    // float[8][128] per-warp column sums of g phi(q)
    static constexpr int racc = drpart + 4096;  // float[128] segment sum of g phi(q)
    static constexpr int bars = racc + 512;
    static constexpr int tmem_slot = bars + 256;
    static constexpr int total = tmem_slot + 16;
};
constexpr size_t kQSmemBytes = QSmem::total + 1024;

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
tc_noncausal_bwd_query_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                              const __grid_constant__ CUtensorMap tm_dq, const float* __restrict__ totS,
                              float* __restrict__ seg_R, int N, int nchunks, int cps, int P, int* err) {
    extern __shared__ uint8_t smem_raw[];
    pdl_enter();  // launched with programmatic dependent launch
    constexpr int kKd = D / 16;  // K steps over a head dimension (a 64-wide head is zero above)
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    auto sQb = [&](int b) { return base + QSmem::Q0 + b * kTileBytes; };
    uint8_t* sP = base + QSmem::P;
    uint8_t* sSb = base + QSmem::Sb;
    uint8_t* sSbLo = base + QSmem::SbLo;
    uint8_t* sOb = base + QSmem::Ob;
    float* zsh = reinterpret_cast<float*>(base + QSmem::zsh);
    float* dpart = reinterpret_cast<float*>(base + QSmem::dpart);
    float* tpart = reinterpret_cast<float*>(base + QSmem::tpart);
    float* gsh = reinterpret_cast<float*>(base + QSmem::gsh);
    float* drpart = reinterpret_cast<float*>(base + QSmem::drpart);
    float* racc = reinterpret_cast<float*>(base + QSmem::racc);
    QBars* bar = reinterpret_cast<QBars*>(base + QSmem::bars);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + QSmem::tmem_slot);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int p = blockIdx.x, bh = blockIdx.y;
    const int cbeg = p * cps, cend = min(nchunks, cbeg + cps), nloc = cend - cbeg;
    check_plan(p, (int)gridDim.x, cbeg, cend, nchunks, N);
    const float* tot = totS + (size_t)bh * kE;

    if (tid == 0) {
        uint64_t* b = reinterpret_cast<uint64_t*>(bar);
        for (int x = 0; x < (int)(sizeof(QBars) / 8); ++x) mbar_init(b + x, 1);
        mbar_init(&bar->empty_q[0], 2);  // one MMA commit + one compute-group arrival each
        mbar_init(&bar->empty_q[1], 2);
        mbar_init(&bar->empty_p, 2);
        fence_mbar_init();
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_do);
        tma_prefetch_desc(&tm_dq);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 256);
        tmem_relinquish();
    }
    if (warp >= 2) {  // S as bf16 hi + lo operands (row r, this thread's 64 columns), z and the sums in fp32
        const int ct = tid - 64, h = (warp - 2) >> 2, r = 32 * (warp & 3) + lane;
#pragma unroll
        for (int cb = 0; cb < 2; ++cb) {
            uint32_t w[32], wl[32];
            const float4* src = reinterpret_cast<const float4*>(tot + (size_t)r * kD + 64 * h + 32 * cb);
#pragma unroll
            for (int x4 = 0; x4 < 8; ++x4) {  // 16-byte loads: the workspace and each record row are 16-byte aligned
                const float4 f = src[x4];
                const float vals[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    w[4 * x4 + e] = __float_as_uint(vals[e]);
                    wl[4 * x4 + e] = __float_as_uint(vals[e] - __bfloat162float(__float2bfloat16_rn(vals[e])));
                }
            }
            row32_to_tile(w, sSb, r, 8 * h + 4 * cb);
            row32_to_tile(wl, sSbLo, r, 8 * h + 4 * cb);
        }
        if (ct < kD) {
            zsh[ct] = tot[(size_t)kD * kD + ct];
            racc[ct] = 0.f;
        }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            int armed_q[2] = {-1, -1}, armed_p = -1;
            for (int i = 0; i < nloc; ++i) {
                const int t0 = (cbeg + i) * kC, b = i & 1;
                if (!mbar_wait(&bar->empty_q[b], ((i >> 1) & 1) ^ 1, err, LA_ERR_TIMEOUT)) break;
                mbar_arrive_expect_tx(&bar->full_q[b], kTileBytes);
                check_tile(0, t0, bh, N), tma_load_3d(sQb(b), &tm_q, 0, t0, bh, &bar->full_q[b]);
                check_tile(64, t0, bh, N), tma_load_3d(sQb(b) + kBlockBytes, &tm_q, 64, t0, bh, &bar->full_q[b]);
                armed_q[b] = i;
                if (!mbar_wait(&bar->empty_p, (i & 1) ^ 1, err, LA_ERR_TIMEOUT)) break;
                mbar_arrive_expect_tx(&bar->full_p, kTileBytes);
                check_tile(0, t0, bh, N), tma_load_3d(sP, &tm_do, 0, t0, bh, &bar->full_p);
                check_tile(64, t0, bh, N), tma_load_3d(sP + kBlockBytes, &tm_do, 64, t0, bh, &bar->full_p);
                armed_p = i;
            }
            // no copy may still be landing when the CTA exits
            for (int b = 0; b < 2; ++b)
                if (armed_q[b] >= 0) mbar_wait(&bar->full_q[b], (armed_q[b] >> 1) & 1, err, LA_ERR_TIMEOUT);
            if (armed_p >= 0) mbar_wait(&bar->full_p, armed_p & 1, err, LA_ERR_TIMEOUT);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t id_kk = idesc_bf16_f32(128, 128, 0, 0);
            constexpr uint32_t id_kmn = idesc_bf16_f32(128, 128, 0, 1);
            constexpr uint32_t id_mnmn = idesc_bf16_f32(128, 128, 1, 1);
            const uint32_t aP = smem_u32(sP), aSb = smem_u32(sSb), aSbLo = smem_u32(sSbLo);
            for (int i = 0; i < nloc; ++i) {
                const uint32_t ph = i & 1;
                const uint32_t aQ = smem_u32(sQb(i & 1));
                if (!mbar_wait(&bar->q_ready, ph, err, LA_ERR_TIMEOUT) ||
                    (i > 0 && !mbar_wait(&bar->y_free, ph ^ 1, err, LA_ERR_TIMEOUT)))
                    break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kKd; ++kk) {  // Y = Q S_hi + Q S_lo (num)
                    mma_ss(tmem + kQY, desc_kmajor(aQ, kk), desc_mnmajor(aSb, kk), id_kmn, kk > 0);
                    mma_ss(tmem + kQY, desc_kmajor(aQ, kk), desc_mnmajor(aSbLo, kk), id_kmn, 1);
                }
                mma_commit(&bar->num_done);
                if (!mbar_wait(&bar->p_ready, ph, err, LA_ERR_TIMEOUT)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kKd; ++kk)  // Y = P S_hi^T + P S_lo^T (dQ~ without the g z term)
                    mma_ss(tmem + kQY, desc_kmajor(aP, kk), desc_kmajor(aSb, kk), id_kk, kk > 0);
#pragma unroll
                for (int kk = 0; kk < kKd; ++kk)
                    mma_ss(tmem + kQY, desc_kmajor(aP, kk), desc_kmajor(aSbLo, kk), id_kk, 1);
                mma_commit(&bar->dq_done);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // R += phi(Q)^T P
                    mma_ss(tmem + kQR, desc_mnmajor(aQ, kk), desc_mnmajor(aP, kk), id_mnmn, (i > 0 || kk > 0));
                mma_commit(&bar->empty_q[i & 1]);  // last MMA reads of this Q buffer and of P in this chunk
                mma_commit(&bar->empty_p);
            }
            mma_commit(&bar->final_mma);
            mbar_wait(&bar->final_mma, 0, err, LA_ERR_TIMEOUT);
        }
    } else {
        const int ct = tid - 64;
        const int h = (warp - 2) >> 2;
        const int r = 32 * (warp & 3) + lane;
        const uint32_t lb = ((uint32_t)(32 * (warp & 3)) << 16) + 64 * h;  // this thread's row half
        bool ok = CG::all(true);
        for (int i = 0; i < nloc && ok; ++i) {
            const uint32_t ph = i & 1;
            const int c0 = (cbeg + i) * kC, n = min(kC, N - c0);
            const bool valid = r < n;
            // (a) phi on Q in place (the buffer is held to the end of the chunk: the dq epilogue
            // reads phi(q) again for phi'(q)); phi(q_r) . z in fp32 on this thread's 64 columns
            uint8_t* sQ = sQb(i & 1);
            if (!CG::all(mbar_wait(&bar->full_q[i & 1], (i >> 1) & 1, err, LA_ERR_TIMEOUT))) { ok = false; break; }
            CG::phi_tile(sQ, nullptr, ct, n, D, nullptr, nullptr);
            fence_proxy_async_smem();
            CG::sync();
            if (ct == 0) mbar_arrive(&bar->q_ready);
            {
                float di = 0.f;
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) {
                    const int lc = 8 * h + c8;
                    const uint4 qv = *reinterpret_cast<const uint4*>(sQ + chunk_off(r, lc));
                    const float4 za = *reinterpret_cast<const float4*>(zsh + 8 * lc);
                    const float4 zb = *reinterpret_cast<const float4*>(zsh + 8 * lc + 4);
                    di += bf_lo(qv.x) * za.x + bf_hi(qv.x) * za.y + bf_lo(qv.y) * za.z + bf_hi(qv.y) * za.w +
                          bf_lo(qv.z) * zb.x + bf_hi(qv.z) * zb.y + bf_lo(qv.w) * zb.z + bf_hi(qv.w) * zb.w;
                }
                dpart[128 * h + r] = di;
            }
            // (b) den; P = dO / den in place (bf16); g = -P . num / den from that bf16 P.  The
            // dO wait is also the barrier after which both halves of phi(q) . z are in.
            if (!CG::all(mbar_wait(&bar->full_p, ph, err, LA_ERR_TIMEOUT))) { ok = false; break; }
            const float den = valid ? dpart[r] + dpart[128 + r] : 1.f;
            const float inv = 1.f / den;
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) {
                uint4* pp = reinterpret_cast<uint4*>(sP + chunk_off(r, 8 * h + c8));
                uint4 v4 = *pp;
                uint32_t* u = reinterpret_cast<uint32_t*>(&v4);
#pragma unroll
                for (int e = 0; e < 4; ++e) u[e] = pack_bf16x2(bf_lo(u[e]) * inv, bf_hi(u[e]) * inv);
                *pp = v4;
            }
            if (!CG::all(mbar_wait(&bar->num_done, ph, err, LA_ERR_TIMEOUT))) { ok = false; break; }
            tc_fence_after();
            {
                float dot = 0.f;
#pragma unroll
                for (int cb = 0; cb < 2; ++cb) {
                    uint32_t w[32];
                    tmem_ld32(tmem + lb + kQY + 32 * cb, w);
                    tmem_ld_wait();
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        const uint4 v4 = *reinterpret_cast<const uint4*>(sP + chunk_off(r, 8 * h + 4 * cb + c4));
                        const uint32_t* u = reinterpret_cast<const uint32_t*>(&v4);
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            dot += bf_lo(u[e]) * __uint_as_float(w[8 * c4 + 2 * e]) +
                                   bf_hi(u[e]) * __uint_as_float(w[8 * c4 + 2 * e + 1]);
                    }
                }
                tpart[128 * h + r] = dot;
            }
            fence_proxy_async_smem();
            CG::sync();
            const float g = valid ? -(tpart[r] + tpart[128 + r]) * inv : 0.f;
            if (h == 0) gsh[r] = g;
            tc_fence_before();
            CG::sync();
            if (ct == 0) {
                mbar_arrive(&bar->p_ready);
                mbar_arrive(&bar->empty_p);  // the compute group's last read of P in this chunk
            }
            // (c) the chunk's column sums of g phi(q) (weighted column sums of the Q tile)
            {
                float zp[2][8];
#pragma unroll
                for (int b = 0; b < 2; ++b)
#pragma unroll
                    for (int e = 0; e < 8; ++e) zp[b][e] = 0.f;
#pragma unroll
                for (int j = 0; j < CG::kJ; ++j) {
                    const uint4 qv = *reinterpret_cast<const uint4*>(sQ + CG::vec_off(ct, j));
                    const uint32_t* u = reinterpret_cast<const uint32_t*>(&qv);
                    const float wr = gsh[CG::vec_row(ct, j)];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        zp[CG::vec_block(j)][2 * e] = fmaf(wr, bf_lo(u[e]), zp[CG::vec_block(j)][2 * e]);
                        zp[CG::vec_block(j)][2 * e + 1] = fmaf(wr, bf_hi(u[e]), zp[CG::vec_block(j)][2 * e + 1]);
                    }
                }
                CG::column_part(zp, drpart, ct);
            }
            CG::sync();  // drpart is complete
            // (d) dq = (dQ~ + g z) * phi'(q) on this thread's 64 columns, staged for one TMA store
            if (ct == kStoreThread) bulk_wait_read_all();  // the previous dq store has left the staging tile
            if (!CG::all(mbar_wait(&bar->dq_done, ph, err, LA_ERR_TIMEOUT))) { ok = false; break; }
            tc_fence_after();
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) {
                uint32_t w[32];
                tmem_ld32(tmem + lb + kQY + 32 * cb, w);
                tmem_ld_wait();
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    const uint4 qv = *reinterpret_cast<const uint4*>(sQ + chunk_off(r, 8 * h + 4 * cb + c4));
                    const uint32_t qu[4] = {qv.x, qv.y, qv.z, qv.w};
                    uint4 o4;
                    uint32_t* ou = reinterpret_cast<uint32_t*>(&o4);
                    const int c = 64 * h + 32 * cb + 8 * c4;
                    const float4 za = *reinterpret_cast<const float4*>(zsh + c);
                    const float4 zb = *reinterpret_cast<const float4*>(zsh + c + 4);
                    const float zr[8] = {za.x, za.y, za.z, za.w, zb.x, zb.y, zb.z, zb.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float a0 = (__uint_as_float(w[8 * c4 + 2 * e]) + g * zr[2 * e]) * dphi_from_phi(bf_lo(qu[e]));
                        const float a1 =
                            (__uint_as_float(w[8 * c4 + 2 * e + 1]) + g * zr[2 * e + 1]) * dphi_from_phi(bf_hi(qu[e]));
                        ou[e] = pack_bf16x2(a0, a1);
                    }
                    *reinterpret_cast<uint4*>(sOb + chunk_off(r, 8 * h + 4 * cb + c4)) = o4;
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            CG::sync();  // every read of this Q buffer by the compute group is done
            if (ct == 0) {
                mbar_arrive(&bar->y_free);
                mbar_arrive(&bar->empty_q[i & 1]);
            }
            if (ct == kStoreThread) {
                check_tile(0, c0, bh, N), tma_store_3d(&tm_dq, sOb, 0, c0, bh);
                if (D > 64) check_tile(64, c0, bh, N), tma_store_3d(&tm_dq, sOb + kBlockBytes, 64, c0, bh);
                bulk_commit();
            }
            if (ct < kD) racc[ct] += CG::column_sum(drpart, ct);
        }
        if (ct == kStoreThread) bulk_wait_all();
        // the segment's sums out: R from TMEM, r from shared memory
        if (ok && nloc > 0 && CG::all(mbar_wait(&bar->final_mma, 0, err, LA_ERR_TIMEOUT))) {
            tc_fence_after();
            float* out = seg_R + ((size_t)bh * P + p) * kE;
            tmem_row_to_global<64>(tmem + lb + kQR, out + (size_t)r * kD + 64 * h);
            if (ct < kD) out[(size_t)kD * kD + ct] = racc[ct];
        }
        tc_fence_before();
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

// ------------------------------------------------------------------ key pass
// TMEM: two accumulator sets at 0 and 256, each DK [+0,+128) dK~ and DV [+128,+256) dV.
// K and V are double-buffered in shared memory and the accumulators in TMEM, and phi on
// the next chunk's K tile runs while this chunk's products are formed, so the products
// of chunk i + 1 overlap the epilogue of chunk i.  Every per-buffer barrier is used once
// per two chunks and never runs a phase ahead of its waiter: a buffer is refilled only
// after its previous chunk has been consumed.
constexpr uint32_t kKDK = 0, kKDV = 128, kKAcc = 256;

struct KBars {
    uint64_t full[2], empty[2];  // K and V buffers; empty: the MMA's last read and the epilogue's
    uint64_t k_ready[2], kv_done[2], acc_free[2];
    uint64_t final_mma;
};

struct KSmem {
    static constexpr int K0 = 0, V0 = 2 * kTileBytes, Rb = 4 * kTileBytes;  // K, V buffers 0 and 1
    static constexpr int Ok = 5 * kTileBytes, Ov = 6 * kTileBytes;          // dk, dv tiles for the TMA stores
    static constexpr int rsh = 7 * kTileBytes;                              // float[128] r
    static constexpr int bars = rsh + 512;
    static constexpr int tmem_slot = bars + 256;
    static constexpr int total = tmem_slot + 16;
};
constexpr size_t kKSmemBytes = KSmem::total + 1024;
static_assert(kKSmemBytes <= 232448, "key pass: shared memory above the per-CTA limit");

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
tc_noncausal_bwd_key_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                            const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                            const float* __restrict__ totR, int N, int nchunks, int cps, int* err) {
    extern __shared__ uint8_t smem_raw[];
    pdl_enter();  // launched with programmatic dependent launch
    constexpr int kKd = D / 16;
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    auto sKb = [&](int b) { return base + KSmem::K0 + b * kTileBytes; };
    auto sVb = [&](int b) { return base + KSmem::V0 + b * kTileBytes; };
    uint8_t* sRb = base + KSmem::Rb;
    uint8_t* sOk = base + KSmem::Ok;
    uint8_t* sOv = base + KSmem::Ov;
    float* rsh = reinterpret_cast<float*>(base + KSmem::rsh);
    KBars* bar = reinterpret_cast<KBars*>(base + KSmem::bars);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + KSmem::tmem_slot);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int p = blockIdx.x, bh = blockIdx.y;
    const int cbeg = p * cps, cend = min(nchunks, cbeg + cps), nloc = cend - cbeg;
    check_plan(p, (int)gridDim.x, cbeg, cend, nchunks, N);
    const float* tot = totR + (size_t)bh * kE;

    if (tid == 0) {
        uint64_t* b = reinterpret_cast<uint64_t*>(bar);
        for (int x = 0; x < (int)(sizeof(KBars) / 8); ++x) mbar_init(b + x, 1);
        mbar_init(&bar->empty[0], 2);  // one MMA commit + one compute-group arrival each
        mbar_init(&bar->empty[1], 2);
        fence_mbar_init();
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_dk);
        tma_prefetch_desc(&tm_dv);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    if (warp >= 2) {  // R as the bf16 operand (row r = dk, this thread's 64 columns), r in fp32
        const int ct = tid - 64, h = (warp - 2) >> 2, r = 32 * (warp & 3) + lane;
#pragma unroll
        for (int cb = 0; cb < 2; ++cb) {
            uint32_t w[32];
            const float4* src = reinterpret_cast<const float4*>(tot + (size_t)r * kD + 64 * h + 32 * cb);
#pragma unroll
            for (int x4 = 0; x4 < 8; ++x4) {  // 16-byte loads: the workspace and each record row are 16-byte aligned
                const float4 f = src[x4];
                w[4 * x4] = __float_as_uint(f.x);
                w[4 * x4 + 1] = __float_as_uint(f.y);
                w[4 * x4 + 2] = __float_as_uint(f.z);
                w[4 * x4 + 3] = __float_as_uint(f.w);
            }
            row32_to_tile(w, sRb, r, 8 * h + 4 * cb);
        }
        if (ct < kD) rsh[ct] = tot[(size_t)kD * kD + ct];
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            int armed[2] = {-1, -1};
            for (int i = 0; i < nloc; ++i) {
                const int t0 = (cbeg + i) * kC, b = i & 1;
                if (!mbar_wait(&bar->empty[b], ((i >> 1) & 1) ^ 1, err, LA_ERR_TIMEOUT)) break;
                mbar_arrive_expect_tx(&bar->full[b], 2 * kTileBytes);
                check_tile(0, t0, bh, N), tma_load_3d(sKb(b), &tm_k, 0, t0, bh, &bar->full[b]);
                check_tile(64, t0, bh, N), tma_load_3d(sKb(b) + kBlockBytes, &tm_k, 64, t0, bh, &bar->full[b]);
                check_tile(0, t0, bh, N), tma_load_3d(sVb(b), &tm_v, 0, t0, bh, &bar->full[b]);
                check_tile(64, t0, bh, N), tma_load_3d(sVb(b) + kBlockBytes, &tm_v, 64, t0, bh, &bar->full[b]);
                armed[b] = i;
            }
            // no copy may still be landing when the CTA exits
            for (int b = 0; b < 2; ++b)
                if (armed[b] >= 0) mbar_wait(&bar->full[b], (armed[b] >> 1) & 1, err, LA_ERR_TIMEOUT);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t id_kk = idesc_bf16_f32(128, 128, 0, 0);
            constexpr uint32_t id_kmn = idesc_bf16_f32(128, 128, 0, 1);
            const uint32_t aRb = smem_u32(sRb);
            for (int i = 0; i < nloc; ++i) {
                const int b = i & 1;
                const uint32_t use = (i >> 1) & 1;  // parity of this buffer's current use
                if (!mbar_wait(&bar->k_ready[b], use, err, LA_ERR_TIMEOUT) ||
                    !mbar_wait(&bar->acc_free[b], use ^ 1, err, LA_ERR_TIMEOUT))
                    break;
                tc_fence_after();
                const uint32_t aK = smem_u32(sKb(b)), aV = smem_u32(sVb(b)), acc = tmem + kKAcc * b;
#pragma unroll
                for (int kk = 0; kk < kKd; ++kk)  // dK~ = V R^T (rows = keys)
                    mma_ss(acc + kKDK, desc_kmajor(aV, kk), desc_kmajor(aRb, kk), id_kk, kk > 0);
#pragma unroll
                for (int kk = 0; kk < kKd; ++kk)  // dV = phi(K) R
                    mma_ss(acc + kKDV, desc_kmajor(aK, kk), desc_mnmajor(aRb, kk), id_kmn, kk > 0);
                mma_commit(&bar->kv_done[b]);
                mma_commit(&bar->empty[b]);  // last MMA read of this K and V buffer
            }
            mma_commit(&bar->final_mma);
            mbar_wait(&bar->final_mma, 0, err, LA_ERR_TIMEOUT);
        }
    } else {
        const int ct = tid - 64;
        const int h = (warp - 2) >> 2;
        const int r = 32 * (warp & 3) + lane;
        const uint32_t lb = ((uint32_t)(32 * (warp & 3)) << 16) + 64 * h;
        bool ok = CG::all(true);
        // phi on K in place for chunk j (buffer j & 1), then hand it to the MMA
        auto phi_k = [&](int j) -> bool {
            const int b = j & 1, n = min(kC, N - (cbeg + j) * kC);
            if (!CG::all(mbar_wait(&bar->full[b], (j >> 1) & 1, err, LA_ERR_TIMEOUT))) return false;
            CG::phi_tile(sKb(b), nullptr, ct, n, D, nullptr, nullptr);
            fence_proxy_async_smem();
            CG::sync();
            if (ct == 0) mbar_arrive(&bar->k_ready[b]);
            return true;
        };
        if (nloc > 0) ok = phi_k(0);
        for (int i = 0; i < nloc && ok; ++i) {
            const int b = i & 1;
            const int c0 = (cbeg + i) * kC;
            // (a) the next chunk's phi while this chunk's products are formed
            if (i + 1 < nloc && !phi_k(i + 1)) { ok = false; break; }
            // (b) dk = (dK~ + r) * phi'(k) (phi(k) read back from the K tile) and dv, this
            // thread's 64 columns of key row r, staged for one TMA store each
            if (ct == kStoreThread) bulk_wait_read_all();  // the previous stores have left the staging tiles
            if (!CG::all(mbar_wait(&bar->kv_done[b], (i >> 1) & 1, err, LA_ERR_TIMEOUT))) { ok = false; break; }
            tc_fence_after();
            const uint8_t* sK = sKb(b);
            const uint32_t acc = tmem + lb + kKAcc * b;
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) {
                uint32_t w[32];
                tmem_ld32(acc + kKDK + 32 * cb, w);
                tmem_ld_wait();
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    const int lc = 8 * h + 4 * cb + c4;
                    const uint4 kv = *reinterpret_cast<const uint4*>(sK + chunk_off(r, lc));
                    const uint32_t* ku = reinterpret_cast<const uint32_t*>(&kv);
                    const float4 ra = *reinterpret_cast<const float4*>(rsh + 8 * lc);
                    const float4 rb = *reinterpret_cast<const float4*>(rsh + 8 * lc + 4);
                    const float rr[8] = {ra.x, ra.y, ra.z, ra.w, rb.x, rb.y, rb.z, rb.w};
                    uint4 o4;
                    uint32_t* ou = reinterpret_cast<uint32_t*>(&o4);
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        ou[e] = pack_bf16x2((__uint_as_float(w[8 * c4 + 2 * e]) + rr[2 * e]) * dphi_from_phi(bf_lo(ku[e])),
                                            (__uint_as_float(w[8 * c4 + 2 * e + 1]) + rr[2 * e + 1]) *
                                                dphi_from_phi(bf_hi(ku[e])));
                    *reinterpret_cast<uint4*>(sOk + chunk_off(r, lc)) = o4;
                }
            }
            tmem_half_row_to_tile(acc + kKDV, sOv, r, h);
            fence_proxy_async_smem();
            tc_fence_before();
            CG::sync();  // this accumulator set is read and this K buffer is no longer used
            if (ct == 0) {
                mbar_arrive(&bar->acc_free[b]);
                mbar_arrive(&bar->empty[b]);
            }
            if (ct == kStoreThread) {
                check_tile(0, c0, bh, N), tma_store_3d(&tm_dk, sOk, 0, c0, bh);
                check_tile(0, c0, bh, N), tma_store_3d(&tm_dv, sOv, 0, c0, bh);
                if (D > 64) {
                    check_tile(64, c0, bh, N), tma_store_3d(&tm_dk, sOk + kBlockBytes, 64, c0, bh);
                    check_tile(64, c0, bh, N), tma_store_3d(&tm_dv, sOv + kBlockBytes, 64, c0, bh);
                }
                bulk_commit();
            }
        }
        if (ct == kStoreThread) bulk_wait_all();
        tc_fence_before();
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

cudaError_t tc_noncausal_bwd_query(const void* q, const void* dout, void* dq, const float* totS, float* seg_R,
                                   const la_shape& s, const Plan& p, cudaStream_t st) {
    const int BH = s.B * s.H;
    CUtensorMap tq, td, tdq;
    const int D = s.Dk;  // = s.Dv: 128, or 64 padded to the 128-wide tiles
    if (!make_tmap_bf16_rows(&tq, q, BH, s.N, D, kC) || !make_tmap_bf16_rows(&td, dout, BH, s.N, D, kC) ||
        !make_tmap_bf16_rows(&tdq, dq, BH, s.N, D, kC))
        return cudaErrorInvalidValue;
    auto kern = D == 128 ? tc_noncausal_bwd_query_kernel<128> : tc_noncausal_bwd_query_kernel<64>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kQSmemBytes);
    if (e != cudaSuccess) return e;
    launch_begin("tc_noncausal_bwd_query", st);
    const cudaError_t le = launch_pdl(kern, dim3(p.P, BH), dim3(kThreads), kQSmemBytes, st, tq, td, tdq, totS, seg_R, s.N, p.nchunks, p.cps, p.P,
                                                       device_error_word());
    const cudaError_t le2 = launch_end("tc_noncausal_bwd_query", st);
    return le != cudaSuccess ? le : le2;
}

cudaError_t tc_noncausal_bwd_key(const void* k, const void* v, void* dk, void* dv, const float* totR,
                                 const la_shape& s, const Plan& p, cudaStream_t st) {
    const int BH = s.B * s.H;
    CUtensorMap tk, tv, tdk, tdv;
    const int D = s.Dk;
    if (!make_tmap_bf16_rows(&tk, k, BH, s.N, D, kC) || !make_tmap_bf16_rows(&tv, v, BH, s.N, D, kC) ||
        !make_tmap_bf16_rows(&tdk, dk, BH, s.N, D, kC) || !make_tmap_bf16_rows(&tdv, dv, BH, s.N, D, kC))
        return cudaErrorInvalidValue;
    auto kern = D == 128 ? tc_noncausal_bwd_key_kernel<128> : tc_noncausal_bwd_key_kernel<64>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kKSmemBytes);
    if (e != cudaSuccess) return e;
    launch_begin("tc_noncausal_bwd_key", st);
    const cudaError_t le = launch_pdl(kern, dim3(p.P, BH), dim3(kThreads), kKSmemBytes, st, tk, tv, tdk, tdv, totR, s.N, p.nchunks, p.cps,
                                                       device_error_word());
    const cudaError_t le2 = launch_end("tc_noncausal_bwd_key", st);
    return le != cudaSuccess ? le : le2;
}

}  // namespace la
