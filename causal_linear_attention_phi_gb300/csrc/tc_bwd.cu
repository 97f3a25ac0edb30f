// tc_bwd.cu -- tensor-core (tcgen05 / TMEM / TMA) kernels of the causal
// backward for bf16 inputs with Dk = Dv = 128, chunks of 128 positions.
//
// The gradient is a cumulative sum ("[논문 리뷰] Transformers are RNNs ..."
// (velog review), 3.5 Gradient Computation): states are recomputed, never
// stored per position.  With den_i = phi(q_i)^T z_i, P_i = dO_i / den_i,
// g_i = -P_i . o_i, per chunk c (A = tril(Q~ K~^T), D = tril(P V^T + g 1^T)):
//   dQ~ = P S_prev^T + g z_prev^T + D K~
//   dK~ = V R_next^T + 1 r_next^T + D^T Q~
//   dV  = K~ R_next + A^T P
// where R_next = sum over later positions of phi(q_i) P_i^T and r_next = sum g_i phi(q_i).
//
// Forward sweep kernel: chunks in order, S and the segment's R contribution in
// TMEM; recomputes num and den as the forward does, derives P and g (g from the
// bf16 P the products use), writes dq and the per-position (den, g).  dq is the
// difference of two terms that nearly cancel when phi(k) varies little, so two
// products carry more than bf16: A = tril(Q~ K~^T), whose entries sit near the
// head size (so a bf16 copy loses their variation), enters A V as a hi + lo pair,
// and D K~ is formed as rowsum(D) 1^T + D (K~ - 1): the row sums exact in fp32,
// the product on a bf16 copy of D and a bf16 copy of phi(K) - 1, which is small
// where phi(k) is near 1 and so keeps its low bits.
// Reverse sweep kernel: chunks in reverse order with R_next in TMEM; every
// product is taken with the keys as the M (TMEM lane) dimension so dk and dv
// come out row by row.  1/den is folded into the query operand, Q' = phi(Q) /
// den, so dO enters unscaled: A'^T = K~ Q'^T (= A^T / den), D'^T = tril(V dO^T
// + (g den) 1^T), dK~ = V R_next^T + 1 r_next^T + D'^T Q', dV = K~ R_next +
// A'^T dO, R_next += Q'^T dO, r_next += sum of (g den) Q'.
//
// Roles: warp 0 TMA, warp 1 TMEM owner and MMA issuer, the other warps the
// compute group: 8 warps in the forward sweep, 16 in the reverse sweep.  For
// row-wise TMEM work warp w reads TMEM lanes 32 (w % 4) .. +31 (row r of a
// 128-row tile) and its share of the columns: half h = (w - 2) / 4 with 8 warps,
// quarter qt = (w - 2) / 4 with 16.  All waits are bounded.
#include "tc_common.cuh"

namespace la {
namespace {
using namespace sm100;
using namespace tc;

using FG = Grp<256>;  // forward sweep: 8 compute warps
using RG = Grp<512>;  // reverse sweep: 16 compute warps (4 per SM sub-partition)
constexpr int kThreadsFS = 64 + 256, kThreadsRS = 64 + 512;  // + the TMA and MMA warps

// ------------------------------------------------------------------ forward sweep
// TMEM: S [0,128) fp32 state; R [128,256) segment sum of phi(q) P^T;
// X [256,384): QK^T fp32 -> A as bf16 hi + lo -> P V^T fp32 -> D bf16.  Each 32-key
// block b of fp32 columns X[32b, 32b+32) is rewritten in place by the thread that
// read it: A_hi (bf16 pairs) in X[32b, 32b+16) and A_lo in X[32b+16, 32b+32), later
// D in X[32b, 32b+16); so the MMA's A operand for K step kk (keys 16kk..16kk+15)
// sits at column 32 (kk / 2) + 8 (kk % 2) (+16 for A_lo).
// Y [384,512): O = phi(Q) S_prev + A V (numerator) -> dQ~.
constexpr uint32_t kFS = 0, kFR = 128, kFX = 256, kFY = 384;
__device__ __forceinline__ uint32_t xcol(int kk) { return 32 * (kk >> 1) + 8 * (kk & 1); }

// Q, V and dO arrive (full_qv) and are released (empty_qv: the MMA's last read of
// them and the compute group's last read of Q) apart from K (full_k, empty_k:
// the dq products read it last), so the next chunk's Q, V and dO load during
// this chunk's D and dq work.
struct FwdSweepBars {
    uint64_t full_qv, empty_qv, full_k, empty_k;
    uint64_t qk_ready, sb_ready, a_ready, p_ready, d_ready;
    uint64_t qk_done, o_done, pv_done, dq_done;
    uint64_t final_mma;
};

struct FwdSweepSmem {
    // KLo: bf16(phi(K) - 1), the operand of D (K~ - 1)
    static constexpr int Q = 0, K = kTileBytes, KLo = 2 * kTileBytes, V = 3 * kTileBytes, P = 4 * kTileBytes;
    static constexpr int Sb = 5 * kTileBytes;   // bf16 S_prev; after the dq products, the dq tile for the TMA store
    static constexpr int zsh = 6 * kTileBytes;  // float[128] z_prev
    static constexpr int zpart = zsh + 512;     // float[8][128] per-warp column sums of this chunk's phi(k)
    static constexpr int racc = zpart + 4096;   // float[128] segment sum of g phi(q)
    static constexpr int drpart = racc + 512;   // float[8][128] per-warp column sums of this chunk's g phi(q)
    static constexpr int gsh = drpart + 4096;   // float[128] g of the chunk's rows
    static constexpr int rpart = gsh + 512;     // float[2][128] row sums of A, later of D, per column half
    static constexpr int dpart = rpart + 1024;  // float[2][128] phi(q) . z_prev, per column half
    static constexpr int tpart = dpart + 1024;  // float[2][128] P . num, per column half
    static constexpr int bars = tpart + 1024;
    static constexpr int tmem_slot = bars + 256;
    static constexpr int total = tmem_slot + 16;
};

// D: the head size, 128 or 64 (padded to the 128-wide tiles); a template
// parameter so that the full-width kernels carry no column test.
template <int D>
__global__ void __launch_bounds__(kThreadsFS, 1)
tc_bwd_forward_sweep_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                            const __grid_constant__ CUtensorMap tm_dq, const float* __restrict__ seg_S,
                            float* __restrict__ seg_R, float* __restrict__ den_g, int N, int nchunks, int cps, int P,
                            int* err) {
    extern __shared__ uint8_t smem_raw[];
    constexpr int kKd = D / 16;  // K steps of a product over a head dimension (a 64-wide head is zero above)
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = base + FwdSweepSmem::Q;
    uint8_t* sK = base + FwdSweepSmem::K;
    uint8_t* sKLo = base + FwdSweepSmem::KLo;
    uint8_t* sV = base + FwdSweepSmem::V;
    uint8_t* sP = base + FwdSweepSmem::P;
    uint8_t* sSb = base + FwdSweepSmem::Sb;
    float* zsh = reinterpret_cast<float*>(base + FwdSweepSmem::zsh);
    float* zpart = reinterpret_cast<float*>(base + FwdSweepSmem::zpart);
    float* racc = reinterpret_cast<float*>(base + FwdSweepSmem::racc);
    float* drpart = reinterpret_cast<float*>(base + FwdSweepSmem::drpart);
    float* gsh = reinterpret_cast<float*>(base + FwdSweepSmem::gsh);
    float* rpart = reinterpret_cast<float*>(base + FwdSweepSmem::rpart);
    float* dpart = reinterpret_cast<float*>(base + FwdSweepSmem::dpart);
    float* tpart = reinterpret_cast<float*>(base + FwdSweepSmem::tpart);
    FwdSweepBars* bar = reinterpret_cast<FwdSweepBars*>(base + FwdSweepSmem::bars);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + FwdSweepSmem::tmem_slot);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int p = blockIdx.x, bh = blockIdx.y;
    const int cbeg = p * cps, cend = min(nchunks, cbeg + cps), nloc = cend - cbeg;
    const size_t E = state_elems(kD, kD);
    check_plan(p, P, cbeg, cend, nchunks, N);
    record_ok(bh, p, P, E - 1, E);

    if (tid == 0) {
        uint64_t* b = reinterpret_cast<uint64_t*>(bar);
        for (int x = 0; x < (int)(sizeof(FwdSweepBars) / 8); ++x) mbar_init(b + x, 1);
        mbar_init(&bar->empty_qv, 2);  // one MMA commit + one compute-group arrival
        fence_mbar_init();
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_do);
        tma_prefetch_desc(&tm_dq);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_enter();  // the previous kernel's outputs (segment records, (den, g)) are visible from here on

    if (warp == 0) {
        if (lane == 0) {
            int armed_qv = -1, armed_k = -1;
            for (int i = 0; i < nloc; ++i) {
                const int t0 = (cbeg + i) * kC;
                if (!mbar_wait(&bar->empty_qv, (i & 1) ^ 1, err, LA_ERR_TIMEOUT)) break;
                mbar_arrive_expect_tx(&bar->full_qv, 3 * kTileBytes);
                check_tile(64, t0, bh, N);
                tma_load_3d(sQ, &tm_q, 0, t0, bh, &bar->full_qv);
                tma_load_3d(sQ + kBlockBytes, &tm_q, 64, t0, bh, &bar->full_qv);
                tma_load_3d(sV, &tm_v, 0, t0, bh, &bar->full_qv);
                tma_load_3d(sV + kBlockBytes, &tm_v, 64, t0, bh, &bar->full_qv);
                tma_load_3d(sP, &tm_do, 0, t0, bh, &bar->full_qv);
                tma_load_3d(sP + kBlockBytes, &tm_do, 64, t0, bh, &bar->full_qv);
                armed_qv = i;
                if (!mbar_wait(&bar->empty_k, (i & 1) ^ 1, err, LA_ERR_TIMEOUT)) break;
                mbar_arrive_expect_tx(&bar->full_k, kTileBytes);
                tma_load_3d(sK, &tm_k, 0, t0, bh, &bar->full_k);
                tma_load_3d(sK + kBlockBytes, &tm_k, 64, t0, bh, &bar->full_k);
                armed_k = i;
            }
            // no copy may still be landing when the CTA exits
            if (armed_qv >= 0) mbar_wait(&bar->full_qv, armed_qv & 1, err, LA_ERR_TIMEOUT);
            if (armed_k >= 0) mbar_wait(&bar->full_k, armed_k & 1, err, LA_ERR_TIMEOUT);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t id_kk = idesc_bf16_f32(128, 128, 0, 0);
            constexpr uint32_t id_kmn = idesc_bf16_f32(128, 128, 0, 1);
            constexpr uint32_t id_mnmn = idesc_bf16_f32(128, 128, 1, 1);
            const uint32_t aQ = smem_u32(sQ), aK = smem_u32(sK), aKLo = smem_u32(sKLo), aV = smem_u32(sV),
                           aP = smem_u32(sP), aSb = smem_u32(sSb);
            for (int i = 0; i < nloc; ++i) {
                const uint32_t ph = i & 1;
                if (!mbar_wait(&bar->sb_ready, ph, err, LA_ERR_TIMEOUT)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kKd; ++kk)  // Y = Q~ S_prev (needs phi(Q) and S_prev only)
                    mma_ss(tmem + kFY, desc_kmajor(aQ, kk), desc_mnmajor(aSb, kk), id_kmn, kk > 0);
                if (!mbar_wait(&bar->qk_ready, ph, err, LA_ERR_TIMEOUT)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kKd; ++kk)  // X = Q~ K~^T
                    mma_ss(tmem + kFX, desc_kmajor(aQ, kk), desc_kmajor(aK, kk), id_kk, kk > 0);
                mma_commit(&bar->qk_done);
                if (!mbar_wait(&bar->a_ready, ph, err, LA_ERR_TIMEOUT)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {  // Y += A V as A_hi V + A_lo V
                    mma_ts(tmem + kFY, tmem + kFX + xcol(kk), desc_mnmajor(aV, kk), id_kmn, 1);
                    mma_ts(tmem + kFY, tmem + kFX + xcol(kk) + 16, desc_mnmajor(aV, kk), id_kmn, 1);
                }
                mma_commit(&bar->o_done);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // S += K~^T V
                    mma_ss(tmem + kFS, desc_mnmajor(aK, kk), desc_mnmajor(aV, kk), id_mnmn, 1);
                if (!mbar_wait(&bar->p_ready, ph, err, LA_ERR_TIMEOUT)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kKd; ++kk)  // X = P V^T
                    mma_ss(tmem + kFX, desc_kmajor(aP, kk), desc_kmajor(aV, kk), id_kk, kk > 0);
                mma_commit(&bar->pv_done);
#pragma unroll
                for (int kk = 0; kk < kKd; ++kk)  // Y = P S_prev^T (Y is free: O was read before p_ready)
                    mma_ss(tmem + kFY, desc_kmajor(aP, kk), desc_kmajor(aSb, kk), id_kk, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // R += Q~^T P
                    mma_ss(tmem + kFR, desc_mnmajor(aQ, kk), desc_mnmajor(aP, kk), id_mnmn, (i > 0 || kk > 0));
                mma_commit(&bar->empty_qv);  // last MMA read of Q, V and P in this chunk
                if (!mbar_wait(&bar->d_ready, ph, err, LA_ERR_TIMEOUT)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // Y += D (K~ - 1); the rowsum(D) 1^T part is added in fp32
                    mma_ts(tmem + kFY, tmem + kFX + xcol(kk), desc_mnmajor(aKLo, kk), id_kmn, 1);
                mma_commit(&bar->dq_done);
                mma_commit(&bar->empty_k);  // last read of K and K~ - 1
            }
            mma_commit(&bar->final_mma);
            mbar_wait(&bar->final_mma, 0, err, LA_ERR_TIMEOUT);
        }
    } else {
        const int ct = tid - 64;
        const int h = (warp - 2) >> 2;
        const int r = 32 * (warp & 3) + lane;
        const uint32_t lb = ((uint32_t)(32 * (warp & 3)) << 16) + 64 * h;  // this thread's row half
        const float* pre = seg_S + ((size_t)bh * P + p) * E;
        global_row_to_tmem<64>(pre + (size_t)r * kD + 64 * h, tmem + lb + kFS);  // S_prev row r, this half
        if (ct < 128) {
            zsh[ct] = record_ok(bh, p, P, (size_t)kD * kD + ct, E) ? pre[(size_t)kD * kD + ct] : 0.f;
            racc[ct] = 0.f;
        }
        if (D <= 64) {  // phi leaves the lo tile's upper column block unwritten: keep it zero
            for (int x = ct; x < kBlockBytes / 16; x += 256)
                reinterpret_cast<uint4*>(sKLo + kBlockBytes)[x] = make_uint4(0u, 0u, 0u, 0u);
            fence_proxy_async_smem();
        }
        tc_fence_before();
        bool ok = FG::all(true);
        float* dgh = den_g + (size_t)bh * N * 2;
        for (int i = 0; i < nloc && ok; ++i) {
            const uint32_t ph = i & 1;
            const int c0 = (cbeg + i) * kC, n = min(kC, N - c0);
            const bool valid = r < n;
            // (a) phi on Q in place; S_prev -> its bf16 copy (rows = dk; this thread's 64
            // columns).  S and Y are settled: the previous chunk's dq_done, which follows
            // every earlier MMA, has been awaited.
            if (ct == kStoreThread) bulk_wait_read_all();  // the previous dq store has left the Sb tile
            if (!FG::all(mbar_wait(&bar->full_qv, ph, err, LA_ERR_TIMEOUT))) { ok = false; break; }
            tc_fence_after();
            FG::phi_tile(sQ, nullptr, ct, n, D, nullptr, nullptr);
            tmem_half_row_to_tile(tmem + lb + kFS, sSb, r, h);
            tc_fence_before();
            fence_proxy_async_smem();
            FG::sync();
            if (ct == 0) mbar_arrive(&bar->sb_ready);
            // (b) phi on K: bf16 phi(K) in place, bf16(phi(K) - 1) beside it, per-warp column
            // sums of the bf16 phi(K) into zpart
            if (!FG::all(mbar_wait(&bar->full_k, ph, err, LA_ERR_TIMEOUT))) { ok = false; break; }
            FG::phi_tile<true>(sK, sKLo, ct, n, D, nullptr, zpart);
            fence_proxy_async_smem();
            FG::sync();
            if (ct == 0) mbar_arrive(&bar->qk_ready);
            // while Q K^T is formed: phi(q_r) on this thread's 64 columns stays in registers for
            // phi'(q) in the dq epilogue (Q is released before it); phi(q_r) . z_prev
            uint32_t qrow[32];
            {
                float di = 0.f;
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) {
                    const int lc = 8 * h + c8;
                    const uint4 qv = *reinterpret_cast<const uint4*>(sQ + chunk_off(r, lc));
                    qrow[4 * c8 + 0] = qv.x;
                    qrow[4 * c8 + 1] = qv.y;
                    qrow[4 * c8 + 2] = qv.z;
                    qrow[4 * c8 + 3] = qv.w;
                    const float4 za = *reinterpret_cast<const float4*>(zsh + 8 * lc);
                    const float4 zb = *reinterpret_cast<const float4*>(zsh + 8 * lc + 4);
                    di += bf_lo(qv.x) * za.x + bf_hi(qv.x) * za.y + bf_lo(qv.y) * za.z + bf_hi(qv.y) * za.w +
                          bf_lo(qv.z) * zb.x + bf_hi(qv.z) * zb.y + bf_lo(qv.w) * zb.z + bf_hi(qv.w) * zb.w;
                }
                dpart[128 * h + r] = di;
            }
            // (c) A = tril(QK^T) as bf16 hi + lo on this thread's keys [64h, 64h+64), in place
            // (see the X layout); its fp32 row sums (equal to those of hi + lo, the operands A V
            // uses, to about 2^-17) go to den
            if (!FG::all(mbar_wait(&bar->qk_done, ph, err, LA_ERR_TIMEOUT))) { ok = false; break; }
            tc_fence_after();
            {
                float rs = 0.f;
#pragma unroll
                for (int cb = 0; cb < 2; ++cb) {
                    const int j0 = 64 * h + 32 * cb;
                    uint32_t hi[16], lo[16];
                    if (j0 > r) {
#pragma unroll
                        for (int x = 0; x < 16; ++x) hi[x] = lo[x] = 0u;
                    } else {
                        uint32_t w[32];
                        tmem_ld32(tmem + lb + kFX + 32 * cb, w);
                        tmem_ld_wait();
                        if (j0 + 31 < (r & ~31)) {  // below the diagonal for the whole warp: no mask
#pragma unroll
                            for (int x = 0; x < 16; ++x) {
                                const float a0 = __uint_as_float(w[2 * x]), a1 = __uint_as_float(w[2 * x + 1]);
                                hi[x] = pack_bf16x2(a0, a1);
                                lo[x] = pack_bf16x2(a0 - bf_lo(hi[x]), a1 - bf_hi(hi[x]));
                                rs += a0 + a1;
                            }
                        } else {
#pragma unroll
                            for (int x = 0; x < 16; ++x) {
                                const int j = j0 + 2 * x;
                                const float a0 = j <= r ? __uint_as_float(w[2 * x]) : 0.f;
                                const float a1 = j + 1 <= r ? __uint_as_float(w[2 * x + 1]) : 0.f;
                                hi[x] = pack_bf16x2(a0, a1);
                                lo[x] = pack_bf16x2(a0 - bf_lo(hi[x]), a1 - bf_hi(hi[x]));
                                rs += a0 + a1;
                            }
                        }
                    }
                    tmem_st16(tmem + lb + kFX + 32 * cb, hi);
                    tmem_st16(tmem + lb + kFX + 32 * cb + 16, lo);
                }
                rpart[128 * h + r] = rs;
                tmem_st_wait();
            }
            tc_fence_before();
            FG::sync();
            if (ct == 0) mbar_arrive(&bar->a_ready);
            // (d) den (the row sums of A and phi(q) . z_prev are in); P = dO / den in place (bf16)
            // on this thread's 64 columns while A V is formed; then g = -P . num / den from
            // that bf16 P
            const float den = valid ? rpart[r] + rpart[128 + r] + dpart[r] + dpart[128 + r] : 1.f;
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
            if (!FG::all(mbar_wait(&bar->o_done, ph, err, LA_ERR_TIMEOUT))) { ok = false; break; }
            tc_fence_after();
            {
                float dot = 0.f;
#pragma unroll
                for (int cb = 0; cb < 2; ++cb) {
                    uint32_t w[32];
                    tmem_ld32(tmem + lb + kFY + 32 * cb, w);
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
            FG::sync();
            const float g = valid ? -(tpart[r] + tpart[128 + r]) * inv : 0.f;
            if (h == 0) {
                gsh[r] = g;
                if (valid && LA_DCHECK(c0 + r < N))
                    *reinterpret_cast<float2*>(dgh + (size_t)(c0 + r) * 2) = make_float2(den, g);
            }
            tc_fence_before();
            FG::sync();
            if (ct == 0) mbar_arrive(&bar->p_ready);
            {
                // segment sum of g phi(q): weighted column sums of the Q tile
                float zp[2][8];
#pragma unroll
                for (int b = 0; b < 2; ++b)
#pragma unroll
                    for (int e = 0; e < 8; ++e) zp[b][e] = 0.f;
#pragma unroll
                for (int j = 0; j < FG::kJ; ++j) {
                    const uint4 qv = *reinterpret_cast<const uint4*>(sQ + FG::vec_off(ct, j));
                    const uint32_t* u = reinterpret_cast<const uint32_t*>(&qv);
                    const float wr = gsh[FG::vec_row(ct, j)];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        zp[FG::vec_block(j)][2 * e] = fmaf(wr, bf_lo(u[e]), zp[FG::vec_block(j)][2 * e]);
                        zp[FG::vec_block(j)][2 * e + 1] = fmaf(wr, bf_hi(u[e]), zp[FG::vec_block(j)][2 * e + 1]);
                    }
                }
                FG::column_part(zp, drpart, ct);
            }
            FG::sync();  // every read of Q by the compute group is done
            if (ct == 0) mbar_arrive(&bar->empty_qv);
            // (e) D = tril(P V^T + g) as one bf16 copy on this thread's keys, in place (see the X
            // layout); its fp32 row sums (this half) into rpart for the rowsum(D) 1^T part of D K~
            if (!FG::all(mbar_wait(&bar->pv_done, ph, err, LA_ERR_TIMEOUT))) { ok = false; break; }
            tc_fence_after();
            {
                float ds = 0.f;
#pragma unroll
                for (int cb = 0; cb < 2; ++cb) {
                    const int j0 = 64 * h + 32 * cb;
                    uint32_t hi[16];
                    if (j0 > r) {
#pragma unroll
                        for (int x = 0; x < 16; ++x) hi[x] = 0u;
                    } else {
                        uint32_t w[32];
                        tmem_ld32(tmem + lb + kFX + 32 * cb, w);
                        tmem_ld_wait();
                        if (j0 + 31 < (r & ~31)) {  // below the diagonal for the whole warp: no mask
#pragma unroll
                            for (int x = 0; x < 16; ++x) {
                                const float d0 = __uint_as_float(w[2 * x]) + g, d1 = __uint_as_float(w[2 * x + 1]) + g;
                                hi[x] = pack_bf16x2(d0, d1);
                                ds += d0 + d1;
                            }
                        } else {
#pragma unroll
                            for (int x = 0; x < 16; ++x) {
                                const int j = j0 + 2 * x;
                                const float d0 = j <= r ? __uint_as_float(w[2 * x]) + g : 0.f;
                                const float d1 = j + 1 <= r ? __uint_as_float(w[2 * x + 1]) + g : 0.f;
                                hi[x] = pack_bf16x2(d0, d1);
                                ds += d0 + d1;
                            }
                        }
                    }
                    tmem_st16(tmem + lb + kFX + 32 * cb, hi);
                }
                rpart[128 * h + r] = ds;
            }
            tmem_st_wait();
            tc_fence_before();
            FG::sync();
            if (ct == 0) mbar_arrive(&bar->d_ready);
            // (f) dq = (dQ~ + rowsum(D) + g z_prev) * phi'(q), this thread's 64 columns, staged in
            // the Sb tile (free once the dq products are done) and written by one TMA store
            // (rows past N are not written)
            if (!FG::all(mbar_wait(&bar->dq_done, ph, err, LA_ERR_TIMEOUT))) { ok = false; break; }
            tc_fence_after();
            const float dsum = rpart[r] + rpart[128 + r];
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) {
                uint32_t w[32];
                tmem_ld32(tmem + lb + kFY + 32 * cb, w);
                tmem_ld_wait();
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    const uint32_t* qu = &qrow[4 * (4 * cb + c4)];
                    uint4 o4;
                    uint32_t* ou = reinterpret_cast<uint32_t*>(&o4);
                    float zr[8];
                    *reinterpret_cast<float4*>(zr) = *reinterpret_cast<const float4*>(zsh + 64 * h + 32 * cb + 8 * c4);
                    *reinterpret_cast<float4*>(zr + 4) =
                        *reinterpret_cast<const float4*>(zsh + 64 * h + 32 * cb + 8 * c4 + 4);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float a0 = (__uint_as_float(w[8 * c4 + 2 * e]) + fmaf(g, zr[2 * e], dsum)) *
                                         dphi_from_phi(bf_lo(qu[e]));
                        const float a1 = (__uint_as_float(w[8 * c4 + 2 * e + 1]) + fmaf(g, zr[2 * e + 1], dsum)) *
                                         dphi_from_phi(bf_hi(qu[e]));
                        ou[e] = pack_bf16x2(a0, a1);
                    }
                    *reinterpret_cast<uint4*>(sSb + chunk_off(r, 8 * h + 4 * cb + c4)) = o4;
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            FG::sync();  // the dq tile is complete and z_prev has been used by every thread
            if (ct == kStoreThread) {
                check_tile(D > 64 ? 64 : 0, c0, bh, N);
                tma_store_3d(&tm_dq, sSb, 0, c0, bh);
                if (D > 64) tma_store_3d(&tm_dq, sSb + kBlockBytes, 64, c0, bh);
                bulk_commit();
            }
            if (ct < 128) {
                zsh[ct] += FG::column_sum(zpart, ct);
                racc[ct] += FG::column_sum(drpart, ct);
            }
        }
        if (ct == kStoreThread) bulk_wait_all();
        // segment sums of the reverse state out: R from TMEM, r from shared memory
        if (ok && nloc > 0 && FG::all(mbar_wait(&bar->final_mma, 0, err, LA_ERR_TIMEOUT))) {
            tc_fence_after();
            float* out = seg_R + ((size_t)bh * P + p) * E;
            tmem_row_to_global<64>(tmem + lb + kFR, out + (size_t)r * kD + 64 * h);
            if (ct < 128 && record_ok(bh, p, P, (size_t)kD * kD + ct, E)) out[(size_t)kD * kD + ct] = racc[ct];
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
    uint64_t dk_free;  // every compute warp has read this chunk's dK~ from TMEM
    uint64_t ready, rb_ready, masks_ready;
    uint64_t at_dt_done, dk_done, dkv_done;  // dk_done: the dK~ products; dkv_done: the dV products too
    uint64_t final_mma;
};

// Kc: a copy of phi(K) for phi'(k) in the dk epilogue, so that the inputs are
// released (by the MMA thread, at dkv_done) while the epilogue still runs; the
// epilogue then overwrites it with the dk tile, and the Rb tile (free after
// the products) with the dv tile, for the TMA stores.
struct RevSweepSmem {
    static constexpr int Q = 0, K = kTileBytes, V = 2 * kTileBytes, P = 3 * kTileBytes, Rb = 4 * kTileBytes;
    static constexpr int Kc = 5 * kTileBytes;
    static constexpr int rsh = 6 * kTileBytes;  // float[128] r_next
    static constexpr int rpart = rsh + 512;     // float[16][128] per-warp column sums of this chunk's (g den) Q'
    static constexpr int gsh = rpart + 8192;    // float[128] g den of the chunk's rows
    static constexpr int ish = gsh + 512;       // float[128] 1/den of the chunk's rows
    static constexpr int bars = ish + 512;
    static constexpr int tmem_slot = bars + 256;
    static constexpr int total = tmem_slot + 16;
};

template <int D>
__global__ void __launch_bounds__(kThreadsRS, 1)
tc_bwd_reverse_sweep_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                            const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                            const float* __restrict__ seg_R, const float* __restrict__ den_g, int N, int nchunks,
                            int cps, int P, int* err) {
    extern __shared__ uint8_t smem_raw[];
    constexpr int kKd = D / 16;  // K steps of a product over a head dimension (a 64-wide head is zero above)
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = base + RevSweepSmem::Q;
    uint8_t* sK = base + RevSweepSmem::K;
    uint8_t* sV = base + RevSweepSmem::V;
    uint8_t* sP = base + RevSweepSmem::P;
    uint8_t* sRb = base + RevSweepSmem::Rb;
    uint8_t* sKc = base + RevSweepSmem::Kc;
    float* rsh = reinterpret_cast<float*>(base + RevSweepSmem::rsh);
    float* rpart = reinterpret_cast<float*>(base + RevSweepSmem::rpart);
    float* gsh = reinterpret_cast<float*>(base + RevSweepSmem::gsh);  // g den
    float* ish = reinterpret_cast<float*>(base + RevSweepSmem::ish);
    RevSweepBars* bar = reinterpret_cast<RevSweepBars*>(base + RevSweepSmem::bars);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + RevSweepSmem::tmem_slot);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int p = blockIdx.x, bh = blockIdx.y;
    const int cbeg = p * cps, cend = min(nchunks, cbeg + cps), nloc = cend - cbeg;
    const size_t E = state_elems(kD, kD);
    check_plan(p, P, cbeg, cend, nchunks, N);
    record_ok(bh, p, P, E - 1, E);

    if (tid == 0) {
        uint64_t* b = reinterpret_cast<uint64_t*>(bar);
        for (int x = 0; x < (int)(sizeof(RevSweepBars) / 8); ++x) mbar_init(b + x, 1);
        mbar_init(&bar->dk_free, RG::kWarps);  // one arrival per compute warp
        fence_mbar_init();
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_do);
        tma_prefetch_desc(&tm_dk);
        tma_prefetch_desc(&tm_dv);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_enter();  // the previous kernel's outputs (segment records, (den, g)) are visible from here on

    if (warp == 0) {
        if (lane == 0) {
            int armed = -1;
            for (int i = 0; i < nloc; ++i) {
                const int t0 = (cend - 1 - i) * kC;
                if (!mbar_wait(&bar->empty, (i & 1) ^ 1, err, LA_ERR_TIMEOUT)) break;
                mbar_arrive_expect_tx(&bar->full, 4 * kTileBytes);
                check_tile(64, t0, bh, N);
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
            // no copy may still be landing when the CTA exits
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
                // V dO^T needs only the tiles as loaded: it runs while phi is applied, once the
                // previous chunk's dK~ has been read out of the DK region
                if (!mbar_wait(&bar->full, ph, err, LA_ERR_TIMEOUT)) break;
                if (i > 0 && !mbar_wait(&bar->dk_free, (i - 1) & 1, err, LA_ERR_TIMEOUT)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kKd; ++kk)  // DK region = V dO^T (rows = keys)
                    mma_ss(tmem + kRDK, desc_kmajor(aV, kk), desc_kmajor(aP, kk), id_kk, kk > 0);
                if (!mbar_wait(&bar->ready, ph, err, LA_ERR_TIMEOUT)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kKd; ++kk)  // DV region = A'^T = K~ Q'^T (rows = keys)
                    mma_ss(tmem + kRDV, desc_kmajor(aK, kk), desc_kmajor(aQ, kk), id_kk, kk > 0);
                mma_commit(&bar->at_dt_done);
                if (!mbar_wait(&bar->rb_ready, ph, err, LA_ERR_TIMEOUT)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // R_next += Q'^T dO (R_next of this chunk is already in Rb)
                    mma_ss(tmem + kRR, desc_mnmajor(aQ, kk), desc_mnmajor(aP, kk), id_mnmn, 1);
                if (!mbar_wait(&bar->masks_ready, ph, err, LA_ERR_TIMEOUT)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kKd; ++kk)  // dK~ = V R_next^T
                    mma_ss(tmem + kRDK, desc_kmajor(aV, kk), desc_kmajor(aRb, kk), id_kk, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // dK~ += D'^T Q'
                    mma_ts(tmem + kRDK, tmem + kRX + 8 * kk, desc_mnmajor(aQ, kk), id_kmn, 1);
                mma_commit(&bar->dk_done);  // the dk epilogue runs during the dV products
#pragma unroll
                for (int kk = 0; kk < kKd; ++kk)  // dV = K~ R_next
                    mma_ss(tmem + kRDV, desc_kmajor(aK, kk), desc_mnmajor(aRb, kk), id_kmn, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // dV += A'^T dO
                    mma_ts(tmem + kRDV, tmem + kRX + 64 + 8 * kk, desc_mnmajor(aP, kk), id_kmn, 1);
                mma_commit(&bar->dkv_done);
                mma_commit(&bar->empty);  // Q, K, V, P: no further read in this chunk
            }
            mma_commit(&bar->final_mma);
            mbar_wait(&bar->final_mma, 0, err, LA_ERR_TIMEOUT);
        }
    } else {
        const int ct = tid - 64;
        const int qt = (warp - 2) >> 2;  // column quarter: columns [32 qt, 32 qt + 32)
        const int r = 32 * (warp & 3) + lane;
        const uint32_t lane0 = (uint32_t)(32 * (warp & 3)) << 16;
        const uint32_t lb = lane0 + 32 * qt;
        const float* suf = seg_R + ((size_t)bh * P + p) * E;
        global_row_to_tmem<32>(suf + (size_t)r * kD + 32 * qt, tmem + lb + kRR);  // R_next row r, this quarter
        if (ct < 128) rsh[ct] = record_ok(bh, p, P, (size_t)kD * kD + ct, E) ? suf[(size_t)kD * kD + ct] : 0.f;
        tc_fence_before();
        bool ok = RG::all(true);
        const float* dgh = den_g + (size_t)bh * N * 2;
        // (den, g) of row ct of chunk ii (rows past N: den 1, g 0); loaded one chunk ahead
        auto load_dg = [&](int ii) {
            const int cc = (cend - 1 - ii) * kC;
            return ct < min(kC, N - cc) && LA_DCHECK(cc + ct < N && cc >= 0)
                       ? *reinterpret_cast<const float2*>(dgh + (size_t)(cc + ct) * 2)
                       : make_float2(1.f, 0.f);
        };
        float2 dg_next = make_float2(1.f, 0.f);
        if (ct < 128 && nloc > 0) dg_next = load_dg(0);
        for (int i = 0; i < nloc && ok; ++i) {
            const uint32_t ph = i & 1;
            const int c0 = (cend - 1 - i) * kC, n = min(kC, N - c0);
            const float2 dg = dg_next;
            if (ct < 128 && i + 1 < nloc) dg_next = load_dg(i + 1);
            // (a) per-row 1/den and g den; Q' = phi(Q) / den with the chunk's sum of (g den) Q';
            // phi on K (and its copy)
            if (ct == kStoreThread) bulk_wait_read_all();  // the previous dk / dv stores have left Kc and Rb
            if (!RG::all(mbar_wait(&bar->full, ph, err, LA_ERR_TIMEOUT))) { ok = false; break; }
            if (ct < 128) {
                const bool v = ct < n;
                ish[ct] = v ? 1.f / dg.x : 0.f;
                gsh[ct] = v ? dg.y * dg.x : 0.f;
            }
            RG::sync();
            RG::phi_tile(sQ, nullptr, ct, n, D, gsh, rpart, nullptr, ish);
            RG::phi_tile(sK, nullptr, ct, n, D, nullptr, nullptr, sKc);
            fence_proxy_async_smem();
            RG::sync();
            if (ct == 0) mbar_arrive(&bar->ready);
            // (b) R_next -> bf16 copy (rows = dk; this thread's 32 columns).  R is settled:
            // the previous chunk's dkv_done follows its R update.
            tc_fence_after();
            {
                uint32_t w[32];
                tmem_ld32(tmem + lb + kRR, w);
                tmem_ld_wait();
                row32_to_tile(w, sRb, r, 4 * qt);
            }
            tc_fence_before();
            fence_proxy_async_smem();
            RG::sync();
            if (ct == 0) mbar_arrive(&bar->rb_ready);
            // (c) masks: row r is key j = r; columns [32 qt, 32 qt + 32) are queries; keep j <= i
            if (!RG::all(mbar_wait(&bar->at_dt_done, ph, err, LA_ERR_TIMEOUT))) { ok = false; break; }
            tc_fence_after();
            {
                const int q0 = 32 * qt;  // first query of this block
                uint32_t pa[16], pd[16];
                if (q0 + 31 < r) {  // every query here is before key r: all masked
#pragma unroll
                    for (int x = 0; x < 16; ++x) pa[x] = pd[x] = 0u;
                } else if ((r | 31) <= q0) {  // every query here is at or after every key of the warp
                    uint32_t wa[32], wd[32];
                    tmem_ld32(tmem + lb + kRDV, wa);
                    tmem_ld32(tmem + lb + kRDK, wd);
                    tmem_ld_wait();
#pragma unroll
                    for (int x = 0; x < 16; ++x) {
                        const int qi = q0 + 2 * x;
                        pa[x] = pack_bf16x2(__uint_as_float(wa[2 * x]), __uint_as_float(wa[2 * x + 1]));
                        pd[x] = pack_bf16x2(__uint_as_float(wd[2 * x]) + gsh[qi], __uint_as_float(wd[2 * x + 1]) + gsh[qi + 1]);
                    }
                } else {
                    uint32_t wa[32], wd[32];
                    tmem_ld32(tmem + lb + kRDV, wa);
                    tmem_ld32(tmem + lb + kRDK, wd);
                    tmem_ld_wait();
#pragma unroll
                    for (int x = 0; x < 16; ++x) {
                        const int qi = q0 + 2 * x;
                        pa[x] = pack_bf16x2(r <= qi ? __uint_as_float(wa[2 * x]) : 0.f,
                                            r <= qi + 1 ? __uint_as_float(wa[2 * x + 1]) : 0.f);
                        pd[x] = pack_bf16x2(r <= qi ? __uint_as_float(wd[2 * x]) + gsh[qi] : 0.f,
                                            r <= qi + 1 ? __uint_as_float(wd[2 * x + 1]) + gsh[qi + 1] : 0.f);
                    }
                }
                tmem_st16(lane0 + tmem + kRX + 64 + 16 * qt, pa);
                tmem_st16(lane0 + tmem + kRX + 16 * qt, pd);
                tmem_st_wait();
            }
            tc_fence_before();
            RG::sync();
            if (ct == 0) mbar_arrive(&bar->masks_ready);
            // (d) dk = (dK~ + r_next) * phi'(k) in place of phi(k) in Kc once the dK~ products
            // are done, then dv into Rb (free once the dV products are done); this thread's 32
            // columns of key row r; one TMA store each (rows past N are not written)
            if (!RG::all(mbar_wait(&bar->dk_done, ph, err, LA_ERR_TIMEOUT))) { ok = false; break; }
            tc_fence_after();
            {
                uint32_t w[32];
                tmem_ld32(tmem + lb + kRDK, w);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar->dk_free);  // the next chunk's V dO^T may overwrite DK
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    uint4* kp = reinterpret_cast<uint4*>(sKc + chunk_off(r, 4 * qt + c4));
                    const uint4 kv = *kp;
                    const uint32_t* ku = reinterpret_cast<const uint32_t*>(&kv);
                    uint4 o4;
                    uint32_t* ou = reinterpret_cast<uint32_t*>(&o4);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int d = 32 * qt + 8 * c4 + 2 * e;
                        ou[e] = pack_bf16x2((__uint_as_float(w[8 * c4 + 2 * e]) + rsh[d]) * dphi_from_phi(bf_lo(ku[e])),
                                            (__uint_as_float(w[8 * c4 + 2 * e + 1]) + rsh[d + 1]) *
                                                dphi_from_phi(bf_hi(ku[e])));
                    }
                    *kp = o4;
                }
            }
            if (!RG::all(mbar_wait(&bar->dkv_done, ph, err, LA_ERR_TIMEOUT))) { ok = false; break; }
            tc_fence_after();
            {
                uint32_t w[32];
                tmem_ld32(tmem + lb + kRDV, w);
                tmem_ld_wait();
                row32_to_tile(w, sRb, r, 4 * qt);
            }
            // (e) stores out; r_next += this chunk's sum of g phi(q) (every thread has used r_next)
            fence_proxy_async_smem();
            tc_fence_before();
            RG::sync();
            if (ct == kStoreThread) {
                check_tile(D > 64 ? 64 : 0, c0, bh, N);
                tma_store_3d(&tm_dk, sKc, 0, c0, bh);
                tma_store_3d(&tm_dv, sRb, 0, c0, bh);
                if (D > 64) {
                    tma_store_3d(&tm_dk, sKc + kBlockBytes, 64, c0, bh);
                    tma_store_3d(&tm_dv, sRb + kBlockBytes, 64, c0, bh);
                }
                bulk_commit();
            }
            if (ct < 128) rsh[ct] += RG::column_sum(rpart, ct);
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

constexpr size_t kFwdSweepSmem = FwdSweepSmem::total + 1024;
constexpr size_t kRevSweepSmem = RevSweepSmem::total + 1024;

}  // namespace

cudaError_t tc_bwd_forward_sweep(const void* q, const void* k, const void* v, const void* dout, void* dq,
                                 const float* seg_S, float* seg_R, float* den_g, const la_shape& s, const Plan& p,
                                 cudaStream_t st) {
    const int BH = s.B * s.H;
    CUtensorMap tq, tk, tv, td;
    CUtensorMap tdq;
    const int D = s.Dk;  // = s.Dv: 128, or 64 padded to the 128-wide tiles
    if (!make_tmap_bf16_rows(&tq, q, BH, s.N, D, kC) || !make_tmap_bf16_rows(&tk, k, BH, s.N, D, kC) ||
        !make_tmap_bf16_rows(&tv, v, BH, s.N, D, kC) || !make_tmap_bf16_rows(&td, dout, BH, s.N, D, kC) ||
        !make_tmap_bf16_rows(&tdq, dq, BH, s.N, D, kC))
        return cudaErrorInvalidValue;
    auto kern = D == 128 ? tc_bwd_forward_sweep_kernel<128> : tc_bwd_forward_sweep_kernel<64>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kFwdSweepSmem);
    if (e != cudaSuccess) return e;
    launch_begin("tc_bwd_forward_sweep", st);
    e = launch_pdl(kern, dim3(p.P, BH), dim3(kThreadsFS), kFwdSweepSmem, st, tq, tk, tv, td, tdq, seg_S, seg_R, den_g,
                   s.N, p.nchunks, p.cps, p.P, device_error_word());
    cudaError_t e2 = launch_end("tc_bwd_forward_sweep", st);
    return e != cudaSuccess ? e : e2;
}

cudaError_t tc_bwd_reverse_sweep(const void* q, const void* k, const void* v, const void* dout, void* dk, void* dv,
                                 const float* seg_R, const float* den_g, const la_shape& s, const Plan& p,
                                 cudaStream_t st) {
    const int BH = s.B * s.H;
    CUtensorMap tq, tk, tv, td;
    CUtensorMap tdk, tdv;
    const int D = s.Dk;  // = s.Dv: 128, or 64 padded to the 128-wide tiles
    if (!make_tmap_bf16_rows(&tq, q, BH, s.N, D, kC) || !make_tmap_bf16_rows(&tk, k, BH, s.N, D, kC) ||
        !make_tmap_bf16_rows(&tv, v, BH, s.N, D, kC) || !make_tmap_bf16_rows(&td, dout, BH, s.N, D, kC) ||
        !make_tmap_bf16_rows(&tdk, dk, BH, s.N, D, kC) || !make_tmap_bf16_rows(&tdv, dv, BH, s.N, D, kC))
        return cudaErrorInvalidValue;
    auto kern = D == 128 ? tc_bwd_reverse_sweep_kernel<128> : tc_bwd_reverse_sweep_kernel<64>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kRevSweepSmem);
    if (e != cudaSuccess) return e;
    launch_begin("tc_bwd_reverse_sweep", st);
    e = launch_pdl(kern, dim3(p.P, BH), dim3(kThreadsRS), kRevSweepSmem, st, tq, tk, tv, td, tdk, tdv, seg_R, den_g,
                   s.N, p.nchunks, p.cps, p.P, device_error_word());
    cudaError_t e2 = launch_end("tc_bwd_reverse_sweep", st);
    return e != cudaSuccess ? e : e2;
}

}  // namespace la
