// tc_retention.cu -- tensor-core (tcgen05 / TMEM / TMA) kernels of retention,
// causal linear attention with a constant decay per head (itwiki 선형 어텐션,
// 발전: 감쇠, 게이트, 델타 규칙: S_t = gamma S_(t-1) + k_t v_t^T, o_t = S_t^T q_t,
// identity feature map, no normaliser), for bf16 heads of Dk = Dv = 128 (or 64,
// zero-padded to the 128-wide tiles) and chunks of C = 128 positions.
//
// Per chunk of n positions (a, b = 0..n-1) with S_in the state entering it:
//   QK  = Q_c K_c^T                                   tcgen05 -> TMEM fp32
//   A   = tril(QK) * gamma^(a-b) -> bf16 in TMEM       compute group
//   O1  = Q_c S_in (S_in as a bf16 copy in smem)       tcgen05 -> TMEM
//   O2  = A V_c                                        tcgen05 -> TMEM (the QK columns, free once A is formed)
//   o_a = gamma^(a+1) O1_a + O2_a -> bf16 -> global    compute group, TMA store
//   S   = gamma^n S_in + K'^T V_c                      the compute group scales S in TMEM while copying
//                                                      S_in out; K' = diag(gamma^(n-1-b)) K_c is formed
//                                                      in place once QK has read K_c; then tcgen05
// No power is divided by: gamma may be 0 (0^0 = 1) or 1.  The powers
// gamma^0 .. gamma^128 are a per-CTA table, formed by square-and-multiply in
// fp64 and rounded once.
//
// The sums pass (kOut = false) forms each segment's local state, started from
// zero, sum_j gamma^(L_end - 1 - j) k_j v_j^T over the segment's positions j
// (L_end its end).  It walks the chunks from the last one back, so the weight
// of a chunk's rows is a running product of table entries: gamma^(n-1-b) times
// gamma^(positions after the chunk).  The decayed scan over segments
// (R_(p+1) = gamma^(L_p) R_p + seg_p) joins the segments.
//
// Roles (320 threads): warp 0 issues TMA loads, warp 1 owns TMEM and issues
// tcgen05.mma, warps 2-9 form A, scale K and S, refresh S_in and write the
// outputs.  Warp w reads TMEM lanes 32*(w%4) .. +31 (row r of a 128-row tile);
// warps 2-5 take columns 0-63 of their rows, warps 6-9 columns 64-127.  Every
// wait is bounded: on timeout the kernel records LA_ERR_TIMEOUT in the sticky
// error word and all roles leave their loops.
#include <cudaTypedefs.h>

#include "tc_common.cuh"

namespace la {
namespace {
using namespace sm100;
using namespace tc;

constexpr int kThreads = 320;  // warp 0 TMA, warp 1 MMA, warps 2-9 compute
constexpr int kComputeThreads = 256;
using CG = Grp<kComputeThreads>;

// TMEM column map (512 columns allocated)
constexpr uint32_t kTmS = 0, kTmQK = 128, kTmO1 = 256, kTmA = 384;

struct __align__(8) Barriers {
    uint64_t q_full, q_empty;
    uint64_t kv_full[2], kv_empty[2];
    uint64_t k_ready;   // sums pass: K' formed
    uint64_t sb_ready;  // S_in copied to Sb and S scaled by gamma^n in TMEM
    uint64_t qk_done, a_ready, o_done, s_done;
    uint64_t o_free;    // the epilogue has read O1 and O2: the QK columns may be overwritten
    uint64_t final_mma;
};

struct SmemLayout {
    // offsets from the 1024-aligned base
    static constexpr int Q = 0;
    static constexpr int K0 = Q + kTileBytes;       // K stages 0, 1
    static constexpr int V0 = K0 + 2 * kTileBytes;  // V stages 0, 1
    static constexpr int Sb = V0 + 2 * kTileBytes;  // bf16 S_in (rows = dk); then the o tile for its TMA store
    static constexpr int pw = Sb + kTileBytes;      // fp32 gamma^0 .. gamma^kC
    static constexpr int bars = pw + 1024;
    static constexpr int tmem_slot = bars + 256;
    static constexpr int total = tmem_slot + 16;
};
constexpr size_t kSmemBytes = SmemLayout::total + 1024;  // + alignment slack
static_assert((kC + 1) * 4 <= 1024, "power table");

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

// Row b of a staged 128 x 128 bf16 tile times base * gamma^(n-1-b) for b < n
// (rows >= n hold TMA zero fill and stay 0), in place.
__device__ __forceinline__ void decay_rows(uint8_t* tile, int ct, int n, const float* pw, float base) {
    uint4 v[CG::kJ];
#pragma unroll
    for (int j = 0; j < CG::kJ; ++j) v[j] = *reinterpret_cast<const uint4*>(tile + CG::vec_off(ct, j));
#pragma unroll
    for (int j = 0; j < CG::kJ; ++j) {
        const int row = CG::vec_row(ct, j);
        const float w = row < n ? base * pw[row < n ? n - 1 - row : 0] : 0.f;
        uint32_t* u = reinterpret_cast<uint32_t*>(&v[j]);
#pragma unroll
        for (int e = 0; e < 4; ++e) u[e] = pack_bf16x2(w * bf_lo(u[e]), w * bf_hi(u[e]));
        *reinterpret_cast<uint4*>(tile + CG::vec_off(ct, j)) = v[j];
    }
}

template <bool kOut, int D>
__global__ void __launch_bounds__(kThreads, 1)
tc_retention_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                    const float* __restrict__ gamma, int H, float* __restrict__ seg, int N, int nchunks, int cps,
                    int P, int* err) {
    extern __shared__ uint8_t smem_raw[];
    pdl_enter();  // launched with programmatic dependent launch
    constexpr int kKd = D / 16;  // K steps of a product over a head dimension (a 64-wide head is zero above)
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = base + SmemLayout::Q;
    uint8_t* sSb = base + SmemLayout::Sb;
    float* pw = reinterpret_cast<float*>(base + SmemLayout::pw);
    Barriers* bar = reinterpret_cast<Barriers*>(base + SmemLayout::bars);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + SmemLayout::tmem_slot);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int p = blockIdx.x, bh = blockIdx.y;
    const int cbeg = p * cps, cend = min(nchunks, cbeg + cps), nloc = cend - cbeg;
    check_plan(p, (int)gridDim.x, cbeg, cend, nchunks, N);
    float* segp = seg + ((size_t)bh * P + p) * (size_t)(kD * kD);
    auto sK = [&](int s) { return base + SmemLayout::K0 + s * kTileBytes; };
    auto sV = [&](int s) { return base + SmemLayout::V0 + s * kTileBytes; };
    // the i-th chunk this CTA handles: in order for the outputs, from the last one back for the sums
    auto chunk_of = [&](int i) { return kOut ? cbeg + i : cend - 1 - i; };

    if (tid == 0) {
        uint64_t* b = reinterpret_cast<uint64_t*>(bar);
        for (int x = 0; x < (int)(sizeof(Barriers) / 8); ++x) mbar_init(b + x, 1);
        fence_mbar_init();
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        if (kOut) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_o);
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    if (warp >= 2) {
        const double g = gamma[bh % H];
        for (int t = tid - 64; t <= kC; t += kComputeThreads) pw[t] = (float)pow_int(g, t);
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
                const int s = i & 1, t0 = chunk_of(i) * kC;
                ok = mbar_wait(&bar->kv_empty[s], ((i >> 1) & 1) ^ 1, err, LA_ERR_TIMEOUT);
                if (!ok) break;
                mbar_arrive_expect_tx(&bar->kv_full[s], 2 * kTileBytes);
                check_tile(0, t0, bh, N), tma_load_3d(sK(s), &tm_k, 0, t0, bh, &bar->kv_full[s]);
                check_tile(64, t0, bh, N), tma_load_3d(sK(s) + kBlockBytes, &tm_k, 64, t0, bh, &bar->kv_full[s]);
                check_tile(0, t0, bh, N), tma_load_3d(sV(s), &tm_v, 0, t0, bh, &bar->kv_full[s]);
                check_tile(64, t0, bh, N), tma_load_3d(sV(s) + kBlockBytes, &tm_v, 64, t0, bh, &bar->kv_full[s]);
                armed_kv[s] = i;
                if (kOut) {
                    ok = mbar_wait(&bar->q_empty, (i & 1) ^ 1, err, LA_ERR_TIMEOUT);
                    if (!ok) break;
                    mbar_arrive_expect_tx(&bar->q_full, kTileBytes);
                    check_tile(0, t0, bh, N), tma_load_3d(sQ, &tm_q, 0, t0, bh, &bar->q_full);
                    check_tile(64, t0, bh, N), tma_load_3d(sQ + kBlockBytes, &tm_q, 64, t0, bh, &bar->q_full);
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
            constexpr uint32_t id_kk = idesc_bf16_f32(128, 128, 0, 0);
            constexpr uint32_t id_kmn = idesc_bf16_f32(128, 128, 0, 1);
            constexpr uint32_t id_mnmn = idesc_bf16_f32(128, 128, 1, 1);
            const uint32_t aQ = smem_u32(sQ), aSb = smem_u32(sSb);
            bool ok = true;
            for (int i = 0; i < nloc && ok; ++i) {
                const int s = i & 1;
                const uint32_t aK = smem_u32(sK(s)), aV = smem_u32(sV(s));
                if (kOut) {
                    ok = mbar_wait(&bar->kv_full[s], (i >> 1) & 1, err, LA_ERR_TIMEOUT) &&
                         mbar_wait(&bar->q_full, i & 1, err, LA_ERR_TIMEOUT) &&
                         (i == 0 || mbar_wait(&bar->o_free, (i - 1) & 1, err, LA_ERR_TIMEOUT));
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kKd; ++kk)  // QK = Q K^T
                        mma_ss(tmem + kTmQK, desc_kmajor(aQ, kk), desc_kmajor(aK, kk), id_kk, kk > 0);
                    mma_commit(&bar->qk_done);
                    if (!(ok = mbar_wait(&bar->sb_ready, i & 1, err, LA_ERR_TIMEOUT))) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kKd; ++kk)  // O1 = Q S_in
                        mma_ss(tmem + kTmO1, desc_kmajor(aQ, kk), desc_mnmajor(aSb, kk), id_kmn, kk > 0);
                    mma_commit(&bar->q_empty);
                    if (!(ok = mbar_wait(&bar->a_ready, i & 1, err, LA_ERR_TIMEOUT))) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)  // O2 = A V, over the consumed QK columns
                        mma_ts(tmem + kTmQK, tmem + kTmA + 8 * kk, desc_mnmajor(aV, kk), id_kmn, kk > 0);
                    mma_commit(&bar->o_done);
                } else {
                    if (!(ok = mbar_wait(&bar->k_ready, i & 1, err, LA_ERR_TIMEOUT))) break;
                    tc_fence_after();
                }
                // S += K'^T V  (K' read as an MN-major A operand; S was scaled by gamma^n first)
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t acc = (kOut || i > 0 || kk > 0) ? 1u : 0u;
                    mma_ss(tmem + kTmS, desc_mnmajor(aK, kk), desc_mnmajor(aV, kk), id_mnmn, acc);
                }
                mma_commit(&bar->s_done);
                mma_commit(&bar->kv_empty[s]);
            }
            // drain: every MMA this thread issued has completed before TMEM is released
            mma_commit(&bar->final_mma);
            mbar_wait(&bar->final_mma, 0, err, LA_ERR_TIMEOUT);
        }
    } else {
        // ------------------------------------------------------------ compute group (256 threads)
        const int ct = tid - 64;                // 0..255
        const int h = (warp - 2) >> 2;          // column half of the rows this thread serves
        const int r = 32 * (warp & 3) + lane;   // TMEM lane / tile row
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        if (kOut) {  // the state entering the segment: S row r, this thread's 64 columns
            global_row_to_tmem<64>(segp + (size_t)r * kD + 64 * h, tmem + lane_base + kTmS + 64 * h);
        }
        tc_fence_before();
        bool ok = CG::all(true);
        float wbase = 1.f;  // sums pass: gamma^(positions of the segment after the current chunk)
        for (int i = 0; i < nloc && ok; ++i) {
            const int s = i & 1;
            const int c0 = chunk_of(i) * kC, n = min(kC, N - c0);
            if (!kOut) {
                // K' = diag(wbase gamma^(n-1-b)) K, then the MMA thread adds K'^T V
                if (!CG::all(mbar_wait(&bar->kv_full[s], (i >> 1) & 1, err, LA_ERR_TIMEOUT))) { ok = false; break; }
                decay_rows(sK(s), ct, n, pw, wbase);
                fence_proxy_async_smem();
                CG::sync();
                if (ct == 0) mbar_arrive(&bar->k_ready);
                wbase *= pw[n];
                continue;
            }
            // (b) S_in -> bf16 Sb; S <- gamma^n S_in in TMEM.  Sb is free once the previous
            // o store has read it and the state update of the previous chunk is complete.
            if (ct == kStoreThread) bulk_wait_read_all();
            if (!CG::all(i == 0 || mbar_wait(&bar->s_done, (i - 1) & 1, err, LA_ERR_TIMEOUT))) { ok = false; break; }
            tc_fence_after();
            const float gn = pw[n];
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) {
                const uint32_t ta = tmem + lane_base + kTmS + 64 * h + 32 * cb;
                uint32_t wv[32];
                tmem_ld32(ta, wv);
                tmem_ld_wait();
                row32_to_tile(wv, sSb, r, 8 * h + 4 * cb);
#pragma unroll
                for (int x = 0; x < 32; ++x) wv[x] = __float_as_uint(gn * __uint_as_float(wv[x]));
                tmem_st32(ta, wv);
            }
            tmem_st_wait();
            tc_fence_before();
            fence_proxy_async_smem();
            CG::sync();
            if (ct == 0) mbar_arrive(&bar->sb_ready);
            // (c) A = tril(QK) * gamma^(a-b) on keys [64 h, 64 h + 64) -> bf16 pairs in TMEM
            // columns [32 h, 32 h + 32); then K' = diag(gamma^(n-1-b)) K in place (QK has read K)
            if (!CG::all(mbar_wait(&bar->qk_done, i & 1, err, LA_ERR_TIMEOUT) &&
                         mbar_wait(&bar->kv_full[s], (i >> 1) & 1, err, LA_ERR_TIMEOUT))) {
                ok = false;
                break;
            }
            tc_fence_after();
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) {
                const int j0 = 64 * h + 32 * cb;  // first key of this 32-column block
                uint32_t pk[16];
                if (j0 > r) {  // entirely above the diagonal
#pragma unroll
                    for (int x = 0; x < 16; ++x) pk[x] = 0u;
                } else {
                    uint32_t wv[32];
                    tmem_ld32(tmem + lane_base + kTmQK + j0, wv);
                    tmem_ld_wait();
                    if (j0 + 31 < (r & ~31)) {  // below the diagonal for every row of the warp
#pragma unroll
                        for (int x = 0; x < 16; ++x) {
                            const int j = j0 + 2 * x;
                            pk[x] = pack_bf16x2(__uint_as_float(wv[2 * x]) * pw[r - j],
                                                __uint_as_float(wv[2 * x + 1]) * pw[r - j - 1]);
                        }
                    } else {
#pragma unroll
                        for (int x = 0; x < 16; ++x) {
                            const int j = j0 + 2 * x;
                            const float a0 = j <= r ? __uint_as_float(wv[2 * x]) * pw[j <= r ? r - j : 0] : 0.f;
                            const float a1 =
                                j + 1 <= r ? __uint_as_float(wv[2 * x + 1]) * pw[j + 1 <= r ? r - j - 1 : 0] : 0.f;
                            pk[x] = pack_bf16x2(a0, a1);
                        }
                    }
                }
                tmem_st16(tmem + lane_base + kTmA + 32 * h + 16 * cb, pk);
            }
            decay_rows(sK(s), ct, n, pw, 1.f);
            tmem_st_wait();
            tc_fence_before();
            fence_proxy_async_smem();
            CG::sync();
            if (ct == 0) mbar_arrive(&bar->a_ready);
            // (d) o = gamma^(a+1) O1 + O2 on this thread's 64 columns, staged in the Sb tile
            // (O1 has read it) and written by one TMA store (rows past N are not written)
            if (!CG::all(mbar_wait(&bar->o_done, i & 1, err, LA_ERR_TIMEOUT))) { ok = false; break; }
            tc_fence_after();
            const float u = pw[r + 1];
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) {
                uint32_t w1[32], w2[32];
                tmem_ld32(tmem + lane_base + kTmO1 + 64 * h + 32 * cb, w1);
                tmem_ld32(tmem + lane_base + kTmQK + 64 * h + 32 * cb, w2);
                tmem_ld_wait();
#pragma unroll
                for (int x = 0; x < 32; ++x)
                    w1[x] = __float_as_uint(fmaf(u, __uint_as_float(w1[x]), __uint_as_float(w2[x])));
                row32_to_tile(w1, sSb, r, 8 * h + 4 * cb);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            CG::sync();
            if (ct == 0) mbar_arrive(&bar->o_free);
            if (ct == kStoreThread) {
                check_tile(0, c0, bh, N), tma_store_3d(&tm_o, sSb, 0, c0, bh);
                if (D > 64) check_tile(64, c0, bh, N), tma_store_3d(&tm_o, sSb + kBlockBytes, 64, c0, bh);
                bulk_commit();
            }
        }
        if (kOut && ct == kStoreThread) bulk_wait_all();
        if (!kOut && ok) {
            // the segment's local state out: S row r, this thread's 64 columns.  The MMA
            // thread's single-use drain barrier marks the last update done.
            if (CG::all(mbar_wait(&bar->final_mma, 0, err, LA_ERR_TIMEOUT))) {
                tc_fence_after();
                tmem_row_to_global<64>(tmem + lane_base + kTmS + 64 * h, segp + (size_t)r * kD + 64 * h);
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

}  // namespace

cudaError_t tc_retention_fwd(const void* q, const void* k, const void* v, const float* gamma, void* o, float* seg,
                             const la_shape& s, const Plan& p, bool out_pass, cudaStream_t st) {
    const int BH = s.B * s.H;
    CUtensorMap tq, tk, tv, to;
    const int D = s.Dk;  // = s.Dv: 128, or 64 padded to the 128-wide tiles
    // the sums pass has no q and no o: it is given the k map in their place and never uses them
    if (!make_tmap_bf16_rows(&tk, k, BH, s.N, D, kC) || !make_tmap_bf16_rows(&tv, v, BH, s.N, D, kC) ||
        !make_tmap_bf16_rows(&tq, q ? q : k, BH, s.N, D, kC) || !make_tmap_bf16_rows(&to, o ? o : k, BH, s.N, D, kC))
        return cudaErrorInvalidValue;
    int* err = device_error_word();
    const dim3 grid(p.P, BH);
    auto kern = out_pass ? (D == 128 ? tc_retention_kernel<true, 128> : tc_retention_kernel<true, 64>)
                         : (D == 128 ? tc_retention_kernel<false, 128> : tc_retention_kernel<false, 64>);
    cudaError_t e =
        cudaFuncSetAttribute((const void*)kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    const char* name = out_pass ? "tc_retention_out" : "tc_retention_sums";
    launch_begin(name, st);
    const cudaError_t le = launch_pdl(kern, grid, dim3(kThreads), kSmemBytes, st, tq, tk, tv, to, gamma, s.H, seg, s.N, p.nchunks, p.cps, p.P, err);
    const cudaError_t le2 = launch_end(name, st);
    return le != cudaSuccess ? le : le2;
}

}  // namespace la
