// tc_apply.cu -- tensor-core (tcgen05 / TMEM / TMA) kernel of the non-causal apply,
// o_i = phi(q_i)^T S / phi(q_i)^T z with the head's totals S = phi(K)^T V and
// z = phi(K)^T 1 ("Transformers은 RNN이다" digest, 핵심 구성요소 2; velog review 3.2;
// itwiki 결합 법칙으로 순서 바꾸기), for bf16 heads of 128 (or 64, padded on chip).
//
// Each CTA owns `cps` chunks of 128 positions of one head.  The totals are copied
// once into shared memory as bf16 operands (S as a 128 x 128 tile, rows = dk; z as
// row 0 of a 16-row operand), then per chunk:
//   phi(Q_c) in place on the TMA-staged tile                compute group
//   O = phi(Q_c) S,  den = phi(Q_c) z                       tcgen05 -> TMEM (two buffers)
//   o = O / den -> bf16 -> shared memory -> TMA store      compute group
// Q is double-buffered and so are O and den in TMEM, so the epilogue of one chunk
// runs while the products of the next are formed.  Roles (320 threads): warp 0
// TMA loads, warp 1 TMEM owner and MMA issuer, warps 2-9 the compute group (warp w
// reads TMEM lanes 32 (w % 4) .. +31, i.e. row r of the chunk, and the column half
// (w - 2) / 4).  Every wait is bounded.
#include <cudaTypedefs.h>

#include "tc_common.cuh"

namespace la {
namespace {
using namespace sm100;
using namespace tc;

constexpr int kThreads = 320;  // warp 0 TMA, warp 1 MMA, warps 2-9 compute
constexpr int kComputeThreads = 256;
using CG = Grp<kComputeThreads>;
constexpr int kSmallBytes = 4096;  // a 16-row x 128-column bf16 K-major operand (two 2 KB blocks)

// TMEM columns (512 allocated): O and den of buffer b at 256 b and 256 b + 128
__device__ __forceinline__ uint32_t tm_o(int b) { return 256u * b; }
__device__ __forceinline__ uint32_t tm_den(int b) { return 256u * b + 128u; }

struct __align__(8) Bars {
    uint64_t q_full[2], q_empty[2], q_ready[2];
    uint64_t o_done[2], o_free[2];
    uint64_t final_mma;
};

struct SmemLayout {
    // offsets from the 1024-aligned base
    static constexpr int Sb = 0;                       // bf16 S (rows = dk)
    static constexpr int Zb = Sb + kTileBytes;         // 16 x 128: row 0 bf16 z, rows 1-15 zero
    static constexpr int Q0 = Zb + kSmallBytes;        // Q stages 0, 1
    static constexpr int O0 = Q0 + 2 * kTileBytes;     // o staging 0, 1 for the TMA stores
    static constexpr int bars = O0 + 2 * kTileBytes;
    static constexpr int tmem_slot = bars + 256;
    static constexpr int total = tmem_slot + 16;
};
constexpr size_t kSmemBytes = SmemLayout::total + 1024;  // + alignment slack

// K-major 16-row operand, K step kk: block kk / 4 (2 KB apart), +32 B inside the row.
__device__ __forceinline__ uint64_t small_desc(uint32_t base, int kk) {
    return smem_desc_sw128(base + (kk >> 2) * 2048 + (kk & 3) * 32, 16, 1024);
}
// Byte offset of element (0, col) of a 16-row K-major operand (row 0: chunks unswizzled).
__device__ __forceinline__ int small_row0(int col) {
    return (col >> 6) * 2048 + (((col & 63) >> 3) << 4) + ((col & 7) << 1);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
tc_noncausal_apply_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_out,
                          const float* __restrict__ totals, int N, int nchunks, int cps, int* err) {
    extern __shared__ uint8_t smem_raw[];
    pdl_enter();  // launched with programmatic dependent launch
    constexpr int kKd = D / 16;  // K steps over dk (a 64-wide head is zero above)
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sSb = base + SmemLayout::Sb;
    uint8_t* sZb = base + SmemLayout::Zb;
    Bars* bar = reinterpret_cast<Bars*>(base + SmemLayout::bars);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + SmemLayout::tmem_slot);
    auto sQ = [&](int s) { return base + SmemLayout::Q0 + s * kTileBytes; };
    auto sO = [&](int s) { return base + SmemLayout::O0 + s * kTileBytes; };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int p = blockIdx.x, bh = blockIdx.y;
    const int cbeg = p * cps, cend = min(nchunks, cbeg + cps), nloc = cend - cbeg;
    check_plan(p, (int)gridDim.x, cbeg, cend, nchunks, N);
    const float* tot = totals + (size_t)bh * (D * D + D);  // unpadded record: S [D][D], then z [D]

    if (tid == 0) {
        uint64_t* b = reinterpret_cast<uint64_t*>(bar);
        for (int x = 0; x < (int)(sizeof(Bars) / 8); ++x) mbar_init(b + x, 1);
        fence_mbar_init();
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_out);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    if (warp >= 2) {
        // the totals as bf16 operands: S row r (this thread's 64 columns), zero outside D x D;
        // the z operand zeroed, then its row 0 written after a group barrier
        const int ct = tid - 64, h = (warp - 2) >> 2, r = 32 * (warp & 3) + lane;
#pragma unroll
        for (int cb = 0; cb < 2; ++cb) {
            uint32_t w[32];
            const int c0 = 64 * h + 32 * cb;  // a 32-column block lies wholly inside or outside D
            if (r < D && c0 < D) {
                // 16-byte loads: the workspace is 16-byte aligned, and so is every record and row
                const float4* src = reinterpret_cast<const float4*>(tot + (size_t)r * D + c0);
#pragma unroll
                for (int x4 = 0; x4 < 8; ++x4) {
                    const float4 f = src[x4];
                    w[4 * x4] = __float_as_uint(f.x);
                    w[4 * x4 + 1] = __float_as_uint(f.y);
                    w[4 * x4 + 2] = __float_as_uint(f.z);
                    w[4 * x4 + 3] = __float_as_uint(f.w);
                }
            } else {
#pragma unroll
                for (int x = 0; x < 32; ++x) w[x] = 0u;
            }
            row32_to_tile(w, sSb, r, 8 * h + 4 * cb);
        }
        for (int x = ct; x < kSmallBytes / 16; x += kComputeThreads)
            reinterpret_cast<uint4*>(sZb)[x] = make_uint4(0u, 0u, 0u, 0u);
        CG::sync();
        if (ct < D)
            *reinterpret_cast<__nv_bfloat16*>(sZb + small_row0(ct)) = __float2bfloat16_rn(tot[(size_t)D * D + ct]);
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int armed[2] = {-1, -1};
            for (int i = 0; i < nloc; ++i) {
                const int s = i & 1, t0 = (cbeg + i) * kC;
                if (!mbar_wait(&bar->q_empty[s], ((i >> 1) & 1) ^ 1, err, LA_ERR_TIMEOUT)) break;
                mbar_arrive_expect_tx(&bar->q_full[s], kTileBytes);
                check_tile(0, t0, bh, N), tma_load_3d(sQ(s), &tm_q, 0, t0, bh, &bar->q_full[s]);
                check_tile(64, t0, bh, N), tma_load_3d(sQ(s) + kBlockBytes, &tm_q, 64, t0, bh, &bar->q_full[s]);
                armed[s] = i;
            }
            // never leave with copies in flight
            for (int s = 0; s < 2; ++s)
                if (armed[s] >= 0) mbar_wait(&bar->q_full[s], (armed[s] >> 1) & 1, err, LA_ERR_TIMEOUT);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t id_kmn = idesc_bf16_f32(128, 128, 0, 1);
            constexpr uint32_t id_k16 = idesc_bf16_f32(128, 16, 0, 0);
            const uint32_t aSb = smem_u32(sSb), aZb = smem_u32(sZb);
            for (int i = 0; i < nloc; ++i) {
                const int s = i & 1;
                const uint32_t aQ = smem_u32(sQ(s));
                // buffer s is free once the epilogue of chunk i - 2 has read it
                if (!mbar_wait(&bar->q_ready[s], (i >> 1) & 1, err, LA_ERR_TIMEOUT) ||
                    (i >= 2 && !mbar_wait(&bar->o_free[s], ((i >> 1) & 1) ^ 1, err, LA_ERR_TIMEOUT)))
                    break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kKd; ++kk) {  // O = phi(Q) S, den = phi(Q) z
                    mma_ss(tmem + tm_o(s), desc_kmajor(aQ, kk), desc_mnmajor(aSb, kk), id_kmn, kk > 0);
                    mma_ss(tmem + tm_den(s), desc_kmajor(aQ, kk), small_desc(aZb, kk), id_k16, kk > 0);
                }
                mma_commit(&bar->o_done[s]);
                mma_commit(&bar->q_empty[s]);
            }
            // drain: every MMA this thread issued has completed before TMEM is released
            mma_commit(&bar->final_mma);
            mbar_wait(&bar->final_mma, 0, err, LA_ERR_TIMEOUT);
        }
    } else {
        // ------------------------------------------------------------ compute group (256 threads)
        const int ct = tid - 64;
        const int h = (warp - 2) >> 2;
        const int r = 32 * (warp & 3) + lane;
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        bool ok = CG::all(true);
        // software pipeline: phi on chunk i, then the epilogue of chunk i - 1
        for (int i = 0; i <= nloc && ok; ++i) {
            if (i < nloc) {
                const int s = i & 1;
                const int n = min(kC, N - (cbeg + i) * kC);
                if (!CG::all(mbar_wait(&bar->q_full[s], (i >> 1) & 1, err, LA_ERR_TIMEOUT))) { ok = false; break; }
                CG::phi_tile(sQ(s), nullptr, ct, n, D, nullptr, nullptr);
                fence_proxy_async_smem();
                CG::sync();
                if (ct == 0) mbar_arrive(&bar->q_ready[s]);
            }
            if (i >= 1) {
                const int j = i - 1, sj = j & 1, c0 = (cbeg + j) * kC;
                // the staging tile sj is free once the store of chunk j - 2 has read it
                if (ct == kStoreThread) bulk_wait_read_all();
                if (!CG::all(mbar_wait(&bar->o_done[sj], (j >> 1) & 1, err, LA_ERR_TIMEOUT))) { ok = false; break; }
                tc_fence_after();
                uint32_t dv[16];
                tmem_ld16(tmem + lane_base + tm_den(sj), dv);
                tmem_ld_wait();
                const float inv = 1.f / __uint_as_float(dv[0]);  // rows past N: never stored
#pragma unroll
                for (int cb = 0; cb < 2; ++cb) {
                    uint32_t w[32];
                    tmem_ld32(tmem + lane_base + tm_o(sj) + 64 * h + 32 * cb, w);
                    tmem_ld_wait();
#pragma unroll
                    for (int x = 0; x < 32; ++x) w[x] = __float_as_uint(__uint_as_float(w[x]) * inv);
                    row32_to_tile(w, sO(sj), r, 8 * h + 4 * cb);
                }
                tc_fence_before();
                fence_proxy_async_smem();
                CG::sync();
                if (ct == 0) mbar_arrive(&bar->o_free[sj]);
                if (ct == kStoreThread) {
                    check_tile(0, c0, bh, N), tma_store_3d(&tm_out, sO(sj), 0, c0, bh);
                    if (D > 64) check_tile(64, c0, bh, N), tma_store_3d(&tm_out, sO(sj) + kBlockBytes, 64, c0, bh);
                    bulk_commit();
                }
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

// totals: [BH][Dk*Dv + Dk] unpadded records (S then z) of the head totals.
cudaError_t tc_noncausal_apply(const void* q, void* o, const float* totals, const la_shape& s, const Plan& p,
                               cudaStream_t st) {
    const int BH = s.B * s.H;
    CUtensorMap tq, to;
    const int D = s.Dk;  // = s.Dv: 128, or 64 padded to the 128-wide tiles
    if (!make_tmap_bf16_rows(&tq, q, BH, s.N, D, kC) || !make_tmap_bf16_rows(&to, o, BH, s.N, D, kC))
        return cudaErrorInvalidValue;
    auto kern = D == 128 ? tc_noncausal_apply_kernel<128> : tc_noncausal_apply_kernel<64>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    launch_begin("tc_noncausal_apply", st);
    const cudaError_t le = launch_pdl(kern, dim3(p.P, BH), dim3(kThreads), kSmemBytes, st, tq, to, totals, s.N, p.nchunks, p.cps, device_error_word());
    const cudaError_t le2 = launch_end("tc_noncausal_apply", st);
    return le != cudaSuccess ? le : le2;
}

}  // namespace la
