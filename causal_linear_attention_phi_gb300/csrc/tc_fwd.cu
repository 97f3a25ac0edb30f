// tc_fwd.cu -- tensor-core (tcgen05 / TMEM / TMA) kernels of the chunked causal
// forward for bf16 inputs with Dk = Dv = 128 and chunks of C = 128 positions.
//
// Per chunk c of a segment ("선형 어텐션" (itwiki), 계산 형태 비교: matrix
// products inside a chunk, the state passed between chunks):
//   QK   = phi(Q_c) phi(K_c)^T                         tcgen05 -> TMEM fp32 (128 x 128)
//   A    = tril(QK) -> bf16, written back to TMEM       compute group
//   O    = phi(Q_c) S_prev + A V_c                      tcgen05 -> TMEM fp32 (128 x 128)
//   den  = phi(Q_c) z_prev + A 1                        tcgen05, N = 16 -> TMEM (column 0)
//   o    = O / den -> bf16 -> global                    compute group
//   S   += phi(K_c)^T V_c,  z += phi(K_c)^T 1           tcgen05 (both accumulate in TMEM)
// The normaliser products use a constant 16 x 128 operand whose row 0 is ones
// (the "append a column of ones" form of phi(Q)(phi(K)^T [V | 1]) in the
// "Transformers은 RNN이다" digest, 핵심 구성요소 2-3).  S_prev and z_prev enter
// as bf16 copies in shared memory, refreshed from the fp32 TMEM state after
// every chunk.  phi is applied in place to the TMA-staged Q and K tiles.
//
// The same kernel with kOut = false only accumulates the segment's sums
// (S, z) for the segment scan.  With kSplit as well, phi(K) enters those sums as a
// hi + lo pair of bf16 operands (S += K_hi^T V + K_lo^T V, and z likewise), the lo
// tiles of the two K stages taking the Q and S_prev tiles that the sums pass leaves
// unused: the non-causal gradient needs S and z to carry phi(K) beyond bf16, since
// its dq is a small difference of terms built from them.
//
// Roles (320 threads): warp 0 issues TMA loads, warp 1 owns TMEM and issues
// tcgen05.mma, warps 2-9 (two warpgroups) transform tiles, mask A, refresh
// S_prev and write outputs.  Warp w reads TMEM lanes 32*(w%4) .. +31 (row r of
// a 128-row tile); warps 2-5 take columns 0-63 of their rows, warps 6-9 the
// columns 64-127.  Every wait is bounded: on timeout the kernel records
// LA_ERR_TIMEOUT in the sticky error word and all roles leave their loops.
#include <cudaTypedefs.h>

#include <mutex>

#include "tc_common.cuh"

namespace la {
namespace {
using namespace sm100;
using namespace tc;

constexpr int kThreads = 320;  // warp 0 TMA, warp 1 MMA, warps 2-9 compute
constexpr int kComputeThreads = 256;
using CG = Grp<kComputeThreads>;
constexpr int kSmallBytes = 4096;  // a 16-row x 128-column bf16 K-major operand (two 2 KB blocks)

// TMEM column map (512 columns allocated)
constexpr uint32_t kTmS = 0, kTmQK = 128, kTmO = 256, kTmA = 384, kTmZ = 448, kTmDen = 464;

struct __align__(8) Barriers {
    uint64_t q_full, q_empty;
    uint64_t kv_full[2], kv_empty[2];
    uint64_t qk_ready[2], sb_ready, a_ready;  // qk_ready per K/V stage: its producer may run one chunk ahead
    uint64_t qk_done, o_done, s_done;
    uint64_t final_mma;
    uint64_t agg_done;  // fused mode: the segment's own sums are complete in TMEM
};

struct SmemLayout {
    // offsets from the 1024-aligned base
    static constexpr int Q = 0;
    static constexpr int K0 = Q + kTileBytes;       // K stages 0, 1
    static constexpr int V0 = K0 + 2 * kTileBytes;  // V stages 0, 1
    static constexpr int Sb = V0 + 2 * kTileBytes;  // bf16 S_prev (rows = dk); once O is done, the o tile for its TMA store
    static constexpr int Ones = Sb + kTileBytes;    // 16 x 128: row 0 ones, rows 1-15 zero
    static constexpr int Zb = Ones + kSmallBytes;   // 16 x 128: row 0 bf16 z_prev, rows 1-15 zero
    static constexpr int bars = Zb + kSmallBytes;
    static constexpr int tmem_slot = bars + 256;
    static constexpr int total = tmem_slot + 16;
};
constexpr size_t kSmemBytes = SmemLayout::total + 1024;  // + alignment slack

// K-major 16-row operand, K step kk: block kk / 4 (2 KB apart), +32 B inside the row.
__device__ __forceinline__ uint64_t desc_small(uint32_t base, int kk) {
    return smem_desc_sw128(base + (kk >> 2) * 2048 + (kk & 3) * 32, 16, 1024);
}
// Byte offset of element (0, col) of a 16-row K-major operand (row 0: chunks unswizzled).
__device__ __forceinline__ int small_row0_off(int col) {
    return (col >> 6) * 2048 + (((col & 63) >> 3) << 4) + ((col & 7) << 1);
}

// The fused causal forward's extra arguments: the chained scan over segments.
struct FusedArgs {
    float* agg;         // [BH][P][E]: each segment's own (S, z) sums, published for later segments
    unsigned* flags;    // [BH][P] publication flags, then the ticket counter; zero at launch
    float* S_out;       // optional [BH][Dk][Dv]: the state after position N (with z_out)
    float* z_out;       // optional [BH][Dk]
    int BH;
    int withhold;       // test only: segment 0 of head 0 never publishes when this is 1
};

// D: the head size, 128 or 64 (padded to the 128-wide tiles); a template
// parameter so that the full-width kernel carries no column test.
//
// kFused (with kOut): one launch for the whole causal forward.  CTAs take their
// (segment, head) from a ticket counter in segment-major order, so a CTA only
// ever waits on CTAs that started before it.  A CTA first forms its segment's
// own sums (S, z) exactly as the sums pass does (same products, same order) and
// publishes them (record in `agg`, flag 1).  It then looks back over the earlier
// segments of its head to the nearest one whose inclusive prefix is published
// (flag 2) and adds, left to right, that prefix and the own sums after it: the
// additions of a sequential exclusive scan, in its order, so the prefixes are
// bit-identical to the separate scan's.  It publishes its own inclusive prefix
// (prefix + own sums) as the next segment's record in `seg` (flag 2), which is
// also what the backward reads, loads its prefix as the starting state and runs
// the output pass.  The last segment skips its own sums unless the state after
// position N is asked for (prefix + own sums, again the scan's order).  Every
// wait is bounded.
template <bool kOut, int D, bool kSplit = false, bool kFused = false>
__global__ void __launch_bounds__(kThreads, 1)
tc_causal_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                     float* __restrict__ seg, int N, int nchunks, int cps, int P, int* err, FusedArgs fa) {
    extern __shared__ uint8_t smem_raw[];
    constexpr int kKd = D / 16;  // K steps of a product over a head dimension (a 64-wide head is zero above)
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = base + SmemLayout::Q;
    uint8_t* sSb = base + SmemLayout::Sb;
    uint8_t* sOnes = base + SmemLayout::Ones;
    uint8_t* sZb = base + SmemLayout::Zb;
    Barriers* bar = reinterpret_cast<Barriers*>(base + SmemLayout::bars);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + SmemLayout::tmem_slot);
    static_assert(!kFused || kOut, "the fused forward is an output pass");

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int p = blockIdx.x, bh = blockIdx.y;
    if (kFused) {  // (segment, head) from the ticket counter, segment-major
        if (tid == 0) tmem_slot[1] = atomicAdd(fa.flags + (size_t)fa.BH * P, 1u);
        __syncthreads();
        const int t = (int)tmem_slot[1];
        LA_DCHECK(t >= 0 && t < fa.BH * P && (int)gridDim.x == fa.BH * P);
        p = t / fa.BH;
        bh = t - p * fa.BH;
    }
    const int cbeg = p * cps, cend = min(nchunks, cbeg + cps), nloc = cend - cbeg;
    const size_t E = state_elems(kD, kD);
    float* segp = seg + ((size_t)bh * P + p) * E;
    if (kFused) {
        LA_DCHECK(bh >= 0 && bh < fa.BH && p >= 0 && p < P && cbeg < cend && cend <= nchunks &&
                  (long long)(cend - 1) * kC < N);
    } else {
        check_plan(p, P, cbeg, cend, nchunks, N);
        record_ok(bh, p, P, E - 1, E);
    }
    const int nBH = kFused ? fa.BH : (int)gridDim.y;  // heads, for the tile checks
    // fused: iterations [0, pre) form the segment's own sums, [pre, pre + nloc) the outputs
    const int npre = kFused && (p < P - 1 || fa.S_out) ? nloc : 0;
    (void)nBH;
    // K and V stage s live at K0 + s * kTileBytes and V0 + s * kTileBytes
    auto sK = [&](int s) { return base + SmemLayout::K0 + s * kTileBytes; };
    auto sV = [&](int s) { return base + SmemLayout::V0 + s * kTileBytes; };
    // the lo part of phi(K) of stage s (kSplit only: the sums pass has no Q and no S_prev)
    auto sKlo = [&](int s) { return s == 0 ? sQ : sSb; };
    static_assert(!(kOut && kSplit), "the split sums are a sums-pass variant");

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
        // constant operand: row 0 ones, rows 1-15 zero (row 0 is unswizzled); Zb rows 1-15 zero
        const int ct = tid - 64;
        for (int x = ct; x < kSmallBytes / 16; x += kComputeThreads) {
            const int row = (x >> 3) & 15;  // 8 chunks of 16 B per 128-B row, 16 rows per 2 KB block
            const uint32_t one2 = 0x3F803F80u;
            const uint4 v = row == 0 ? make_uint4(one2, one2, one2, one2) : make_uint4(0u, 0u, 0u, 0u);
            reinterpret_cast<uint4*>(sOnes)[x] = v;
            reinterpret_cast<uint4*>(sZb)[x] = make_uint4(0u, 0u, 0u, 0u);
        }
        if (kSplit)  // lo tiles zeroed once: a 64-wide head never writes their upper column block
            for (int x = ct; x < kTileBytes / 16; x += kComputeThreads) {
                reinterpret_cast<uint4*>(sQ)[x] = make_uint4(0u, 0u, 0u, 0u);
                reinterpret_cast<uint4*>(sSb)[x] = make_uint4(0u, 0u, 0u, 0u);
            }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_enter();  // the previous kernel's outputs (segment records) are visible from here on

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int armed_kv[2] = {-1, -1}, armed_q = -1;
            bool ok = true;
            // it: K/V stage iterations (own sums, then outputs, in the fused mode); i: output chunk
            for (int it = 0; it < npre + nloc && ok; ++it) {
                const int i = it - npre;
                const int s = it & 1, t0 = (cbeg + (i < 0 ? it : i)) * kC;
                ok = mbar_wait(&bar->kv_empty[s], ((it >> 1) & 1) ^ 1, err, LA_ERR_TIMEOUT);
                if (!ok) break;
                mbar_arrive_expect_tx(&bar->kv_full[s], 2 * kTileBytes);
                check_tile(64, t0, bh, N, nBH);
                tma_load_3d(sK(s), &tm_k, 0, t0, bh, &bar->kv_full[s]);
                tma_load_3d(sK(s) + kBlockBytes, &tm_k, 64, t0, bh, &bar->kv_full[s]);
                tma_load_3d(sV(s), &tm_v, 0, t0, bh, &bar->kv_full[s]);
                tma_load_3d(sV(s) + kBlockBytes, &tm_v, 64, t0, bh, &bar->kv_full[s]);
                armed_kv[s] = it;
                if (kOut && i >= 0) {
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
            constexpr uint32_t id_kk = idesc_bf16_f32(128, 128, 0, 0);
            constexpr uint32_t id_kmn = idesc_bf16_f32(128, 128, 0, 1);
            constexpr uint32_t id_mnmn = idesc_bf16_f32(128, 128, 1, 1);
            constexpr uint32_t id_k16 = idesc_bf16_f32(128, 16, 0, 0);   // N = 16, both K-major
            constexpr uint32_t id_mn16 = idesc_bf16_f32(128, 16, 1, 0);  // N = 16, A MN-major
            const uint32_t aQ = smem_u32(sQ), aSb = smem_u32(sSb), aOnes = smem_u32(sOnes), aZb = smem_u32(sZb);
            bool ok = true;
            for (int it = 0; it < npre + nloc && ok; ++it) {
                const int i = it - npre, s = it & 1;
                const uint32_t aK = smem_u32(sK(s)), aV = smem_u32(sV(s));
                if (!(ok = mbar_wait(&bar->qk_ready[s], (it >> 1) & 1, err, LA_ERR_TIMEOUT))) break;
                tc_fence_after();
                if (kFused && i < 0) {
                    // the segment's own sums: the products and order of the sums pass
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t acc = (it > 0 || kk > 0) ? 1u : 0u;
                        mma_ss(tmem + kTmS, desc_mnmajor(aK, kk), desc_mnmajor(aV, kk), id_mnmn, acc);
                        mma_ss(tmem + kTmZ, desc_mnmajor(aK, kk), desc_small(aOnes, kk), id_mn16, acc);
                    }
                    mma_commit(&bar->kv_empty[s]);
                    if (it == npre - 1) mma_commit(&bar->agg_done);
                    continue;
                }
                if (kOut) {
#pragma unroll
                    for (int kk = 0; kk < kKd; ++kk)  // QK = Q~ K~^T
                        mma_ss(tmem + kTmQK, desc_kmajor(aQ, kk), desc_kmajor(aK, kk), id_kk, kk > 0);
                    mma_commit(&bar->qk_done);
                    if (!(ok = mbar_wait(&bar->sb_ready, i & 1, err, LA_ERR_TIMEOUT))) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kKd; ++kk) {  // O = Q~ S_prev, den = Q~ z_prev
                        mma_ss(tmem + kTmO, desc_kmajor(aQ, kk), desc_mnmajor(aSb, kk), id_kmn, kk > 0);
                        mma_ss(tmem + kTmDen, desc_kmajor(aQ, kk), desc_small(aZb, kk), id_k16, kk > 0);
                    }
                    mma_commit(&bar->q_empty);
                    if (!(ok = mbar_wait(&bar->a_ready, i & 1, err, LA_ERR_TIMEOUT))) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {  // O += A V, den += A 1
                        mma_ts(tmem + kTmO, tmem + kTmA + 8 * kk, desc_mnmajor(aV, kk), id_kmn, 1);
                        mma_ts(tmem + kTmDen, tmem + kTmA + 8 * kk, desc_small(aOnes, kk), id_k16, 1);
                    }
                    mma_commit(&bar->o_done);
                }
                // S += K~^T V, z += K~^T 1  (K tile read as an MN-major A operand)
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t acc = (kOut || i > 0 || kk > 0) ? 1u : 0u;
                    mma_ss(tmem + kTmS, desc_mnmajor(aK, kk), desc_mnmajor(aV, kk), id_mnmn, acc);
                    mma_ss(tmem + kTmZ, desc_mnmajor(aK, kk), desc_small(aOnes, kk), id_mn16, acc);
                }
                if (kSplit) {
                    const uint32_t aKlo = smem_u32(sKlo(s));
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        mma_ss(tmem + kTmS, desc_mnmajor(aKlo, kk), desc_mnmajor(aV, kk), id_mnmn, 1);
                        mma_ss(tmem + kTmZ, desc_mnmajor(aKlo, kk), desc_small(aOnes, kk), id_mn16, 1);
                    }
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
        const int ct = tid - 64;                       // 0..255
        const int h = (warp - 2) >> 2;                 // column half of the rows this thread serves
        const int r = 32 * (warp & 3) + lane;          // TMEM lane / tile row
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        if (kOut && !kFused) {
            // initial state from the scanned segment prefix: S row r (this thread's 64 columns), z[r]
            const float* pre = segp + (size_t)r * kD + 64 * h;
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) {
                uint32_t w[32];
#pragma unroll
                for (int x = 0; x < 32; x += 4) {
                    const float4 f = *reinterpret_cast<const float4*>(pre + 32 * cb + x);
                    w[x] = __float_as_uint(f.x);
                    w[x + 1] = __float_as_uint(f.y);
                    w[x + 2] = __float_as_uint(f.z);
                    w[x + 3] = __float_as_uint(f.w);
                }
                tmem_st32(tmem + lane_base + kTmS + 64 * h + 32 * cb, w);
            }
            if (h == 0) {
                uint32_t zw[16];
                const uint32_t zv = record_ok(bh, p, P, (size_t)kD * kD + r, E) ? __float_as_uint(segp[(size_t)kD * kD + r]) : 0u;
#pragma unroll
                for (int x = 0; x < 16; ++x) zw[x] = zv;
                tmem_st16(tmem + lane_base + kTmZ, zw);
            }
            tmem_st_wait();
        }
        tc_fence_before();
        bool ok = CG::all(true);
        if (kFused) {
            // (own sums) phi on this segment's K tiles for the sums products
            for (int it = 0; it < npre && ok; ++it) {
                const int s = it & 1;
                const int c0 = (cbeg + it) * kC, n = min(kC, N - c0);
                if (!CG::all(mbar_wait(&bar->kv_full[s], (it >> 1) & 1, err, LA_ERR_TIMEOUT))) { ok = false; break; }
                CG::phi_tile(sK(s), nullptr, ct, n, D, nullptr, nullptr);
                fence_proxy_async_smem();
                CG::sync();
                if (ct == 0) mbar_arrive(&bar->qk_ready[s]);
            }
            // publish them (segments with a successor): S row r (this thread's 64 columns) and z[r]
            // to this segment's record, then its flag = 1 (release, after every thread's stores and
            // fences).  The withheld segment (self-test) never publishes anything.
            const bool withheld = fa.withhold && p == 0 && bh == 0;
            unsigned* fl = fa.flags + (size_t)bh * P;
            if (ok && npre > 0) {
                ok = CG::all(mbar_wait(&bar->agg_done, 0, err, LA_ERR_TIMEOUT));
                tc_fence_after();
                if (ok && p < P - 1) {
                    float* own = fa.agg + ((size_t)bh * P + p) * E;
                    tmem_row_to_global<64>(tmem + lane_base + kTmS + 64 * h, own + (size_t)r * kD + 64 * h);
                    if (h == 0) {
                        uint32_t zv[16];
                        tmem_ld16(tmem + lane_base + kTmZ, zv);
                        tmem_ld_wait();
                        own[(size_t)kD * kD + r] = __uint_as_float(zv[0]);
                    }
                    __threadfence();
                    CG::sync();
                    if (ct == 0 && !withheld) flag_release(fl + p, 1u);
                }
            }
            // exclusive prefix.  Thread 0 walks back from segment p - 1 to the nearest segment b
            // whose inclusive prefix is published (flag 2: it sits in record b + 1 of seg), past
            // segments whose own sums are published (flag 1); every thread then adds, left to
            // right, that inclusive prefix (or zero when there is none, b = -1) and the own sums of
            // segments b + 1 .. p - 1.  Each addition is the one a sequential scan over the
            // segments makes, in its order, so the prefix is bit-identical to it whatever b is.
            float run[64];
            float run_z = 0.f;
#pragma unroll
            for (int x = 0; x < 64; ++x) run[x] = 0.f;
            if (ok && p > 0) {
                bool w = true;
                if (ct == 0) {
                    int b = p - 1;
                    const long long t0 = clock64();
                    for (;;) {  // bounded: gives up after kWaitLimitCycles in all
                        const unsigned f = flag_acquire(fl + b);
                        if (f == 2u) break;
                        if (f == 1u) {
                            if (b == 0) { b = -1; break; }
                            --b;
                            continue;
                        }
                        if (clock64() - t0 > kWaitLimitCycles) {
                            atomicCAS(err, 0, LA_ERR_TIMEOUT);
                            w = false;
                            break;
                        }
                        __nanosleep(128);
                    }
                    tmem_slot[2] = (uint32_t)(b + 1);
                }
                ok = CG::all(w);  // a barrier: thread 0's acquires precede every thread's record loads
                const int b = (int)tmem_slot[2] - 1;
                if (ok && b >= 0) {
                    const float* rec = segp - ((size_t)(p - 1 - b)) * E;  // seg record b + 1 of this head
                    const float4* src = reinterpret_cast<const float4*>(rec + (size_t)r * kD + 64 * h);
#pragma unroll
                    for (int x = 0; x < 16; ++x) {
                        const float4 f = __ldcg(src + x);
                        run[4 * x] = f.x;
                        run[4 * x + 1] = f.y;
                        run[4 * x + 2] = f.z;
                        run[4 * x + 3] = f.w;
                    }
                    if (h == 0) run_z = __ldcg(rec + (size_t)kD * kD + r);
                }
                for (int q2 = b + 1; q2 < p && ok; ++q2) {
                    const float* rec = fa.agg + ((size_t)bh * P + q2) * E;
                    const float4* src = reinterpret_cast<const float4*>(rec + (size_t)r * kD + 64 * h);
#pragma unroll
                    for (int x = 0; x < 16; ++x) {
                        const float4 f = __ldcg(src + x);
                        run[4 * x] += f.x;
                        run[4 * x + 1] += f.y;
                        run[4 * x + 2] += f.z;
                        run[4 * x + 3] += f.w;
                    }
                    if (h == 0) run_z += __ldcg(rec + (size_t)kD * kD + r);
                }
            }
            if (ok) {
                // the first segment's prefix record (zero) for the backward; every other segment's
                // record b + 1 is written by segment b as its inclusive prefix
                if (p == 0) {
                    float4* dst = reinterpret_cast<float4*>(segp + (size_t)r * kD + 64 * h);
#pragma unroll
                    for (int x = 0; x < 16; ++x) dst[x] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (h == 0) segp[(size_t)kD * kD + r] = 0.f;
                }
                // the inclusive prefix (prefix + own sums, still in TMEM; the scan's order): the next
                // segment's prefix record, then flag 2
                if (p < P - 1 && npre > 0) {
                    float4* dst = reinterpret_cast<float4*>(segp + E + (size_t)r * kD + 64 * h);
#pragma unroll
                    for (int cb = 0; cb < 2; ++cb) {
                        uint32_t w32[32];
                        tmem_ld32(tmem + lane_base + kTmS + 64 * h + 32 * cb, w32);
                        tmem_ld_wait();
#pragma unroll
                        for (int x = 0; x < 8; ++x)
                            dst[8 * cb + x] = make_float4(run[32 * cb + 4 * x] + __uint_as_float(w32[4 * x]),
                                                          run[32 * cb + 4 * x + 1] + __uint_as_float(w32[4 * x + 1]),
                                                          run[32 * cb + 4 * x + 2] + __uint_as_float(w32[4 * x + 2]),
                                                          run[32 * cb + 4 * x + 3] + __uint_as_float(w32[4 * x + 3]));
                    }
                    if (h == 0) {
                        uint32_t zv[16];
                        tmem_ld16(tmem + lane_base + kTmZ, zv);
                        tmem_ld_wait();
                        segp[E + (size_t)kD * kD + r] = run_z + __uint_as_float(zv[0]);
                    }
                    __threadfence();
                    CG::sync();
                    if (ct == 0 && !withheld) flag_release(fl + p, 2u);
                }
                // the state after position N: prefix + own sums (still in TMEM), the scan's order
                if (fa.S_out && p == P - 1) {
#pragma unroll
                    for (int cb = 0; cb < 2; ++cb) {
                        uint32_t w32[32];
                        tmem_ld32(tmem + lane_base + kTmS + 64 * h + 32 * cb, w32);
                        tmem_ld_wait();
                        if (r < D && 64 * h < D) {
                            float4* so = reinterpret_cast<float4*>(fa.S_out + ((size_t)bh * D + r) * D + 64 * h + 32 * cb);
#pragma unroll
                            for (int x = 0; x < 8; ++x)
                                so[x] = make_float4(run[32 * cb + 4 * x] + __uint_as_float(w32[4 * x]),
                                                    run[32 * cb + 4 * x + 1] + __uint_as_float(w32[4 * x + 1]),
                                                    run[32 * cb + 4 * x + 2] + __uint_as_float(w32[4 * x + 2]),
                                                    run[32 * cb + 4 * x + 3] + __uint_as_float(w32[4 * x + 3]));
                        }
                    }
                    if (h == 0) {
                        uint32_t zv[16];
                        tmem_ld16(tmem + lane_base + kTmZ, zv);
                        tmem_ld_wait();
                        if (r < D) fa.z_out[(size_t)bh * D + r] = run_z + __uint_as_float(zv[0]);
                    }
                }
                // the prefix as the starting state in TMEM
#pragma unroll
                for (int cb = 0; cb < 2; ++cb) {
                    uint32_t w32[32];
#pragma unroll
                    for (int x = 0; x < 32; ++x) w32[x] = __float_as_uint(run[32 * cb + x]);
                    tmem_st32(tmem + lane_base + kTmS + 64 * h + 32 * cb, w32);
                }
                if (h == 0) {
                    uint32_t zw[16];
#pragma unroll
                    for (int x = 0; x < 16; ++x) zw[x] = __float_as_uint(run_z);
                    tmem_st16(tmem + lane_base + kTmZ, zw);
                }
                tmem_st_wait();
            }
            tc_fence_before();
            ok = CG::all(ok);
        }
        bool k_applied = false;  // phi on this chunk's K was applied while the previous chunk's O was formed
        for (int i = 0; i < nloc && ok; ++i) {
            const int it = npre + i, s = it & 1;  // it: K/V stage iteration (own sums came first)
            const int c0 = (cbeg + i) * kC, n = min(kC, N - c0);
            // (a) phi on the K (unless done already) and Q tiles
            if (kOut && ct == kStoreThread) bulk_wait_read_all();  // the previous o store has left the Sb tile
            bool w = mbar_wait(&bar->kv_full[s], (it >> 1) & 1, err, LA_ERR_TIMEOUT);
            if (kOut) w = w && mbar_wait(&bar->q_full, i & 1, err, LA_ERR_TIMEOUT);
            if (!CG::all(w)) { ok = false; break; }
            // (a stage's lo tile is free here: its last reader, the previous chunk's MMAs on this
            // stage, completed before the stage was reloaded)
            if (!k_applied) CG::phi_tile(sK(s), kSplit ? sKlo(s) : nullptr, ct, n, D, nullptr, nullptr);
            if (kOut) CG::phi_tile(sQ, nullptr, ct, n, D, nullptr, nullptr);
            fence_proxy_async_smem();
            CG::sync();
            if (ct == 0) mbar_arrive(&bar->qk_ready[s]);
            if (!kOut) continue;
            // (b) S_prev, z_prev -> bf16 operands (row r = dk, this thread's 64 dv columns = block h)
            if (i > 0) {
                if (!CG::all(mbar_wait(&bar->s_done, (i - 1) & 1, err, LA_ERR_TIMEOUT))) { ok = false; break; }
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
            if (h == 0) {
                uint32_t zv[16];
                tmem_ld16(tmem + lane_base + kTmZ, zv);
                tmem_ld_wait();
                *reinterpret_cast<__nv_bfloat16*>(sZb + small_row0_off(r)) = __float2bfloat16_rn(__uint_as_float(zv[0]));
            }
            tc_fence_before();
            fence_proxy_async_smem();
            CG::sync();
            if (ct == 0) mbar_arrive(&bar->sb_ready);
            // (c) A = tril(QK^T) on keys [64 h, 64 h + 64) -> bf16 pairs into TMEM columns [32 h, 32 h + 32)
            if (!CG::all(mbar_wait(&bar->qk_done, i & 1, err, LA_ERR_TIMEOUT))) { ok = false; break; }
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
                        for (int x = 0; x < 16; ++x)
                            pk[x] = pack_bf16x2(__uint_as_float(wv[2 * x]), __uint_as_float(wv[2 * x + 1]));
                    } else {
#pragma unroll
                        for (int x = 0; x < 16; ++x)
                            pk[x] = pack_bf16x2(j0 + 2 * x <= r ? __uint_as_float(wv[2 * x]) : 0.f,
                                                j0 + 2 * x + 1 <= r ? __uint_as_float(wv[2 * x + 1]) : 0.f);
                    }
                }
                tmem_st16(tmem + lane_base + kTmA + 32 * h + 16 * cb, pk);
            }
            tmem_st_wait();
            tc_fence_before();
            CG::sync();
            if (ct == 0) mbar_arrive(&bar->a_ready);
            // (c') while O is formed: phi on the next chunk's K (the other K/V stage) if it
            // has landed; that stage's previous chunk finished with it before it was reloaded
            k_applied = false;
            if (i + 1 < nloc && CG::all(mbar_try_wait(&bar->kv_full[s ^ 1], ((it + 1) >> 1) & 1))) {
                CG::phi_tile(sK(s ^ 1), nullptr, ct, min(kC, N - (c0 + kC)), D, nullptr, nullptr);
                fence_proxy_async_smem();
                k_applied = true;
            }
            // (d) o = O / den on this thread's 64 columns, staged in the Sb tile (free once
            // O is complete) and written by one TMA store (rows past N are not written)
            if (!CG::all(mbar_wait(&bar->o_done, i & 1, err, LA_ERR_TIMEOUT))) { ok = false; break; }
            tc_fence_after();
            uint32_t dv[16];
            tmem_ld16(tmem + lane_base + kTmDen, dv);
            tmem_ld_wait();
            const float inv = 1.f / __uint_as_float(dv[0]);
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) {
                uint32_t wv[32];
                tmem_ld32(tmem + lane_base + kTmO + 64 * h + 32 * cb, wv);
                tmem_ld_wait();
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint4 v4;
                    v4.x = pack_bf16x2(__uint_as_float(wv[8 * q4 + 0]) * inv, __uint_as_float(wv[8 * q4 + 1]) * inv);
                    v4.y = pack_bf16x2(__uint_as_float(wv[8 * q4 + 2]) * inv, __uint_as_float(wv[8 * q4 + 3]) * inv);
                    v4.z = pack_bf16x2(__uint_as_float(wv[8 * q4 + 4]) * inv, __uint_as_float(wv[8 * q4 + 5]) * inv);
                    v4.w = pack_bf16x2(__uint_as_float(wv[8 * q4 + 6]) * inv, __uint_as_float(wv[8 * q4 + 7]) * inv);
                    *reinterpret_cast<uint4*>(sSb + chunk_off(r, 8 * h + 4 * cb + q4)) = v4;
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            CG::sync();
            if (ct == kStoreThread) {
                check_tile(D > 64 ? 64 : 0, c0, bh, N, nBH);
                tma_store_3d(&tm_o, sSb, 0, c0, bh);
                if (D > 64) tma_store_3d(&tm_o, sSb + kBlockBytes, 64, c0, bh);
                bulk_commit();
            }
        }
        if (kOut && ct == kStoreThread) bulk_wait_all();
        if (!kOut && ok && nloc > 0) {
            // segment sums out: S row r (this thread's 64 columns) and z[r] from TMEM.  The MMA
            // thread's single-use drain barrier marks the last update done.
            if (CG::all(mbar_wait(&bar->final_mma, 0, err, LA_ERR_TIMEOUT))) {
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
                if (h == 0) {
                    uint32_t zv[16];
                    tmem_ld16(tmem + lane_base + kTmZ, zv);
                    tmem_ld_wait();
                    if (record_ok(bh, p, P, (size_t)kD * kD + r, E)) segp[(size_t)kD * kD + r] = __uint_as_float(zv[0]);
                }
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

// A [BH][N][D] bf16 tensor as a 3-D TMA map with 64 x box_rows x 1 boxes and the
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
                          const Plan& p, bool out_pass, cudaStream_t st, bool split_k) {
    const int BH = s.B * s.H;
    CUtensorMap tq, tk, tv, to;
    const int D = s.Dk;  // = s.Dv: 128, or 64 padded to the 128-wide tiles
    // the sums pass has no q and no o: it is given the k map in their place and never uses them
    if (!make_tmap_bf16_rows(&tk, k, BH, s.N, D, kC) || !make_tmap_bf16_rows(&tv, v, BH, s.N, D, kC) ||
        !make_tmap_bf16_rows(&tq, q ? q : k, BH, s.N, D, kC) || !make_tmap_bf16_rows(&to, o ? o : k, BH, s.N, D, kC))
        return cudaErrorInvalidValue;
    int* err = device_error_word();
    dim3 grid(p.P, BH);
    if (out_pass && split_k) return cudaErrorInvalidValue;
    auto kern = out_pass  ? (D == 128 ? tc_causal_fwd_kernel<true, 128> : tc_causal_fwd_kernel<true, 64>)
                : split_k ? (D == 128 ? tc_causal_fwd_kernel<false, 128, true> : tc_causal_fwd_kernel<false, 64, true>)
                          : (D == 128 ? tc_causal_fwd_kernel<false, 128> : tc_causal_fwd_kernel<false, 64>);
    cudaError_t e = cudaFuncSetAttribute((const void*)kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    const char* name = out_pass ? "tc_causal_fwd_out" : split_k ? "tc_segment_sums_split" : "tc_segment_sums";
    launch_begin(name, st);
    e = launch_pdl(kern, grid, dim3(kThreads), kSmemBytes, st, tq, tk, tv, to, seg, s.N, p.nchunks, p.cps, p.P, err,
                   FusedArgs{});
    cudaError_t e2 = launch_end(name, st);
    return e != cudaSuccess ? e : e2;
}

cudaError_t tc_causal_fwd_fused(const void* q, const void* k, const void* v, void* o, float* seg, float* agg,
                                unsigned* flags, float* S_out, float* z_out, const la_shape& s, const Plan& p,
                                cudaStream_t st, bool withhold_first) {
    const int BH = s.B * s.H;
    CUtensorMap tq, tk, tv, to;
    const int D = s.Dk;  // = s.Dv: 128, or 64 padded to the 128-wide tiles
    if (!make_tmap_bf16_rows(&tk, k, BH, s.N, D, kC) || !make_tmap_bf16_rows(&tv, v, BH, s.N, D, kC) ||
        !make_tmap_bf16_rows(&tq, q, BH, s.N, D, kC) || !make_tmap_bf16_rows(&to, o, BH, s.N, D, kC))
        return cudaErrorInvalidValue;
    if ((long long)BH * p.P > 0x7FFFFFFFll) return cudaErrorInvalidValue;
    auto kern = D == 128 ? tc_causal_fwd_kernel<true, 128, false, true> : tc_causal_fwd_kernel<true, 64, false, true>;
    cudaError_t e = cudaFuncSetAttribute((const void*)kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    // the publication flags and the ticket counter start at zero
    e = cudaMemsetAsync(flags, 0, ((size_t)BH * p.P + 1) * sizeof(unsigned), st);
    if (e != cudaSuccess) return e;
    const FusedArgs fa{agg, flags, S_out, z_out, BH, withhold_first ? 1 : 0};
    launch_begin("tc_causal_fwd_fused", st);
    kern<<<dim3((unsigned)(BH * p.P)), kThreads, kSmemBytes, st>>>(tq, tk, tv, to, seg, s.N, p.nchunks, p.cps, p.P,
                                                                   device_error_word(), fa);
    return launch_end("tc_causal_fwd_fused", st);
}

}  // namespace la
