// tc_common.cuh -- shared pieces of the tcgen05 kernels (bf16, D = 128, C = 128).
//
// Tile layout: a 128-row x 128-column bf16 tile is two 64-column blocks of
// 128 rows x 128 B, each written by TMA with the 128-byte swizzle: inside a
// block, the 16-byte chunk `lc` of row `row` sits at physical chunk
// lc ^ (row & 7).  The same physical tile serves as a K-major operand (rows =
// M or N, contiguous K) and as an MN-major operand (rows = K, contiguous M/N)
// of tcgen05.mma; see smem_desc_sw128.
#pragma once

#include "la_internal.cuh"
#include "sm100.cuh"

namespace la {
namespace tc {
using namespace sm100;

constexpr int kC = 128;             // chunk length
constexpr int kD = 128;             // Dk = Dv of the tiles (a 64-wide head is zero-padded)
constexpr int kTileBytes = 32768;   // one 128 x 128 bf16 tile
constexpr int kBlockBytes = 16384;  // one 64-column block
// The compute thread that issues a kernel's TMA stores and waits for them: one
// that has no per-column work at the end of a chunk (compute threads 0-127 do).
constexpr int kStoreThread = 128;

// K-major operand, K step kk (16 elements): block kk / 4, +32 B inside the 128-B row.
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t tile, int kk) {
    return smem_desc_sw128(tile + (kk >> 2) * kBlockBytes + (kk & 3) * 32, 16, 1024);
}
// MN-major operand, K step kk (16 rows): +2048 B; the two 64-wide M/N blocks are kBlockBytes apart.
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t tile, int kk) {
    return smem_desc_sw128(tile + kk * 2048, kBlockBytes, 1024);
}

// Byte offset of logical 16-byte chunk lc (0..15, 8 columns each) of `row`.
__device__ __forceinline__ int chunk_off(int row, int lc) {
    LA_DCHECK(row >= 0 && row < kC && lc >= 0 && lc < 16);
    return (lc >> 3) * kBlockBytes + row * 128 + (((lc & 7) ^ (row & 7)) << 4);
}

// Debug build: the work split of a chunked kernel launched on a (P, BH) grid: this CTA's
// segment p holds chunks [cbeg, cend) of a head, all starting inside the sequence.
__device__ __forceinline__ void check_plan(int p, int P, int cbeg, int cend, int nchunks, int N) {
    LA_DCHECK(p >= 0 && p < P && (int)gridDim.x == P && blockIdx.y < gridDim.y && cbeg >= 0 && cbeg < cend &&
              cend <= nchunks && (long long)(cend - 1) * kC < N && (long long)nchunks * kC < (long long)N + kC);
}
// Debug build: a TMA tile (x, row) of head bh of a [BH][N][D] map: x a multiple of 8
// elements (16 bytes) inside the 128-wide tile, the first row inside the sequence.  TMA
// clips rows past N by itself; the check catches a wrong coordinate.
__device__ __forceinline__ void check_tile(int x, int row, int bh, int N, int BH = -1) {
    LA_DCHECK(x >= 0 && (x & 7) == 0 && x < kD && row >= 0 && row < N && bh >= 0 &&
              bh < (BH < 0 ? (int)gridDim.y : BH));
}
// Debug build: a state record index (head bh, segment p of P) and an element offset in it.
__device__ __forceinline__ bool record_ok(int bh, int p, int P, size_t off, size_t E) {
    return LA_DCHECK(bh >= 0 && bh < (int)gridDim.y && p >= 0 && p < P && off < E);
}
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
// kCols fp32 values of a row from global memory into TMEM columns (initial states).
template <int kCols = 128>
__device__ __forceinline__ void global_row_to_tmem(const float* src, uint32_t taddr) {
#pragma unroll
    for (int cb = 0; cb < kCols / 32; ++cb) {
        uint32_t w[32];
#pragma unroll
        for (int x = 0; x < 32; x += 4) {
            const float4 f = *reinterpret_cast<const float4*>(src + 32 * cb + x);
            w[x] = __float_as_uint(f.x);
            w[x + 1] = __float_as_uint(f.y);
            w[x + 2] = __float_as_uint(f.z);
            w[x + 3] = __float_as_uint(f.w);
        }
        tmem_st32(taddr + 32 * cb, w);
    }
    tmem_st_wait();
}

// kCols fp32 TMEM columns of a row to global memory.
template <int kCols = 128>
__device__ __forceinline__ void tmem_row_to_global(uint32_t taddr, float* dst) {
#pragma unroll
    for (int cb = 0; cb < kCols / 32; ++cb) {
        uint32_t w[32];
        tmem_ld32(taddr + 32 * cb, w);
        tmem_ld_wait();
#pragma unroll
        for (int x = 0; x < 32; x += 4)
            *reinterpret_cast<float4*>(dst + 32 * cb + x) = make_float4(
                __uint_as_float(w[x]), __uint_as_float(w[x + 1]), __uint_as_float(w[x + 2]), __uint_as_float(w[x + 3]));
    }
}

// 32 fp32 values -> logical 16-byte chunks lc0 .. lc0 + 3 of `row` of a bf16 tile.
__device__ __forceinline__ void row32_to_tile(const uint32_t (&w)[32], uint8_t* tile, int row, int lc0) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint4 v4;
        v4.x = pack_bf16x2(__uint_as_float(w[8 * q + 0]), __uint_as_float(w[8 * q + 1]));
        v4.y = pack_bf16x2(__uint_as_float(w[8 * q + 2]), __uint_as_float(w[8 * q + 3]));
        v4.z = pack_bf16x2(__uint_as_float(w[8 * q + 4]), __uint_as_float(w[8 * q + 5]));
        v4.w = pack_bf16x2(__uint_as_float(w[8 * q + 6]), __uint_as_float(w[8 * q + 7]));
        *reinterpret_cast<uint4*>(tile + chunk_off(row, lc0 + q)) = v4;
    }
}

// 64 fp32 TMEM columns of this thread's row (column half h) -> the same half of a bf16 tile row.
__device__ __forceinline__ void tmem_half_row_to_tile(uint32_t taddr, uint8_t* tile, int row, int h) {
#pragma unroll
    for (int cb = 0; cb < 2; ++cb) {
        uint32_t w[32];
        tmem_ld32(taddr + 32 * cb, w);
        tmem_ld_wait();
        row32_to_tile(w, tile, row, 8 * h + 4 * cb);
    }
}

// ------------------------------------------------------------------ compute group
// The compute warps of a CTA (G threads, G = 256 or 512): thread ct = tid - 64
// (warps 0 and 1 are the TMA and MMA roles).  For whole-tile elementwise work,
// thread ct owns the 16-byte vectors ct + G j (j < 2048 / G): block j / (J / 2),
// row ((ct >> 3) + (G / 8) (j % (J / 2))) & 127, physical chunk ct & 7, logical
// chunk lc = (ct & 7) ^ ((ct >> 3) & 7), i.e. columns 64 block + 8 lc + e.
template <int G>
struct Grp {
    static_assert(G == 256 || G == 512, "compute group of 8 or 16 warps");
    static constexpr int kJ = 2048 / G;  // 16-byte vectors of a 128 x 128 bf16 tile per thread
    static constexpr int kWarps = G / 32;

    // Barrier over the group (named barrier 1) that ANDs a predicate across it,
    // so every thread takes the same branch after a bounded wait.
    __device__ static __forceinline__ bool all(bool v) {
        uint32_t r;
        asm volatile(
            "{\n\t.reg .pred p, q;\n\t"
            "setp.ne.u32 p, %1, 0;\n\t"
            "bar.red.and.pred q, 1, %2, p;\n\t"
            "selp.u32 %0, 1, 0, q;\n\t}"
            : "=r"(r)
            : "r"((uint32_t)v), "n"(G)
            : "memory");
        return r != 0;
    }
    __device__ static __forceinline__ void sync() { named_barrier(1, G); }

    __device__ static __forceinline__ int vec_block(int j) { return j / (kJ / 2); }
    __device__ static __forceinline__ int vec_row(int ct, int j) { return ((ct >> 3) + (G / 8) * (j % (kJ / 2))) & 127; }
    __device__ static __forceinline__ int vec_off(int ct, int j) {
        LA_DCHECK(ct >= 0 && ct < G && j >= 0 && j < kJ);
        return vec_block(j) * kBlockBytes + vec_row(ct, j) * 128 + (ct & 7) * 16;
    }
    __device__ static __forceinline__ int vec_lc(int ct) { return (ct & 7) ^ ((ct >> 3) & 7); }

    // Column partial sums zp[block][e] (for columns 64 block + 8 lc + e of this
    // thread) summed over the four lanes of the warp that share lc (lanes l,
    // l^9, l^18, l^27) and stored by lanes 0-7 as this warp's row of
    // part[kWarps][128] (no atomics: column_sum adds the rows after a barrier).
    __device__ static __forceinline__ void column_part(float (&zp)[2][8], float* part, int ct) {
#pragma unroll
        for (int b = 0; b < 2; ++b)
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                float x = zp[b][e];
                x += __shfl_xor_sync(0xffffffffu, x, 9);
                x += __shfl_xor_sync(0xffffffffu, x, 18);
                zp[b][e] = x;
            }
        if ((ct & 31) < 8) {
            float* row = part + (ct >> 5) * 128 + 8 * vec_lc(ct);
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                *reinterpret_cast<float4*>(row + 64 * b) = make_float4(zp[b][0], zp[b][1], zp[b][2], zp[b][3]);
                *reinterpret_cast<float4*>(row + 64 * b + 4) = make_float4(zp[b][4], zp[b][5], zp[b][6], zp[b][7]);
            }
        }
    }
    // Column c (0..127) of part[kWarps][128] summed over the warps.
    __device__ static __forceinline__ float column_sum(const float* part, int c) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) s += part[128 * w + c];
        return s;
    }

    // phi in place on a staged tile (rows >= n and columns >= dcols exactly 0:
    // a head narrower than the tile is zero-padded), times scale[row] when
    // scale is given.  With colpart, the column sums of the rounded values
    // (weighted by w[row] when w is given) go to colpart as per-warp partials
    // (column_part).  With lo_tile, also writes lo = bf16(phi - hi) there, or,
    // with kMinusOne, bf16(phi - 1) (0 outside the rows and columns in range);
    // with copy_tile, a second copy of the rounded values.
    template <bool kMinusOne = false>
    __device__ static __forceinline__ void phi_tile(uint8_t* tile, uint8_t* lo_tile, int ct, int n, int dcols,
                                                    const float* w, float* colpart, uint8_t* copy_tile = nullptr,
                                                    const float* scale = nullptr) {
        // a whole tile (every row and column in range: all chunks but a short last one of a
        // full-width head) takes the copy of the body without the per-element range test; a
        // 64-wide head leaves the upper column block alone (its TMA zero fill stays in place,
        // and the lo and copy tiles there feed only output columns that are never stored)
        if (n >= kC && dcols >= kD)
            phi_tile_body<true, false, kMinusOne>(tile, lo_tile, ct, n, dcols, w, colpart, copy_tile, scale);
        else if (dcols <= kD / 2)
            phi_tile_body<false, true, kMinusOne>(tile, lo_tile, ct, n, dcols, w, colpart, copy_tile, scale);
        else
            phi_tile_body<false, false, kMinusOne>(tile, lo_tile, ct, n, dcols, w, colpart, copy_tile, scale);
    }
    template <bool kWhole, bool kHalf, bool kMinusOne = false>
    __device__ static __forceinline__ void phi_tile_body(uint8_t* tile, uint8_t* lo_tile, int ct, int n, int dcols,
                                                         const float* w, float* colpart, uint8_t* copy_tile,
                                                         const float* scale) {
        float zp[2][8];
#pragma unroll
        for (int b = 0; b < 2; ++b)
#pragma unroll
            for (int e = 0; e < 8; ++e) zp[b][e] = 0.f;
        uint4 v[kJ];
#pragma unroll
        for (int j = 0; j < kJ; ++j)
            if (!kHalf || vec_block(j) == 0) v[j] = *reinterpret_cast<const uint4*>(tile + vec_off(ct, j));
#pragma unroll
        for (int j = 0; j < kJ; ++j) {
            if (kHalf && vec_block(j) != 0) continue;
            const int row = vec_row(ct, j);
            uint32_t* u = reinterpret_cast<uint32_t*>(&v[j]);
            uint4 l;
            uint32_t* ul = reinterpret_cast<uint32_t*>(&l);
            const bool valid = kWhole || (row < n && (kHalf || 64 * vec_block(j) + 8 * vec_lc(ct) < dcols));
            const float wr = (w && valid) ? w[row] : 1.f;
            const float sr = scale ? scale[row] : 1.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float a = valid ? phi_f(bf_lo(u[e])) * sr : 0.f, b = valid ? phi_f(bf_hi(u[e])) * sr : 0.f;
                u[e] = pack_bf16x2(a, b);
                if (kMinusOne)
                    ul[e] = valid ? pack_bf16x2(a - 1.f, b - 1.f) : 0u;
                else
                    ul[e] = pack_bf16x2(a - bf_lo(u[e]), b - bf_hi(u[e]));
                if (colpart) {
                    zp[vec_block(j)][2 * e] = fmaf(wr, bf_lo(u[e]), zp[vec_block(j)][2 * e]);
                    zp[vec_block(j)][2 * e + 1] = fmaf(wr, bf_hi(u[e]), zp[vec_block(j)][2 * e + 1]);
                }
            }
            *reinterpret_cast<uint4*>(tile + vec_off(ct, j)) = v[j];
            if (lo_tile) *reinterpret_cast<uint4*>(lo_tile + vec_off(ct, j)) = l;
            if (copy_tile) *reinterpret_cast<uint4*>(copy_tile + vec_off(ct, j)) = v[j];
        }
        if (colpart) column_part(zp, colpart, ct);
    }
};

}  // namespace tc

// Host: a [BH][N][D] bf16 tensor as a 3-D TMA map with 64 x box_rows x 1 boxes
// and the 128-byte swizzle; rows past N inside a head read as zeros.
bool make_tmap_bf16_rows(CUtensorMap* map, const void* ptr, int BH, int N, int D, int box_rows);

}  // namespace la
