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
constexpr int kD = 128;             // Dk = Dv
constexpr int kTileBytes = 32768;   // one 128 x 128 bf16 tile
constexpr int kBlockBytes = 16384;  // one 64-column block

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
    return (lc >> 3) * kBlockBytes + row * 128 + (((lc & 7) ^ (row & 7)) << 4);
}
// Byte offset of element (row, col).
__device__ __forceinline__ int elem_off(int row, int col) { return chunk_off(row, col >> 3) + ((col & 7) << 1); }

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf_at(const uint8_t* tile, int row, int col) {
    const uint16_t h = *reinterpret_cast<const uint16_t*>(tile + elem_off(row, col));
    return __uint_as_float((uint32_t)h << 16);
}

// Barrier over the 128-thread compute warpgroup (named barrier 1) that ANDs a
// predicate across it, so every thread takes the same branch after a bounded wait.
__device__ __forceinline__ bool wg_all(bool v) {
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

// phi in place on a staged tile, rows >= n set to exactly 0.  Thread t
// (0..127) handles the 16-byte vectors t + 128 j (block j / 8, row
// ((t >> 3) + 16 j) & 127); the swizzle only permutes chunks within a row, so
// an elementwise map ignores it.
__device__ __forceinline__ void phi_tile(uint8_t* tile, int t, int n) {
#pragma unroll 4
    for (int j = 0; j < 16; ++j) {
        const int row = ((t >> 3) + 16 * j) & 127;
        uint4* p = reinterpret_cast<uint4*>(tile + (j >> 3) * kBlockBytes + row * 128 + (t & 7) * 16);
        uint4 w = *p;
        uint32_t* u = reinterpret_cast<uint32_t*>(&w);
        const bool valid = row < n;
#pragma unroll
        for (int e = 0; e < 4; ++e)
            u[e] = valid ? pack_bf16x2(phi_f(bf_lo(u[e])), phi_f(bf_hi(u[e]))) : 0u;
        *p = w;
    }
}

// phi in place as the bf16 "hi" part, plus lo = bf16(phi - hi) into `lo_tile`
// (same layout), so that hi + lo carries phi to about 2^-17 relative.
__device__ __forceinline__ void phi_tile_split(uint8_t* tile, uint8_t* lo_tile, int t, int n) {
#pragma unroll 4
    for (int j = 0; j < 16; ++j) {
        const int row = ((t >> 3) + 16 * j) & 127;
        const int off = (j >> 3) * kBlockBytes + row * 128 + (t & 7) * 16;
        uint4 w = *reinterpret_cast<const uint4*>(tile + off);
        uint32_t* u = reinterpret_cast<uint32_t*>(&w);
        uint4 l;
        uint32_t* ul = reinterpret_cast<uint32_t*>(&l);
        const bool valid = row < n;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float a = valid ? phi_f(bf_lo(u[e])) : 0.f, b = valid ? phi_f(bf_hi(u[e])) : 0.f;
            u[e] = pack_bf16x2(a, b);
            ul[e] = pack_bf16x2(a - bf_lo(u[e]), b - bf_hi(u[e]));
        }
        *reinterpret_cast<uint4*>(tile + off) = w;
        *reinterpret_cast<uint4*>(lo_tile + off) = l;
    }
}

// Row `row` scaled by 1/den[row] in place (rows >= n are left as loaded: zero).
__device__ __forceinline__ void scale_rows_tile(uint8_t* tile, int t, const float* inv_den) {
#pragma unroll 4
    for (int j = 0; j < 16; ++j) {
        const int row = ((t >> 3) + 16 * j) & 127;
        uint4* p = reinterpret_cast<uint4*>(tile + (j >> 3) * kBlockBytes + row * 128 + (t & 7) * 16);
        uint4 w = *p;
        uint32_t* u = reinterpret_cast<uint32_t*>(&w);
        const float s = inv_den[row];
#pragma unroll
        for (int e = 0; e < 4; ++e) u[e] = pack_bf16x2(bf_lo(u[e]) * s, bf_hi(u[e]) * s);
        *p = w;
    }
}

// Sum over rows 0..n-1 of column `col` of a tile, each row weighted by w[row] (or 1).
__device__ __forceinline__ float column_sum(const uint8_t* tile, int col, int n, const float* w) {
    float acc = 0.f;
    for (int row = 0; row < n; ++row) acc = fmaf(w ? w[row] : 1.f, bf_at(tile, row, col), acc);
    return acc;
}

// One TMEM row (32 lanes per warp) of 128 fp32 columns into a bf16 tile row
// (rows = TMEM lanes), e.g. the fp32 state S -> its bf16 MMA operand copy.
__device__ __forceinline__ void tmem_row_to_tile(uint32_t taddr, uint8_t* tile, int row) {
#pragma unroll
    for (int cb = 0; cb < 4; ++cb) {
        uint32_t w[32];
        tmem_ld32(taddr + 32 * cb, w);
        tmem_ld_wait();
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
            uint4 v4;
            v4.x = pack_bf16x2(__uint_as_float(w[8 * q4 + 0]), __uint_as_float(w[8 * q4 + 1]));
            v4.y = pack_bf16x2(__uint_as_float(w[8 * q4 + 2]), __uint_as_float(w[8 * q4 + 3]));
            v4.z = pack_bf16x2(__uint_as_float(w[8 * q4 + 4]), __uint_as_float(w[8 * q4 + 5]));
            v4.w = pack_bf16x2(__uint_as_float(w[8 * q4 + 6]), __uint_as_float(w[8 * q4 + 7]));
            *reinterpret_cast<uint4*>(tile + chunk_off(row, 4 * cb + q4)) = v4;
        }
    }
}

// The same row as a hi + lo pair of bf16 tiles, hi = bf16(x), lo = bf16(x - hi):
// a product with (hi + lo) carries the fp32 state to about 2^-17 relative, which
// the backward needs where two large inter-chunk terms cancel.
__device__ __forceinline__ void tmem_row_to_tiles_split(uint32_t taddr, uint8_t* hi, uint8_t* lo, int row) {
#pragma unroll
    for (int cb = 0; cb < 4; ++cb) {
        uint32_t w[32];
        tmem_ld32(taddr + 32 * cb, w);
        tmem_ld_wait();
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t h4[4], l4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float x0 = __uint_as_float(w[8 * q4 + 2 * e]), x1 = __uint_as_float(w[8 * q4 + 2 * e + 1]);
                h4[e] = pack_bf16x2(x0, x1);
                l4[e] = pack_bf16x2(x0 - bf_lo(h4[e]), x1 - bf_hi(h4[e]));
            }
            const int off = chunk_off(row, 4 * cb + q4);
            *reinterpret_cast<uint4*>(hi + off) = make_uint4(h4[0], h4[1], h4[2], h4[3]);
            *reinterpret_cast<uint4*>(lo + off) = make_uint4(l4[0], l4[1], l4[2], l4[3]);
        }
    }
}

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

// ------------------------------------------------------------------ 256-thread compute group
// Warps 2-9 of a CTA: thread ct = tid - 64.  For row-wise TMEM work, warp w owns
// TMEM lanes 32*(w%4) .. +31 and column half h = (w - 2) / 4 of those rows.  For
// whole-tile elementwise work, thread ct owns the 16-byte vectors ct + 256 j
// (j < 8): block j / 4, row ((ct >> 3) + 32 j) & 127, physical chunk ct & 7,
// logical chunk lc = (ct & 7) ^ ((ct >> 3) & 7), i.e. columns 64*(j/4) + 8*lc + e.
constexpr int kGroupThreads = 256;

__device__ __forceinline__ bool grp_all(bool v) {
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
__device__ __forceinline__ void grp_sync() { named_barrier(1, kGroupThreads); }

__device__ __forceinline__ int grp_vec_row(int ct, int j) { return ((ct >> 3) + 32 * j) & 127; }
__device__ __forceinline__ int grp_vec_off(int ct, int j) {
    return (j >> 2) * kBlockBytes + grp_vec_row(ct, j) * 128 + (ct & 7) * 16;
}
__device__ __forceinline__ int grp_vec_lc(int ct) { return (ct & 7) ^ ((ct >> 3) & 7); }

// Column partial sums zp[block][e] (for columns 64*block + 8*lc + e of this
// thread) summed over the four lanes of the warp that share lc (lanes l, l^9,
// l^18, l^27) and stored by lanes 0-7 as this warp's row of part[8][128]
// (no atomics: the eight warps' rows are added by grp_column_sum after a
// group barrier).
__device__ __forceinline__ void grp_column_part(float (&zp)[2][8], float* part, int ct) {
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
        float* row = part + (ct >> 5) * 128 + 8 * grp_vec_lc(ct);
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            *reinterpret_cast<float4*>(row + 64 * b) = make_float4(zp[b][0], zp[b][1], zp[b][2], zp[b][3]);
            *reinterpret_cast<float4*>(row + 64 * b + 4) = make_float4(zp[b][4], zp[b][5], zp[b][6], zp[b][7]);
        }
    }
}
// Column c (0..127) of part[8][128] summed over the eight warps.
__device__ __forceinline__ float grp_column_sum(const float* part, int c) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) s += part[128 * w + c];
    return s;
}

// phi in place on a staged tile (rows >= n exactly 0).  With colpart, the
// column sums of the rounded values (weighted by w[row] when w is given) go to
// colpart[8][128] as per-warp partials (see grp_column_part).  With lo_tile,
// also writes lo = bf16(phi - hi) there; with copy_tile, a second copy of the
// rounded phi.
__device__ __forceinline__ void grp_phi_tile(uint8_t* tile, uint8_t* lo_tile, int ct, int n, const float* w,
                                             float* colpart, uint8_t* copy_tile = nullptr) {
    float zp[2][8];
#pragma unroll
    for (int b = 0; b < 2; ++b)
#pragma unroll
        for (int e = 0; e < 8; ++e) zp[b][e] = 0.f;
    uint4 v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = *reinterpret_cast<const uint4*>(tile + grp_vec_off(ct, j));
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int row = grp_vec_row(ct, j);
        uint32_t* u = reinterpret_cast<uint32_t*>(&v[j]);
        uint4 l;
        uint32_t* ul = reinterpret_cast<uint32_t*>(&l);
        const bool valid = row < n;
        const float wr = (w && valid) ? w[row] : 1.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float a = valid ? phi_f(bf_lo(u[e])) : 0.f, b = valid ? phi_f(bf_hi(u[e])) : 0.f;
            u[e] = pack_bf16x2(a, b);
            ul[e] = pack_bf16x2(a - bf_lo(u[e]), b - bf_hi(u[e]));
            if (colpart) {
                zp[j >> 2][2 * e] = fmaf(wr, bf_lo(u[e]), zp[j >> 2][2 * e]);
                zp[j >> 2][2 * e + 1] = fmaf(wr, bf_hi(u[e]), zp[j >> 2][2 * e + 1]);
            }
        }
        *reinterpret_cast<uint4*>(tile + grp_vec_off(ct, j)) = v[j];
        if (lo_tile) *reinterpret_cast<uint4*>(lo_tile + grp_vec_off(ct, j)) = l;
        if (copy_tile) *reinterpret_cast<uint4*>(copy_tile + grp_vec_off(ct, j)) = v[j];
    }
    if (colpart) grp_column_part(zp, colpart, ct);
}

// Every row of a staged tile scaled by s[row], rounded to bf16, in place.
__device__ __forceinline__ void grp_scale_rows(uint8_t* tile, int ct, const float* s) {
    uint4 v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = *reinterpret_cast<const uint4*>(tile + grp_vec_off(ct, j));
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint32_t* u = reinterpret_cast<uint32_t*>(&v[j]);
        const float f = s[grp_vec_row(ct, j)];
#pragma unroll
        for (int e = 0; e < 4; ++e) u[e] = pack_bf16x2(bf_lo(u[e]) * f, bf_hi(u[e]) * f);
        *reinterpret_cast<uint4*>(tile + grp_vec_off(ct, j)) = v[j];
    }
}

}  // namespace tc

// Host: a [BH][N][D] bf16 tensor as a 3-D TMA map with 64 x box_rows x 1 boxes
// and the 128-byte swizzle; rows past N inside a head read as zeros.
bool make_tmap_bf16_rows(CUtensorMap* map, const void* ptr, int BH, int N, int D, int box_rows);

}  // namespace la
