// simt_common.cuh -- pieces shared by the CUDA-core (FFMA) kernels: the
// 256-thread 16 x 16 layout, the shared-memory carver and the chunk tile load.
#pragma once

#include "la_internal.cuh"

namespace la {
namespace simt {

constexpr int kC = 64;         // chunk length of the CUDA-core kernels
constexpr int kThreads = 256;  // 16 x 16
constexpr int kMaxT = 8;       // 128 / 16: largest register tile extent

struct Smem {
    // carve a float array of `n` elements, 16-byte aligned
    char* p;
    __device__ float* take(size_t n) {
        float* r = reinterpret_cast<float*>(p);
        p += ((n * sizeof(float) + 15) / 16) * 16;
        return r;
    }
};

// Load rows [c0, c0 + n) of one head's [N][D] matrix into dst[C][ld] as fp32,
// applying phi when asked; rows n..C-1 are zero (a masked tail is exactly 0,
// never phi(0) = 1).
template <typename T>
__device__ __forceinline__ void load_tile(float* dst, int ld, const T* __restrict__ src, int c0, int n, int D,
                                          bool apply_phi) {
    for (int idx = threadIdx.x; idx < kC * D; idx += kThreads) {
        int t = idx / D, d = idx - t * D;
        float x = 0.f;
        if (t < n) {
            x = to_f32(src[(size_t)(c0 + t) * D + d]);
            if (apply_phi) x = phi_f(x);
        }
        dst[t * ld + d] = x;
    }
}

// Bytes of a float array of n elements as carved by Smem::take.
inline size_t smem_floats(size_t n) { return ((n * 4 + 15) / 16) * 16; }

}  // namespace simt
}  // namespace la
