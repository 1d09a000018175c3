// common.cuh -- internal helpers shared by the libtt translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "tt.h"

namespace tt {

// ---------------------------------------------------------------- host side
// Records a message for tt_last_error() and returns `s`.
tt_status fail(tt_status s, const char *fmt, ...);
// Maps a CUDA error to TT_ERR_CUDA with its message (TT_OK for cudaSuccess).
tt_status cuda_status(cudaError_t e, const char *what);
// SM count of the current device (cached per device).
int sm_count();

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Simple bump allocator over a caller-provided workspace.
struct Carve {
    char *base;
    size_t off = 0;
    explicit Carve(void *p) : base(static_cast<char *>(p)) {}
    template <typename T>
    T *take(size_t n) {
        off = align_up(off, 256);
        T *p = reinterpret_cast<T *>(base ? base + off : nullptr);
        off += n * sizeof(T);
        return p;
    }
    size_t bytes() const { return align_up(off, 256); }
};

// ---------------------------------------------------------------- device side
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// Round-to-nearest-even fp32 -> bf16 bits (inputs are finite or NaN).
__device__ __forceinline__ uint32_t f32_to_bf16_bits(float f) {
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0x7FC0u;  // NaN
    return (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

}  // namespace tt
