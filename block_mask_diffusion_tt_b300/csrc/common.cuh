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

// A logits producer of the in-block loop: a function and its context.
struct LoopProducer {
    tt_status (*fn)(void *ctx, int32_t step, const int32_t *tokens, const uint8_t *is_masked,
                    void *logits, tt_stream_t stream);
    void *ctx;
};
// The in-block iteration (unmask.cu): tt_denoise_block_loop's steps; with
// init_active (device uint8[B], nullable) a start at step 0 masks only the
// positions of the sequences that take part.
tt_status run_block_loop(const tt_unmask_desc *d, int32_t steps_per_block, int32_t start_step,
                         int32_t stop_step, const LoopProducer &prod, void *logits_buf,
                         int32_t *tokens, uint8_t *is_masked, int32_t *steps_used,
                         int32_t *committed_step, const uint8_t *init_active, void *workspace,
                         size_t workspace_bytes, cudaStream_t stream, int32_t timeout_ms,
                         int32_t *steps_run, const char *fn);
// Bytes of the workspace run_block_loop needs (0 on an invalid desc).
size_t block_loop_workspace_bytes(const tt_unmask_desc *d);

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

// Packed fp32 pairs (sm_100 f32x2 instructions).
__device__ __forceinline__ uint64_t pk2(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void upk2(uint64_t r, float &a, float &b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// ---------------------------------------------------------------- mbarriers
// Every wait on an mbarrier is bounded: after kWaitLimitNs it records an error code
// and returns false, so a kernel that would otherwise wait forever stops instead.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// try_wait that may suspend the thread until the phase completes (or hint_ns
// passes), so a waiting warp takes no issue slots from the warps doing work.
__device__ __forceinline__ bool mbar_try_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Arrive that takes `after` as an input, so the arithmetic producing it cannot be
// scheduled below the arrive (a volatile asm orders memory accesses, not arithmetic).
__device__ __forceinline__ void mbar_arrive_after(uint32_t bar, float after) {
    asm volatile("{\n\t.reg .f32 dep;\n\tmov.f32 dep, %1;\n\t"
                 "mbarrier.arrive.shared::cta.b64 _, [%0];\n\t}\n" ::"r"(bar),
                 "f"(after)
                 : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// Waits for the phase of `parity` to complete.  Gives up (false) when another
// role has flagged an error or after kWaitLimitNs, flagging `code`.  Thread-level
// (the TMA producer runs on one thread).
static __device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, volatile int *err,
                                            int code) {
    const uint64_t t0 = globaltimer();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try(bar, parity)) return true;
        if ((i & 63) == 0) {
            if (*err) return false;
            if (globaltimer() - t0 > kWaitLimitNs) {
                atomicCAS(const_cast<int *>(err), 0, code);
                return false;
            }
        }
    }
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *err,
                                          int code) {
    if (mbar_try(bar, parity)) return true;
    return mbar_wait_slow(bar, parity, err, code);
}
// Warp-collective form: every lane of a converged warp calls it and all get the
// same answer.  Inline, so a wait that is already satisfied costs a few cycles.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *err,
                                          int code) {
    if (__any_sync(0xFFFFFFFFu, mbar_try(bar, parity))) return true;
    uint64_t t0 = 0;
    for (uint32_t i = 1;; ++i) {
        if (__any_sync(0xFFFFFFFFu, mbar_try(bar, parity))) return true;
        if ((i & 255) == 0) {
            int stop = 0;
            if ((threadIdx.x & 31) == 0) {
                const uint64_t now = globaltimer();
                if (t0 == 0) t0 = now;
                if (*err) {
                    stop = 1;
                } else if (now - t0 > kWaitLimitNs) {
                    atomicCAS(const_cast<int *>(err), 0, code);
                    stop = 1;
                }
            }
            if (__shfl_sync(0xFFFFFFFFu, stop, 0)) return false;
        }
    }
}
// Warp-collective wait that sleeps between polls (__nanosleep, backing off from 32
// to 256 ns, then a try_wait that may suspend): for warps that wait most of the
// time, where spinning would take issue slots from the warps doing the work.  Same
// bounds and error flag as warp_wait.
__device__ __forceinline__ bool warp_wait_sleep(uint32_t bar, uint32_t parity, volatile int *err,
                                                int code) {
    if (__any_sync(0xFFFFFFFFu, mbar_try(bar, parity))) return true;
    uint64_t t0 = 0;
    uint32_t nap = 32;
    for (uint32_t i = 1;; ++i) {
        __nanosleep(nap);
        if (nap < 256) nap <<= 1;
        if (__any_sync(0xFFFFFFFFu, mbar_try_sleep(bar, parity, 20000u))) return true;
        if ((i & 15) == 0) {
            int stop = 0;
            if ((threadIdx.x & 31) == 0) {
                const uint64_t now = globaltimer();
                if (t0 == 0) t0 = now;
                if (*err) {
                    stop = 1;
                } else if (now - t0 > kWaitLimitNs) {
                    atomicCAS(const_cast<int *>(err), 0, code);
                    stop = 1;
                }
            }
            if (__shfl_sync(0xFFFFFFFFu, stop, 0)) return false;
        }
    }
}
// Thread-level form of warp_wait_sleep.
static __device__ __noinline__ bool mbar_wait_sleep(uint32_t bar, uint32_t parity,
                                                    volatile int *err, int code) {
    if (mbar_try(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    uint32_t nap = 32;
    for (uint32_t i = 1;; ++i) {
        __nanosleep(nap);
        if (nap < 256) nap <<= 1;
        if (mbar_try_sleep(bar, parity, 20000u)) return true;
        if ((i & 15) == 0) {
            if (*err) return false;
            if (globaltimer() - t0 > kWaitLimitNs) {
                atomicCAS(const_cast<int *>(err), 0, code);
                return false;
            }
        }
    }
}
// Bounded wait that ignores the error flag (used to drain copies in flight).
static __device__ __noinline__ bool mbar_drain(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = globaltimer();
    while (!mbar_try(bar, parity))
        if (globaltimer() - t0 > kWaitLimitNs) return false;
    return true;
}

// TMA tile load; `policy` is an L2 cache policy (createpolicy).

// Bulk copy global -> shared (16-byte aligned, size a multiple of 16) completing
// on an mbarrier; `policy` is an L2 cache policy (createpolicy).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                          uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}
// Data read once: first in line for eviction from L2.
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
// Data several SMs read at about the same time: last in line for eviction from L2.
__device__ __forceinline__ uint64_t l2_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

}  // namespace tt
