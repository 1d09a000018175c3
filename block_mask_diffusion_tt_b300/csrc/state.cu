// state.cu -- Mamba-2 state seeding: the denoiser's Mamba-2 layers start from the
// context tower's conv/SSM boundary states, layer by layer.
//
// Method (dothoosh.com "فرآیند انتشار در برابر رمزگشایی متوالی در مدل جدید انویدیا",
// architecture bullets: each denoiser Mamba-2 layer takes its initial state directly
// from the context tower's Mamba state; aitrends.kr "Nemotron-Labs-TwoTower-30B-A3B-
// Base-BF16", section "technical features": the context tower's conv/SSM boundary
// states are injected as the initial states of the denoiser's Mamba layers).
//
// One launch copies every (layer, state part, sequence) taking part: blockIdx.y picks
// the (layer, part, sequence) item, blockIdx.x a chunk of it; each thread moves
// 16-byte vectors with kUnroll loads in flight before their stores.  A copy of bytes:
// HBM-bound, every byte read once and written once.
#include "common.cuh"

namespace tt {
namespace {

constexpr int kSeedThreads = 512;
constexpr int kSeedUnroll = 8;
constexpr int64_t kChunkVec = static_cast<int64_t>(kSeedThreads) * kSeedUnroll;  // per CTA pass

struct SeedArgs {
    const char *src[TT_STATE_MAX_LAYERS * TT_STATE_MAX_PARTS];
    char *dst[TT_STATE_MAX_LAYERS * TT_STATE_MAX_PARTS];
    int64_t vecs[TT_STATE_MAX_PARTS];        // 16-byte vectors per sequence of each part
    int64_t src_stride[TT_STATE_MAX_PARTS];  // bytes between sequences
    int64_t dst_stride[TT_STATE_MAX_PARTS];
    int B, n_parts;
    const uint8_t *active;
};

__global__ void __launch_bounds__(kSeedThreads) state_seed_kernel(const SeedArgs a) {
    const int item = blockIdx.y;  // (layer * n_parts + part) * B + b
    const int b = item % a.B;
    const int lp = item / a.B;
    const int part = lp % a.n_parts;
    if (a.active && !a.active[b]) return;
    const int64_t n = a.vecs[part];
    const int4 *s = reinterpret_cast<const int4 *>(a.src[lp] + b * a.src_stride[part]);
    int4 *d = reinterpret_cast<int4 *>(a.dst[lp] + b * a.dst_stride[part]);
    for (int64_t v0 = static_cast<int64_t>(blockIdx.x) * kChunkVec + threadIdx.x; v0 < n;
         v0 += static_cast<int64_t>(gridDim.x) * kChunkVec) {
        int4 q[kSeedUnroll];
#pragma unroll
        for (int u = 0; u < kSeedUnroll; ++u) {
            const int64_t v = v0 + static_cast<int64_t>(u) * kSeedThreads;
            if (v < n) q[u] = __ldcs(s + v);
        }
#pragma unroll
        for (int u = 0; u < kSeedUnroll; ++u) {
            const int64_t v = v0 + static_cast<int64_t>(u) * kSeedThreads;
            if (v < n) __stcs(d + v, q[u]);
        }
    }
}

}  // namespace
}  // namespace tt

using namespace tt;

extern "C" tt_status tt_mamba_state_seed(const tt_state_desc *desc, const void *const *src,
                                         void *const *dst, const uint8_t *active,
                                         tt_stream_t stream) {
    const char *fn = "tt_mamba_state_seed";
    if (!desc) return fail(TT_ERR_INVALID_ARG, "%s: null desc", fn);
    if (desc->B < 0) return fail(TT_ERR_INVALID_ARG, "%s: B < 0", fn);
    if (desc->n_layers < 1 || desc->n_layers > TT_STATE_MAX_LAYERS)
        return fail(TT_ERR_INVALID_ARG, "%s: n_layers=%d (1..%d)", fn, desc->n_layers,
                    TT_STATE_MAX_LAYERS);
    if (desc->n_parts < 1 || desc->n_parts > TT_STATE_MAX_PARTS)
        return fail(TT_ERR_INVALID_ARG, "%s: n_parts=%d (1..%d)", fn, desc->n_parts,
                    TT_STATE_MAX_PARTS);
    if (desc->B == 0) return TT_OK;
    if (!src || !dst) return fail(TT_ERR_INVALID_ARG, "%s: null pointer array", fn);
    SeedArgs a;
    int64_t max_vecs = 0;
    for (int p = 0; p < desc->n_parts; ++p) {
        const int64_t bytes = desc->bytes[p];
        if (bytes <= 0 || bytes % 16)
            return fail(TT_ERR_UNSUPPORTED, "%s: part %d bytes %lld (a positive multiple of 16)",
                        fn, p, (long long)bytes);
        if (desc->src_stride[p] < bytes || desc->dst_stride[p] < bytes ||
            desc->src_stride[p] % 16 || desc->dst_stride[p] % 16)
            return fail(TT_ERR_UNSUPPORTED,
                        "%s: part %d strides must be multiples of 16 bytes, at least its size", fn,
                        p);
        a.vecs[p] = bytes / 16;
        a.src_stride[p] = desc->src_stride[p];
        a.dst_stride[p] = desc->dst_stride[p];
        if (a.vecs[p] > max_vecs) max_vecs = a.vecs[p];
    }
    const int items = desc->n_layers * desc->n_parts;
    for (int i = 0; i < items; ++i) {
        if (!src[i] || !dst[i]) return fail(TT_ERR_INVALID_ARG, "%s: null pointer %d", fn, i);
        if (reinterpret_cast<uintptr_t>(src[i]) % 16 || reinterpret_cast<uintptr_t>(dst[i]) % 16)
            return fail(TT_ERR_INVALID_ARG, "%s: pointer %d not 16-byte aligned", fn, i);
        a.src[i] = static_cast<const char *>(src[i]);
        a.dst[i] = static_cast<char *>(dst[i]);
    }
    const int64_t ny = static_cast<int64_t>(items) * desc->B;
    if (ny > 65535) return fail(TT_ERR_UNSUPPORTED, "%s: n_layers*n_parts*B > 65535", fn);
    a.B = desc->B;
    a.n_parts = desc->n_parts;
    a.active = active;
    int64_t nx = (max_vecs + kChunkVec - 1) / kChunkVec;
    if (nx > 65535) nx = 65535;  // each CTA then loops over several chunks
    dim3 grid(static_cast<unsigned>(nx), static_cast<unsigned>(ny));
    state_seed_kernel<<<grid, kSeedThreads, 0, static_cast<cudaStream_t>(stream)>>>(a);
    return cuda_status(cudaGetLastError(), "tt_mamba_state_seed launch");
}
