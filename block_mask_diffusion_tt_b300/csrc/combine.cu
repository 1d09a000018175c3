// combine.cu -- joins two attention results over disjoint key sets into the result
// over their union, by their log-sum-exps.
//
// With the block's own keys and the context prefix's keys attended separately (the
// aitrends.kr page, "Nemotron-Labs-TwoTower-30B-A3B-Base-BF16", section "technical
// features", names in-block self-attention and layer-aligned attention to the context
// separately), each result is o_i = sum_j w_ij v_j / Z_i with lse_i = log Z_i.  The
// softmax over the union of the two key sets is then
//     o = (e^(lse_1 - M) o_1 + e^(lse_2 - M) o_2) / (e^(lse_1 - M) + e^(lse_2 - M)),
//     lse = M + log(e^(lse_1 - M) + e^(lse_2 - M)),   M = max(lse_1, lse_2),
// and a side without keys (lse = -inf) weighs nothing.
//
// One thread per (b, s, h) row and 8 output columns: 16-byte loads of both inputs, one
// 16-byte store.  Memory-bound; each byte is read or written once.
#include "common.cuh"

namespace tt {
namespace {

constexpr int kCombineThreads = 256;

__global__ void __launch_bounds__(kCombineThreads)
    lse_combine_kernel(int64_t rows, int S, int Hq, int cols8, const uint4 *o1, const float *lse1,
                       const uint4 *o2, const float *lse2, uint4 *out, float *lse_out) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * kCombineThreads + threadIdx.x;
    if (i >= rows * cols8) return;
    const int64_t row = i / cols8;  // (b, s, h) in [B, S, Hq] order
    const int h = static_cast<int>(row % Hq);
    const int64_t bs = row / Hq;
    const int s = static_cast<int>(bs % S);
    const int64_t b = bs / S;
    const int64_t li = (b * Hq + h) * S + s;  // [B, Hq, S]
    const float l1 = lse1[li], l2 = lse2[li];
    const float M = fmaxf(l1, l2);
    float w1 = 0.f, w2 = 0.f;
    if (M != -INFINITY) {
        w1 = l1 == -INFINITY ? 0.f : __expf(l1 - M);
        w2 = l2 == -INFINITY ? 0.f : __expf(l2 - M);
    }
    const float den = w1 + w2;
    const float inv = den > 0.f ? 1.f / den : 0.f;
    const float a1 = w1 * inv, a2 = w2 * inv;
    const uint4 x = o1[i], y = o2[i];
    uint4 r;
    r.x = pack_bf16x2(a1 * bf16_lo(x.x) + a2 * bf16_lo(y.x), a1 * bf16_hi(x.x) + a2 * bf16_hi(y.x));
    r.y = pack_bf16x2(a1 * bf16_lo(x.y) + a2 * bf16_lo(y.y), a1 * bf16_hi(x.y) + a2 * bf16_hi(y.y));
    r.z = pack_bf16x2(a1 * bf16_lo(x.z) + a2 * bf16_lo(y.z), a1 * bf16_hi(x.z) + a2 * bf16_hi(y.z));
    r.w = pack_bf16x2(a1 * bf16_lo(x.w) + a2 * bf16_lo(y.w), a1 * bf16_hi(x.w) + a2 * bf16_hi(y.w));
    out[i] = r;
    if (lse_out && i % cols8 == 0) lse_out[li] = den > 0.f ? M + __logf(den) : -INFINITY;
}

}  // namespace
}  // namespace tt

using namespace tt;

extern "C" tt_status tt_attn_lse_combine(int32_t B, int32_t S, int32_t Hq, int32_t d,
                                         const void *o1, const float *lse1, const void *o2,
                                         const float *lse2, void *out, float *lse_out,
                                         tt_stream_t stream) {
    const char *fn = "tt_attn_lse_combine";
    if (B < 0 || S < 1 || Hq < 1 || d < 8 || d % 8)
        return fail(TT_ERR_INVALID_ARG, "%s: bad shape B=%d S=%d Hq=%d d=%d", fn, B, S, Hq, d);
    if (B == 0) return TT_OK;
    if (!o1 || !o2 || !lse1 || !lse2 || !out) return fail(TT_ERR_INVALID_ARG, "%s: null pointer", fn);
    const void *p16[3] = {o1, o2, out};
    for (int i = 0; i < 3; ++i)
        if (reinterpret_cast<uintptr_t>(p16[i]) % 16)
            return fail(TT_ERR_INVALID_ARG, "%s: outputs/inputs not 16-byte aligned", fn);
    const int64_t rows = static_cast<int64_t>(B) * S * Hq;
    const int64_t n = rows * (d / 8);
    const int64_t blocks = (n + kCombineThreads - 1) / kCombineThreads;
    if (blocks > 2147483647LL) return fail(TT_ERR_UNSUPPORTED, "%s: too large", fn);
    lse_combine_kernel<<<static_cast<unsigned>(blocks), kCombineThreads, 0,
                         static_cast<cudaStream_t>(stream)>>>(
        rows, S, Hq, d / 8, static_cast<const uint4 *>(o1), lse1, static_cast<const uint4 *>(o2),
        lse2, static_cast<uint4 *>(out), lse_out);
    return cuda_status(cudaGetLastError(), "tt_attn_lse_combine launch");
}
