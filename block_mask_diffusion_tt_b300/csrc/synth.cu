// synth.cu -- device implementation of the counter-based synthetic logits
// generator (a stand-in for the denoiser forward in benches and tests).
//
// Definition (SplitMix64 output function, Steele, Lea & Flood, OOPSLA 2014;
// finaliser constants of Stafford's Mix13), written here independently of the
// Python generator and checked bit-for-bit against it:
//   key  = mix64(mix64(seed ^ TAG_LOGITS) + (step+1)*GAMMA)
//   word = mix64(key + (n+1)*GAMMA), n = ((b*S+s)*V + v)*3 + j
//   z    = (sum of twelve 16-bit fields - 393216) * (sigma/65536), fp32
//   spike row: w = mix64(mix64(key ^ TAG_SPIKE) + (row+1)*GAMMA),
//              (w>>32) < threshold -> +8 at token (w & 0xFFFFFFFF) % V
#include "common.cuh"

namespace tt {
namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;
constexpr uint64_t kTagLogits = 0x6C6F67697473ull;
constexpr uint64_t kTagSpike = 0x7370696B65ull;

__host__ __device__ __forceinline__ uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

__device__ __forceinline__ uint32_t fields16(uint64_t w) {
    return static_cast<uint32_t>(w & 0xFFFF) + static_cast<uint32_t>((w >> 16) & 0xFFFF) +
           static_cast<uint32_t>((w >> 32) & 0xFFFF) + static_cast<uint32_t>(w >> 48);
}

template <bool BF16>
__global__ void __launch_bounds__(256) synth_logits_kernel(uint64_t key, uint64_t skey, int S,
                                                           int V, float sig, uint64_t thr,
                                                           void *out) {
    const int row = blockIdx.y;
    const uint64_t w = mix64(skey + (static_cast<uint64_t>(row) + 1) * kGamma);
    const bool spike = (w >> 32) < thr;
    const int spike_tok = static_cast<int>((w & 0xFFFFFFFFull) % static_cast<uint64_t>(V));
    for (int v = blockIdx.x * blockDim.x + threadIdx.x; v < V; v += gridDim.x * blockDim.x) {
        const uint64_t n = (static_cast<uint64_t>(row) * V + v) * 3;
        uint32_t acc = 0;
#pragma unroll
        for (int j = 0; j < 3; ++j) acc += fields16(mix64(key + (n + j + 1) * kGamma));
        float z = __fmul_rn(static_cast<float>(static_cast<int>(acc) - 393216), sig);
        if (spike && v == spike_tok) z = __fadd_rn(z, 8.0f);
        const size_t idx = static_cast<size_t>(row) * V + v;
        if (BF16)
            static_cast<uint16_t *>(out)[idx] = static_cast<uint16_t>(f32_to_bf16_bits(z));
        else
            static_cast<float *>(out)[idx] = z;
    }
}

}  // namespace
}  // namespace tt

using namespace tt;

extern "C" {

tt_status tt_synth_logits(uint64_t seed, int32_t step, int32_t B, int32_t S, int32_t V,
                          tt_dtype dtype, float sigma, uint64_t spike_threshold, void *out,
                          tt_stream_t stream) {
    const char *fn = "tt_synth_logits";
    if (B < 0 || S < 1 || V < 1 || step < 0) return fail(TT_ERR_INVALID_ARG, "%s: bad shape", fn);
    if (dtype != TT_F32 && dtype != TT_BF16) return fail(TT_ERR_INVALID_ARG, "%s: bad dtype", fn);
    if (!(sigma >= 0.f) || !isfinite(sigma)) return fail(TT_ERR_INVALID_ARG, "%s: bad sigma", fn);
    if (static_cast<int64_t>(B) * S > 65535) return fail(TT_ERR_UNSUPPORTED, "%s: B*S > 65535", fn);
    if (B == 0) return TT_OK;
    if (!out) return fail(TT_ERR_INVALID_ARG, "%s: null output", fn);
    const uint64_t key = mix64(mix64(seed ^ kTagLogits) + (static_cast<uint64_t>(step) + 1) * kGamma);
    const uint64_t skey = mix64(key ^ kTagSpike);
    const float sig = sigma / 65536.0f;
    const int bx = (V + 255) / 256 < 64 ? (V + 255) / 256 : 64;
    dim3 grid(bx, B * S);
    if (dtype == TT_BF16)
        synth_logits_kernel<true><<<grid, 256, 0, (cudaStream_t)stream>>>(key, skey, S, V, sig,
                                                                           spike_threshold, out);
    else
        synth_logits_kernel<false><<<grid, 256, 0, (cudaStream_t)stream>>>(key, skey, S, V, sig,
                                                                            spike_threshold, out);
    return cuda_status(cudaGetLastError(), fn);
}

tt_status tt_synth_logits_producer(void *user, int32_t step, const int32_t *tokens,
                                   const uint8_t *is_masked, void *logits_out,
                                   tt_stream_t stream) {
    (void)tokens;
    (void)is_masked;
    const tt_synth_params *p = static_cast<const tt_synth_params *>(user);
    if (!p) return fail(TT_ERR_INVALID_ARG, "tt_synth_logits_producer: null params");
    const int i = step < TT_SYNTH_MAX_STEPS ? step : TT_SYNTH_MAX_STEPS - 1;
    return tt_synth_logits(p->seed, step, p->B, p->S, p->V, p->dtype, p->sigma,
                           p->spike_threshold[i < 0 ? 0 : i], logits_out, stream);
}

}  // extern "C"
