// adaln.cu -- adaLN-single: the per-timestep scale, shift and gate of one denoiser
// layer, computed once per step from the diffusion timestep.
//
// Method (aitrends.kr "Nemotron-Labs-TwoTower-30B-A3B-Base-BF16", section "technical
// features": time conditioning by an adaLN-single module that injects scale, shift and
// gate into every denoiser layer per timestep, about 1.5 M added parameters;
// dothoosh.com "فرآیند انتشار در برابر رمزگشایی متوالی در مدل جدید انویدیا",
// architecture bullets).  Per sequence b with timestep t_b:
//   e   = [cos(t w_i)]_{i<F/2} ++ [sin(t w_i)]_{i<F/2},  w_i = 10000^(-i/(F/2))
//   h   = SiLU(W1 e + b1)                         (W1 [Dh, F])
//   m   = W2 h + b2 + embed[layer]                (W2 [3N, Dh], embed [layers, 3N])
//   shift, scale, gate = m[0:N], m[N:2N], m[2N:3N]
//
// One kernel: every CTA first computes h for all sequences into shared memory (B*Dh
// values, each a dot product of length F), then each thread owns output rows of W2
// and dots each row with every sequence's h, so W2 is read once for the whole batch.
#include <math.h>

#include <mutex>

#include "common.cuh"

namespace tt {
namespace {

constexpr int kAdaThreads = 256;
constexpr int kAdaMaxB = 64;     // sequences per pass over W2
constexpr int kAdaMaxF = 1024;
constexpr int kAdaMaxDh = 512;

struct AdaArgs {
    const float *t, *w1, *b1, *w2, *b2, *embed;
    float *shift, *scale, *gate;
    int B, F, Dh, N, layer;
};

__global__ void __launch_bounds__(kAdaThreads) adaln_kernel(const AdaArgs a) {
    extern __shared__ float sh[];  // h[kAdaMaxB][Dh] then e[F]
    float *h = sh;
    float *e = sh + kAdaMaxB * a.Dh;
    const int half = a.F / 2;
    const int rows = 3 * a.N;
    const int o = blockIdx.x * kAdaThreads + threadIdx.x;  // output row of W2
    for (int b0 = 0; b0 < a.B; b0 += kAdaMaxB) {
        const int nb = min(kAdaMaxB, a.B - b0);
        __syncthreads();
        // h for sequences b0 .. b0+nb-1: the embedding of one sequence at a time
        for (int bi = 0; bi < nb; ++bi) {
            const float t = a.t[b0 + bi];
            for (int i = threadIdx.x; i < half; i += kAdaThreads) {
                // w_i = 10000^(-i/half) = 2^(-i/half * log2(10000))
                const float w = exp2f(-static_cast<float>(i) / half * 13.287712379549449f);
                float sv, cv;
                sincosf(t * w, &sv, &cv);
                e[i] = cv;
                e[half + i] = sv;
            }
            __syncthreads();
            for (int j = threadIdx.x; j < a.Dh; j += kAdaThreads) {
                const float *wr = a.w1 + static_cast<size_t>(j) * a.F;
                float acc = a.b1[j];
                for (int f = 0; f < a.F; ++f) acc = fmaf(wr[f], e[f], acc);
                h[bi * a.Dh + j] = acc / (1.f + expf(-acc));  // SiLU
            }
            __syncthreads();
        }
        if (o < rows) {
            const float *wr = a.w2 + static_cast<size_t>(o) * a.Dh;
            const float base = a.b2[o] + a.embed[static_cast<size_t>(a.layer) * rows + o];
            float *dst = o < a.N ? a.shift : (o < 2 * a.N ? a.scale : a.gate);
            const int col = o % a.N;
            for (int bi = 0; bi < nb; ++bi) {
                const float *hb = h + bi * a.Dh;
                float acc = base;
                for (int j = 0; j < a.Dh; ++j) acc = fmaf(wr[j], hb[j], acc);
                dst[static_cast<size_t>(b0 + bi) * a.N + col] = acc;
            }
        }
    }
}

}  // namespace
}  // namespace tt

using namespace tt;

extern "C" tt_status tt_adaln_single(const tt_adaln_desc *desc, const float *t, const float *w1,
                                     const float *b1, const float *w2, const float *b2,
                                     const float *embed, float *shift, float *scale, float *gate,
                                     tt_stream_t stream) {
    const char *fn = "tt_adaln_single";
    if (!desc) return fail(TT_ERR_INVALID_ARG, "%s: null desc", fn);
    const tt_adaln_desc &d = *desc;
    if (d.B < 0 || d.F < 2 || d.F % 2 || d.Dh < 1 || d.N < 1 || d.layer < 0 || d.n_layers < 1 ||
        d.layer >= d.n_layers)
        return fail(TT_ERR_INVALID_ARG, "%s: bad sizes B=%d F=%d Dh=%d N=%d layer=%d/%d", fn, d.B,
                    d.F, d.Dh, d.N, d.layer, d.n_layers);
    if (d.F > kAdaMaxF || d.Dh > kAdaMaxDh)
        return fail(TT_ERR_UNSUPPORTED, "%s: F <= %d and Dh <= %d", fn, kAdaMaxF, kAdaMaxDh);
    if (d.B == 0) return TT_OK;
    if (!t || !w1 || !b1 || !w2 || !b2 || !embed || !shift || !scale || !gate)
        return fail(TT_ERR_INVALID_ARG, "%s: null pointer", fn);
    const int64_t rows = 3LL * d.N;
    if (rows > (int64_t(1) << 30)) return fail(TT_ERR_UNSUPPORTED, "%s: N too large", fn);
    AdaArgs a{t, w1, b1, w2, b2, embed, shift, scale, gate, d.B, d.F, d.Dh, d.N, d.layer};
    const size_t smem = sizeof(float) * (static_cast<size_t>(kAdaMaxB) * d.Dh + d.F);
    if (smem > 48 * 1024) {  // once per device: the largest dynamic shared memory the kernel takes
        static std::once_flag once[64];
        static cudaError_t set_err[64];
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return cuda_status(e, "tt_adaln_single");
        if (dev < 0 || dev >= 64) return fail(TT_ERR_UNSUPPORTED, "%s: device index %d >= 64", fn, dev);
        std::call_once(once[dev], [dev] {
            set_err[dev] = cudaFuncSetAttribute(
                adaln_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                static_cast<int>(sizeof(float) * (kAdaMaxB * kAdaMaxDh + kAdaMaxF)));
        });
        if (set_err[dev] != cudaSuccess) return cuda_status(set_err[dev], "tt_adaln_single: smem attribute");
    }
    const unsigned grid = static_cast<unsigned>((rows + kAdaThreads - 1) / kAdaThreads);
    adaln_kernel<<<grid, kAdaThreads, smem, static_cast<cudaStream_t>(stream)>>>(a);
    return cuda_status(cudaGetLastError(), "tt_adaln_single launch");
}
