// kv.cu -- appends a committed block's K/V to the context cache of every layer.
//
// Method (dothoosh.com "فرآیند انتشار در برابر رمزگشایی متوالی در مدل جدید انویدیا",
// section "two-tower mechanism"): once a block is fully committed it becomes clean
// context; the context tower takes it in, and the next block attends to the longer
// prefix.  Here the block's K/V rows of each layer are copied into rows
// [L_b, L_b + S) of that layer's cache and the prefix length grows by S.
//
// Two launches.  The copy: one CTA per (layer, K or V, sequence) moves that
// block's S x Hkv rows as 16-byte vectors (coalesced on both sides: a row is d
// contiguous elements), kKvUnroll loads in flight per thread before their stores,
// to rows [L_b, L_b + S).  Then one small CTA advances every length taking part;
// stream order puts it after all copies, which read the old lengths.  A sequence
// that is not active, or whose block would not fit under Lmax, is left as it is;
// the second case is counted in a device word.
#include "common.cuh"

namespace tt {
namespace {

constexpr int kKvThreads = 256;
constexpr int kKvUnroll = 4;
constexpr int kLenThreads = 256;

struct KvArgs {
    const uint16_t *kb[TT_KV_MAX_LAYERS];
    const uint16_t *vb[TT_KV_MAX_LAYERS];
    uint16_t *kc[TT_KV_MAX_LAYERS];
    uint16_t *vc[TT_KV_MAX_LAYERS];
    int64_t cs[3], bs[3];  // cache [B, Hkv, Lmax, d] and block [B, S, Hkv, d] strides
    int B, S, Hkv, d, Lmax, nl;
    int32_t *lens;
    const uint8_t *active;
    int32_t *overflow;
};

__device__ __forceinline__ bool takes_part(const KvArgs &a, int b, int L) {
    const bool act = a.active == nullptr || a.active[b] != 0;
    return act && L >= 0 && static_cast<int64_t>(L) + a.S <= a.Lmax;
}

// blockIdx.x = layer * 2 + (0: K, 1: V), blockIdx.y = sequence
__global__ void __launch_bounds__(kKvThreads) kv_copy_kernel(const KvArgs a) {
    const int b = blockIdx.y, l = blockIdx.x >> 1, kv = blockIdx.x & 1;
    const int L = a.lens[b];
    if (!takes_part(a, b, L)) return;
    const int vpr = a.d / 8;  // 16-byte vectors per row
    const int total = a.S * a.Hkv * vpr;
    const uint16_t *sb = (kv ? a.vb[l] : a.kb[l]) + b * a.bs[0];
    uint16_t *db = (kv ? a.vc[l] : a.kc[l]) + b * a.cs[0];
    for (int i0 = threadIdx.x; i0 < total; i0 += kKvUnroll * kKvThreads) {
        uint4 val[kKvUnroll];
        uint16_t *dst[kKvUnroll];
#pragma unroll
        for (int u = 0; u < kKvUnroll; ++u) {
            const int i = i0 + u * kKvThreads;
            dst[u] = nullptr;
            if (i < total) {
                const int s = i / (a.Hkv * vpr);
                const int g = (i / vpr) % a.Hkv;
                const int v = i % vpr;
                const uint16_t *src = sb + s * a.bs[1] + g * a.bs[2] + 8 * v;
                dst[u] = db + g * a.cs[1] + static_cast<int64_t>(L + s) * a.cs[2] + 8 * v;
                val[u] = __ldcs(reinterpret_cast<const uint4 *>(src));
            }
        }
#pragma unroll
        for (int u = 0; u < kKvUnroll; ++u)
            if (dst[u]) *reinterpret_cast<uint4 *>(dst[u]) = val[u];
    }
}

__global__ void __launch_bounds__(kLenThreads) kv_len_kernel(const KvArgs a) {
    for (int b = threadIdx.x; b < a.B; b += kLenThreads) {
        const int L = a.lens[b];
        if (takes_part(a, b, L)) {
            a.lens[b] = L + a.S;
        } else if ((a.active == nullptr || a.active[b] != 0) && a.overflow) {
            atomicAdd(a.overflow, 1);
        }
    }
}

tt_status validate_kv(const tt_kv_desc *d, const char *fn) {
    if (!d) return fail(TT_ERR_INVALID_ARG, "%s: null desc", fn);
    if (d->B < 0 || d->B > 65535 || d->S < 1 || d->Hkv < 1 || d->Lmax < 0)
        return fail(TT_ERR_INVALID_ARG, "%s: bad shape B=%d S=%d Hkv=%d Lmax=%d", fn, d->B, d->S,
                    d->Hkv, d->Lmax);
    if (d->d < 8 || d->d > 512 || d->d % 8 != 0)
        return fail(TT_ERR_UNSUPPORTED, "%s: d=%d (a multiple of 8, at most 512)", fn, d->d);
    if (d->n_layers < 1 || d->n_layers > TT_KV_MAX_LAYERS)
        return fail(TT_ERR_INVALID_ARG, "%s: n_layers=%d (1..%d)", fn, d->n_layers,
                    TT_KV_MAX_LAYERS);
    const int64_t *st[2] = {d->ctx_strides, d->blk_strides};
    for (int i = 0; i < 2; ++i) {
        if (st[i][3] != 1) return fail(TT_ERR_UNSUPPORTED, "%s: innermost stride must be 1", fn);
        for (int j = 0; j < 3; ++j)
            if (st[i][j] <= 0 || st[i][j] % 8 != 0)
                return fail(TT_ERR_UNSUPPORTED,
                            "%s: strides must be positive multiples of 8 elements", fn);
    }
    const int64_t per_seq = static_cast<int64_t>(d->n_layers) * 2 * d->S * d->Hkv * (d->d / 8);
    if (per_seq >= (int64_t(1) << 31)) return fail(TT_ERR_UNSUPPORTED, "%s: block too large", fn);
    return TT_OK;
}

}  // namespace
}  // namespace tt

extern "C" tt_status tt_kv_append(const tt_kv_desc *desc, void *const *k_ctx, void *const *v_ctx,
                                  int32_t *ctx_lens, const void *const *k_blk,
                                  const void *const *v_blk, const uint8_t *active,
                                  int32_t *overflow, tt_stream_t stream) {
    using namespace tt;
    const char *fn = "tt_kv_append";
    tt_status st = validate_kv(desc, fn);
    if (st != TT_OK) return st;
    if (desc->B == 0) return TT_OK;
    if (!k_ctx || !v_ctx || !k_blk || !v_blk || !ctx_lens)
        return fail(TT_ERR_INVALID_ARG, "%s: null pointer", fn);
    KvArgs a;
    for (int l = 0; l < desc->n_layers; ++l) {
        const void *p[4] = {k_ctx[l], v_ctx[l], k_blk[l], v_blk[l]};
        for (int i = 0; i < 4; ++i) {
            if (!p[i]) return fail(TT_ERR_INVALID_ARG, "%s: null pointer for layer %d", fn, l);
            if (reinterpret_cast<uintptr_t>(p[i]) % 16)
                return fail(TT_ERR_INVALID_ARG, "%s: layer %d pointer not 16-byte aligned", fn, l);
        }
        a.kc[l] = static_cast<uint16_t *>(k_ctx[l]);
        a.vc[l] = static_cast<uint16_t *>(v_ctx[l]);
        a.kb[l] = static_cast<const uint16_t *>(k_blk[l]);
        a.vb[l] = static_cast<const uint16_t *>(v_blk[l]);
    }
    for (int l = desc->n_layers; l < TT_KV_MAX_LAYERS; ++l) {
        a.kc[l] = a.vc[l] = nullptr;
        a.kb[l] = a.vb[l] = nullptr;
    }
    for (int j = 0; j < 3; ++j) {
        a.cs[j] = desc->ctx_strides[j];
        a.bs[j] = desc->blk_strides[j];
    }
    a.S = desc->S;
    a.Hkv = desc->Hkv;
    a.d = desc->d;
    a.Lmax = desc->Lmax;
    a.nl = desc->n_layers;
    a.B = desc->B;
    a.lens = ctx_lens;
    a.active = active;
    a.overflow = overflow;
    const cudaStream_t st_ = static_cast<cudaStream_t>(stream);
    kv_copy_kernel<<<dim3(2 * desc->n_layers, desc->B), kKvThreads, 0, st_>>>(a);
    tt_status s2 = cuda_status(cudaGetLastError(), "tt_kv_append copy launch");
    if (s2 != TT_OK) return s2;
    kv_len_kernel<<<1, kLenThreads, 0, st_>>>(a);
    return cuda_status(cudaGetLastError(), "tt_kv_append length launch");
}
