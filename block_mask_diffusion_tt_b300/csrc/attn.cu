// attn.cu -- block-query attention of one denoiser attention layer.
//
// Method (dothoosh.com "فرآیند انتشار در برابر رمزگشایی متوالی در مدل جدید انویدیا",
// section "two-tower mechanism"; aitrends.kr "Nemotron-Labs-TwoTower-30B-A3B-Base-BF16",
// section "technical features"): the S block queries of denoiser layer i attend,
// through one softmax, to context-tower layer i's K/V of the committed prefix
// followed by the block's own S keys; every block query sees every block key.
// Grouped-query heads: query head h reads KV head h / (Hq/Hkv).
//
// Work decomposition (all on the device, from ctx_lens):
//  * a "pair" is (sequence b, KV head g, row group rg): the R = S*Hq/Hkv query
//    rows (s, h in group g) that share one K/V stream, cut into groups of 256;
//  * pair p owns ceil(L_b/64) context tiles of 64 keys plus one block tile;
//  * all tiles of all pairs are laid end to end and cut into P equal ranges, one
//    per CTA (P = min(#SMs, tiles/kMinTiles)); a CTA walks its range pair by pair;
//  * a pair whose tiles fall in one CTA is finished in registers; otherwise each
//    CTA writes an fp32 partial (O, running max m, sum l) and the last CTA to
//    arrive (per-pair counter) merges them: M = max m_c,
//    O = sum 2^(m_c-M) O_c / sum 2^(m_c-M) l_c.  No CTA waits on another.
//
// Per tile: Q K^T and P V on the tensor cores (bf16 mma.sync m16n8k16, fp32
// accumulate), online softmax in the exp2 domain, K/V staged in shared memory
// through a 3-stage cp.async ring with zero fill for keys past the prefix.
#include <math.h>

#include <mutex>

#include "common.cuh"

namespace tt {
namespace {

constexpr int kRows = 256;   // query rows per pair
constexpr int kWarps = 16;   // 16 rows per warp
constexpr int kThreads = kWarps * 32;
constexpr int kTN = 64;      // keys per tile
constexpr int kStages = 3;
constexpr int kMaxPairs = 4096;
constexpr int kMinTiles = 4;  // smallest tile range worth a partial
constexpr float kLn2 = 0.69314718055994531f;

struct AttnArgs {
    const uint16_t *q, *kctx, *vctx, *kblk, *vblk;
    uint16_t *out;
    float *lse;
    int64_t qs[4], kcs[4], vcs[4], kbs[4], vbs[4], os[4];
    const int32_t *lens;
    int B, S, Hq, Hkv, G, Lmax, R, NRG, npairs, P;
    float scale_log2;
    float *part_o;    // [slots][256][D]
    float2 *part_ml;  // [slots][256]
    unsigned *pair_cnt;
};

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
    const int n = valid ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// CTA (of P) whose tile range holds flattened tile t, T tiles in total.
__device__ __forceinline__ int owner_of(int64_t t, int P, int64_t T) {
    return static_cast<int>(((t + 1) * P - 1) / T);
}

struct PairInfo {
    int b, g, rg, L, nctx_tiles, rows;
};

__device__ __forceinline__ PairInfo pair_info(const AttnArgs &a, int p) {
    PairInfo pi;
    pi.rg = p % a.NRG;
    const int bg = p / a.NRG;
    pi.g = bg % a.Hkv;
    pi.b = bg / a.Hkv;
    int L = a.lens[pi.b];
    pi.L = L < 0 ? 0 : (L > a.Lmax ? a.Lmax : L);
    pi.nctx_tiles = (pi.L + kTN - 1) / kTN;
    pi.rows = min(kRows, a.R - pi.rg * kRows);
    return pi;
}

template <int D>
struct Layout {
    static constexpr int kStride = D + 8;  // bf16 elements per smem row (conflict-free ldmatrix)
    static constexpr int kQBytes = kRows * kStride * 2;
    static constexpr int kTileBytes = kTN * kStride * 2;
    static constexpr int kStageBytes = 2 * kTileBytes;  // K then V
    static constexpr int kBytes = kQBytes + kStages * kStageBytes;
};

// Enqueues the cp.async copies of tile `tile` of pair `pi` into stage memory.
template <int D>
__device__ __forceinline__ void load_tile(const AttnArgs &a, const PairInfo &pi, int tile,
                                          uint16_t *ks, uint16_t *vs) {
    constexpr int kChunks = D / 8;  // 16-byte chunks per row
    const bool block_tile = tile == pi.nctx_tiles;
    const int nvalid = block_tile ? a.S : min(kTN, pi.L - tile * kTN);
    for (int i = threadIdx.x; i < kTN * kChunks; i += kThreads) {
        const int j = i / kChunks, ch = i % kChunks;
        const bool valid = j < nvalid;
        const uint16_t *ksrc, *vsrc;
        if (block_tile) {
            const int jj = valid ? j : 0;
            ksrc = a.kblk + pi.b * a.kbs[0] + jj * a.kbs[1] + pi.g * a.kbs[2] + ch * 8;
            vsrc = a.vblk + pi.b * a.vbs[0] + jj * a.vbs[1] + pi.g * a.vbs[2] + ch * 8;
        } else {
            const int64_t key = valid ? static_cast<int64_t>(tile) * kTN + j : 0;
            ksrc = a.kctx + pi.b * a.kcs[0] + pi.g * a.kcs[1] + key * a.kcs[2] + ch * 8;
            vsrc = a.vctx + pi.b * a.vcs[0] + pi.g * a.vcs[1] + key * a.vcs[2] + ch * 8;
        }
        const int off = j * Layout<D>::kStride + ch * 8;
        cp_async16(smem_u32(ks + off), ksrc, valid);
        cp_async16(smem_u32(vs + off), vsrc, valid);
    }
}

template <int D>
__device__ __forceinline__ void load_q(const AttnArgs &a, const PairInfo &pi, uint16_t *qs) {
    constexpr int kChunks = D / 8;
    for (int i = threadIdx.x; i < kRows * kChunks; i += kThreads) {
        const int r = i / kChunks, ch = i % kChunks;
        const bool valid = r < pi.rows;
        const int rr = pi.rg * kRows + (valid ? r : 0);
        const int s = rr / a.G, h = pi.g * a.G + rr % a.G;
        const uint16_t *src = a.q + pi.b * a.qs[0] + s * a.qs[1] + h * a.qs[2] + ch * 8;
        cp_async16(smem_u32(qs + r * Layout<D>::kStride + ch * 8), src, valid);
    }
}

// Writes one finished row pair (rows g and g+8 of the warp) for a single-part pair.
template <int D>
__device__ __forceinline__ void store_rows(const AttnArgs &a, const PairInfo &pi, int row,
                                           const float (&o)[D / 8][4], int half, float inv_l,
                                           float m, float l) {
    if (row >= pi.rows) return;
    const int rr = pi.rg * kRows + row;
    const int s = rr / a.G, h = pi.g * a.G + rr % a.G;
    const int c = threadIdx.x & 3;
    uint16_t *dst = a.out + pi.b * a.os[0] + s * a.os[1] + h * a.os[2];
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) {
        const uint32_t v = pack_bf16x2(o[nt][2 * half] * inv_l, o[nt][2 * half + 1] * inv_l);
        *reinterpret_cast<uint32_t *>(dst + nt * 8 + 2 * c) = v;
    }
    if (a.lse && c == 0)
        a.lse[(static_cast<int64_t>(pi.b) * a.Hq + h) * a.S + s] = (m + __log2f(l)) * kLn2;
}

template <int D>
__device__ void merge_pair(const AttnArgs &a, const PairInfo &pi, int p, int c_first, int c_last) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int kPer = D / 32;  // columns per lane
    for (int r = warp; r < pi.rows; r += kWarps) {
        float M = -INFINITY;
        for (int c = c_first; c <= c_last; ++c) {
            const float2 ml = __ldcg(a.part_ml + static_cast<size_t>(c + p) * kRows + r);
            M = fmaxf(M, ml.x);
        }
        float den = 0.f, acc[kPer];
#pragma unroll
        for (int j = 0; j < kPer; ++j) acc[j] = 0.f;
        for (int c = c_first; c <= c_last; ++c) {
            const size_t slot = static_cast<size_t>(c + p);
            const float2 ml = __ldcg(a.part_ml + slot * kRows + r);
            const float w = ex2_approx(ml.x - M);
            den += w * ml.y;
            const float *src = a.part_o + (slot * kRows + r) * D + lane * kPer;
            if constexpr (kPer == 4) {
                const float4 v = __ldcg(reinterpret_cast<const float4 *>(src));
                acc[0] += w * v.x; acc[1] += w * v.y; acc[2] += w * v.z; acc[3] += w * v.w;
            } else {
                const float2 v = __ldcg(reinterpret_cast<const float2 *>(src));
                acc[0] += w * v.x; acc[1] += w * v.y;
            }
        }
        const float inv = 1.f / den;
        const int rr = pi.rg * kRows + r;
        const int s = rr / a.G, h = pi.g * a.G + rr % a.G;
        uint16_t *dst = a.out + pi.b * a.os[0] + s * a.os[1] + h * a.os[2] + lane * kPer;
        if constexpr (kPer == 4) {
            uint2 v;
            v.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
            v.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
            *reinterpret_cast<uint2 *>(dst) = v;
        } else {
            *reinterpret_cast<uint32_t *>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
        }
        if (a.lse && lane == 0)
            a.lse[(static_cast<int64_t>(pi.b) * a.Hq + h) * a.S + s] = (M + __log2f(den)) * kLn2;
    }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) block_attn_mma_kernel(const AttnArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    uint16_t *qs = reinterpret_cast<uint16_t *>(smem);
    uint16_t *stage0 = reinterpret_cast<uint16_t *>(smem + Layout<D>::kQBytes);
    int *prefix = reinterpret_cast<int *>(smem + Layout<D>::kBytes);  // [npairs + 1]
    __shared__ int warp_sums[kWarps];
    __shared__ int is_last;

    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;

    // ---- tile counts per pair and their exclusive prefix sum
    {
        const int per = (a.npairs + kThreads - 1) / kThreads;
        const int p0 = min(a.npairs, t * per), p1 = min(a.npairs, p0 + per);
        int local = 0;
        for (int p = p0; p < p1; ++p) {
            int L = a.lens[p / (a.Hkv * a.NRG)];
            L = L < 0 ? 0 : (L > a.Lmax ? a.Lmax : L);
            local += (L + kTN - 1) / kTN + 1;
        }
        int incl = local;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(0xFFFFFFFFu, incl, off);
            if (lane >= off) incl += v;
        }
        if (lane == 31) warp_sums[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            int w = lane < kWarps ? warp_sums[lane] : 0;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int v = __shfl_up_sync(0xFFFFFFFFu, w, off);
                if (lane >= off) w += v;
            }
            if (lane < kWarps) warp_sums[lane] = w;  // inclusive warp totals
        }
        __syncthreads();
        int run = incl - local + (warp > 0 ? warp_sums[warp - 1] : 0);
        for (int p = p0; p < p1; ++p) {
            prefix[p] = run;
            int L = a.lens[p / (a.Hkv * a.NRG)];
            L = L < 0 ? 0 : (L > a.Lmax ? a.Lmax : L);
            run += (L + kTN - 1) / kTN + 1;
        }
        if (t == kThreads - 1) prefix[a.npairs] = run;
        __syncthreads();
    }
    const int64_t T = prefix[a.npairs];
    int64_t parts = T / kMinTiles;
    parts = parts < 1 ? 1 : (parts > a.P ? a.P : parts);
    const int P = static_cast<int>(parts);
    const int cta = blockIdx.x;
    if (cta >= P) return;
    const int64_t t_begin = static_cast<int64_t>(cta) * T / P;
    const int64_t t_end = static_cast<int64_t>(cta + 1) * T / P;

    const int g8 = lane >> 2, c4 = lane & 3;
    const int row0 = warp * 16;

    for (int64_t tcur = t_begin; tcur < t_end;) {
        // pair holding tile tcur: last p with prefix[p] <= tcur
        int lo = 0, hi = a.npairs;  // invariant: prefix[lo] <= tcur < prefix[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (prefix[mid] <= tcur) lo = mid; else hi = mid;
        }
        const int p = lo;
        const int64_t ps = prefix[p], pe = prefix[p + 1];
        const int64_t seg_end = min(t_end, pe);
        const PairInfo pi = pair_info(a, p);
        const int tile0 = static_cast<int>(tcur - ps), ntiles = static_cast<int>(seg_end - tcur);
        const int c_first = owner_of(ps, P, T), c_last = owner_of(pe - 1, P, T);

        // ---- pipeline prologue: Q, then the first kStages-1 tiles
        load_q<D>(a, pi, qs);
        cp_async_commit();
#pragma unroll
        for (int st = 0; st < kStages - 1; ++st) {
            if (st < ntiles) {
                uint16_t *ks = stage0 + st * (Layout<D>::kStageBytes / 2);
                load_tile<D>(a, pi, tile0 + st, ks, ks + Layout<D>::kTileBytes / 2);
            }
            cp_async_commit();
        }

        float o[D / 8][4];
#pragma unroll
        for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
        float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};

        for (int it = 0; it < ntiles; ++it) {
            cp_async_wait<kStages - 2>();
            __syncthreads();
            {  // refill the stage freed by the previous tile
                const int nt_load = it + kStages - 1;
                if (nt_load < ntiles) {
                    uint16_t *ks = stage0 + (nt_load % kStages) * (Layout<D>::kStageBytes / 2);
                    load_tile<D>(a, pi, tile0 + nt_load, ks, ks + Layout<D>::kTileBytes / 2);
                }
                cp_async_commit();
            }
            const uint16_t *ks = stage0 + (it % kStages) * (Layout<D>::kStageBytes / 2);
            const uint16_t *vs = ks + Layout<D>::kTileBytes / 2;
            const int tile = tile0 + it;
            const bool block_tile = tile == pi.nctx_tiles;
            const int nvalid = block_tile ? a.S : min(kTN, pi.L - tile * kTN);

            // S = Q K^T for this warp's 16 rows x 64 keys
            float sc[kTN / 8][4];
#pragma unroll
            for (int i = 0; i < kTN / 8; ++i) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                uint32_t af[4];
                {
                    const int mi = lane >> 3;
                    const int r = row0 + (mi & 1) * 8 + (lane & 7);
                    const int col = kk * 16 + (mi >> 1) * 8;
                    ldsm_x4(smem_u32(qs + r * Layout<D>::kStride + col), af);
                }
#pragma unroll
                for (int np = 0; np < kTN / 16; ++np) {
                    uint32_t bf[4];
                    const int mi = lane >> 3;
                    const int key = np * 16 + (mi >> 1) * 8 + (lane & 7);
                    const int col = kk * 16 + (mi & 1) * 8;
                    ldsm_x4(smem_u32(ks + key * Layout<D>::kStride + col), bf);
                    mma_bf16(sc[2 * np], af, bf[0], bf[1]);
                    mma_bf16(sc[2 * np + 1], af, bf[2], bf[3]);
                }
            }
            // online softmax (exp2 domain), two rows per thread: g8 and g8+8
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                float mx = -INFINITY;
#pragma unroll
                for (int nt = 0; nt < kTN / 8; ++nt) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int key = nt * 8 + 2 * c4 + e;
                        float x = sc[nt][2 * hr + e] * a.scale_log2;
                        x = key < nvalid ? x : -INFINITY;
                        sc[nt][2 * hr + e] = x;
                        mx = fmaxf(mx, x);
                    }
                }
                mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
                const float mnew = fmaxf(m[hr], mx);
                const float corr = ex2_approx(m[hr] - mnew);
                m[hr] = mnew;
                l[hr] *= corr;
#pragma unroll
                for (int i = 0; i < D / 8; ++i) {
                    o[i][2 * hr] *= corr;
                    o[i][2 * hr + 1] *= corr;
                }
                float ls = 0.f;
#pragma unroll
                for (int nt = 0; nt < kTN / 8; ++nt) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float pv = ex2_approx(sc[nt][2 * hr + e] - mnew);
                        sc[nt][2 * hr + e] = pv;
                        ls += pv;
                    }
                }
                l[hr] += ls;
            }
            // O += P V
#pragma unroll
            for (int j = 0; j < kTN / 16; ++j) {
                uint32_t pf[4];
                pf[0] = pack_bf16x2(sc[2 * j][0], sc[2 * j][1]);
                pf[1] = pack_bf16x2(sc[2 * j][2], sc[2 * j][3]);
                pf[2] = pack_bf16x2(sc[2 * j + 1][0], sc[2 * j + 1][1]);
                pf[3] = pack_bf16x2(sc[2 * j + 1][2], sc[2 * j + 1][3]);
#pragma unroll
                for (int dp = 0; dp < D / 16; ++dp) {
                    uint32_t bf[4];
                    const int mi = lane >> 3;
                    const int key = j * 16 + (mi & 1) * 8 + (lane & 7);
                    const int col = dp * 16 + (mi >> 1) * 8;
                    ldsm_x4_t(smem_u32(vs + key * Layout<D>::kStride + col), bf);
                    mma_bf16(o[2 * dp], pf, bf[0], bf[1]);
                    mma_bf16(o[2 * dp + 1], pf, bf[2], bf[3]);
                }
            }
        }
        cp_async_wait<0>();
        __syncthreads();  // stages and Q are free for the next segment

#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            l[hr] += __shfl_xor_sync(0xFFFFFFFFu, l[hr], 1);
            l[hr] += __shfl_xor_sync(0xFFFFFFFFu, l[hr], 2);
        }
        if (c_first == c_last) {
#pragma unroll
            for (int hr = 0; hr < 2; ++hr)
                store_rows<D>(a, pi, row0 + g8 + 8 * hr, o, hr, 1.f / l[hr], m[hr], l[hr]);
        } else {
            const size_t slot = static_cast<size_t>(cta + p);
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int r = row0 + g8 + 8 * hr;
                float *dst = a.part_o + (slot * kRows + r) * D;
#pragma unroll
                for (int nt = 0; nt < D / 8; ++nt)
                    *reinterpret_cast<float2 *>(dst + nt * 8 + 2 * c4) =
                        make_float2(o[nt][2 * hr], o[nt][2 * hr + 1]);
                if (c4 == 0) a.part_ml[slot * kRows + r] = make_float2(m[hr], l[hr]);
            }
            __syncthreads();
            if (t == 0) {
                __threadfence();
                const unsigned old = atomicAdd(a.pair_cnt + p, 1u);
                is_last = old == static_cast<unsigned>(c_last - c_first);
                if (is_last) __threadfence();
            }
            __syncthreads();
            if (is_last) {
                merge_pair<D>(a, pi, p, c_first, c_last);
                if (t == 0) a.pair_cnt[p] = 0;
            }
        }
        tcur = seg_end;
    }
}

// ---------------------------------------------------------------- host
struct Geometry {
    int G, R, NRG, npairs, P;
};

tt_status validate(const tt_attn_desc *d, Geometry *geo, const char *fn) {
    if (!d) return fail(TT_ERR_INVALID_ARG, "%s: null desc", fn);
    if (d->B < 0 || d->S < 1 || d->Hq < 1 || d->Hkv < 1 || d->Lmax < 0)
        return fail(TT_ERR_INVALID_ARG, "%s: bad shape B=%d S=%d Hq=%d Hkv=%d Lmax=%d", fn, d->B,
                    d->S, d->Hq, d->Hkv, d->Lmax);
    if (d->Hq % d->Hkv != 0) return fail(TT_ERR_INVALID_ARG, "%s: Hq %% Hkv != 0", fn);
    if (d->d != 64 && d->d != 128) return fail(TT_ERR_UNSUPPORTED, "%s: d=%d (64 or 128)", fn, d->d);
    if (d->S > 64) return fail(TT_ERR_UNSUPPORTED, "%s: S=%d > 64", fn, d->S);
    if (isnan(d->scale) || isinf(d->scale)) return fail(TT_ERR_INVALID_ARG, "%s: bad scale", fn);
    const int64_t *st[6] = {d->q_strides, d->kctx_strides, d->vctx_strides, d->kblk_strides,
                            d->vblk_strides, d->o_strides};
    for (int i = 0; i < 6; ++i) {
        if (st[i][3] != 1) return fail(TT_ERR_UNSUPPORTED, "%s: innermost stride must be 1", fn);
        for (int j = 0; j < 3; ++j)
            if (st[i][j] <= 0 || st[i][j] % 8 != 0)
                return fail(TT_ERR_UNSUPPORTED,
                            "%s: strides must be positive multiples of 8 elements", fn);
    }
    geo->G = d->Hq / d->Hkv;
    geo->R = d->S * geo->G;
    geo->NRG = (geo->R + kRows - 1) / kRows;
    const int64_t np = static_cast<int64_t>(d->B) * d->Hkv * geo->NRG;
    if (np > kMaxPairs)
        return fail(TT_ERR_UNSUPPORTED, "%s: B*Hkv*ceil(S*Hq/Hkv/256) = %lld > %d", fn,
                    (long long)np, kMaxPairs);
    geo->npairs = static_cast<int>(np);
    geo->P = sm_count();
    if (geo->P <= 0) return fail(TT_ERR_CUDA, "%s: no CUDA device", fn);
    return TT_OK;
}

struct AttnWs {
    unsigned *pair_cnt;
    float2 *part_ml;
    float *part_o;
    size_t bytes;
};

AttnWs carve_attn(void *ws, const tt_attn_desc *d, const Geometry &g) {
    Carve c(ws);
    AttnWs w;
    const size_t slots = static_cast<size_t>(g.P) + g.npairs;
    w.pair_cnt = c.take<unsigned>(static_cast<size_t>(g.npairs));
    w.part_ml = c.take<float2>(slots * kRows);
    w.part_o = c.take<float>(slots * kRows * d->d);
    w.bytes = c.bytes();
    return w;
}

template <int D>
tt_status launch(const AttnArgs &a, int smem_bytes, cudaStream_t stream) {
    static bool configured[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(block_attn_mma_kernel<D>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             smem_bytes > 200 * 1024 ? smem_bytes : 200 * 1024);
        if (e != cudaSuccess) return cuda_status(e, "tt_block_attn: smem attribute");
        configured[dev] = true;
    }
    block_attn_mma_kernel<D><<<a.P, kThreads, smem_bytes, stream>>>(a);
    return cuda_status(cudaGetLastError(), "tt_block_attn launch");
}

}  // namespace
}  // namespace tt

using namespace tt;

extern "C" {

size_t tt_block_attn_workspace_size(const tt_attn_desc *d) {
    Geometry g;
    if (validate(d, &g, "tt_block_attn_workspace_size") != TT_OK) return 0;
    return carve_attn(nullptr, d, g).bytes;
}

tt_status tt_block_attn(const tt_attn_desc *d, const void *q, const void *k_ctx, const void *v_ctx,
                        const int32_t *ctx_lens, const void *k_blk, const void *v_blk, void *out,
                        float *lse, void *workspace, size_t workspace_bytes, tt_stream_t stream) {
    const char *fn = "tt_block_attn";
    Geometry g;
    tt_status st = validate(d, &g, fn);
    if (st != TT_OK) return st;
    if (d->B == 0) return TT_OK;
    if (!q || !k_blk || !v_blk || !out || !ctx_lens || (d->Lmax > 0 && (!k_ctx || !v_ctx)))
        return fail(TT_ERR_INVALID_ARG, "%s: null pointer", fn);
    const void *ptrs[6] = {q, k_ctx, v_ctx, k_blk, v_blk, out};
    for (int i = 0; i < 6; ++i)
        if (reinterpret_cast<uintptr_t>(ptrs[i]) % 16)
            return fail(TT_ERR_INVALID_ARG, "%s: tensor base not 16-byte aligned", fn);
    if (reinterpret_cast<uintptr_t>(ctx_lens) % 4 || (lse && reinterpret_cast<uintptr_t>(lse) % 4))
        return fail(TT_ERR_INVALID_ARG, "%s: ctx_lens/lse misaligned", fn);
    AttnWs w = carve_attn(workspace, d, g);
    if (!workspace || workspace_bytes < w.bytes)
        return fail(TT_ERR_WORKSPACE, "%s: workspace of %zu bytes, %zu needed", fn, workspace_bytes,
                    w.bytes);
    if (reinterpret_cast<uintptr_t>(workspace) % 256)
        return fail(TT_ERR_WORKSPACE, "%s: workspace not 256-byte aligned", fn);

    AttnArgs a;
    a.q = static_cast<const uint16_t *>(q);
    a.kctx = static_cast<const uint16_t *>(k_ctx ? k_ctx : q);
    a.vctx = static_cast<const uint16_t *>(v_ctx ? v_ctx : q);
    a.kblk = static_cast<const uint16_t *>(k_blk);
    a.vblk = static_cast<const uint16_t *>(v_blk);
    a.out = static_cast<uint16_t *>(out);
    a.lse = lse;
    for (int i = 0; i < 4; ++i) {
        a.qs[i] = d->q_strides[i];
        a.kcs[i] = d->kctx_strides[i];
        a.vcs[i] = d->vctx_strides[i];
        a.kbs[i] = d->kblk_strides[i];
        a.vbs[i] = d->vblk_strides[i];
        a.os[i] = d->o_strides[i];
    }
    a.lens = ctx_lens;
    a.B = d->B;
    a.S = d->S;
    a.Hq = d->Hq;
    a.Hkv = d->Hkv;
    a.G = g.G;
    a.Lmax = d->Lmax;
    a.R = g.R;
    a.NRG = g.NRG;
    a.npairs = g.npairs;
    a.P = g.P;
    const double scale = d->scale > 0.f ? d->scale : 1.0 / sqrt(static_cast<double>(d->d));
    a.scale_log2 = static_cast<float>(scale * 1.4426950408889634);
    a.part_o = w.part_o;
    a.part_ml = w.part_ml;
    a.pair_cnt = w.pair_cnt;
    const int extra = (g.npairs + 1) * static_cast<int>(sizeof(int));
    if (d->d == 128) return launch<128>(a, Layout<128>::kBytes + extra, (cudaStream_t)stream);
    return launch<64>(a, Layout<64>::kBytes + extra, (cudaStream_t)stream);
}

}  // extern "C"

// ---------------------------------------------------------------- no-allocation variant
// Scratch of tt_block_attn_noalloc: a fixed device array in this module, present
// on every device that loads the library for as long as the process lives.
namespace tt {
namespace {

constexpr size_t kStaticScratchBytes = size_t(32) << 20;  // 32 MiB per device
static __device__ __align__(256) unsigned char g_attn_static_scratch[kStaticScratchBytes];

std::mutex g_static_mu;
void *g_static_ptr[64] = {nullptr};  // device address of the array, per device

// Device address of the static scratch on the current device.  The first call on
// a device resolves it with cudaGetSymbolAddress (the array's name is only a host
// stand-in in host code).
tt_status static_scratch(void **out, const char *fn) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_status(e, fn);
    if (dev < 0 || dev >= 64) return fail(TT_ERR_UNSUPPORTED, "%s: device index %d >= 64", fn, dev);
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (!g_static_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_attn_static_scratch);
        if (e != cudaSuccess) return cuda_status(e, "cudaGetSymbolAddress(static scratch)");
        g_static_ptr[dev] = p;
    }
    *out = g_static_ptr[dev];
    return TT_OK;
}

// Layout of the static scratch for `slots` partial slots.
AttnWs carve_static(void *base, int npairs, size_t slots, int d) {
    Carve c(base);
    AttnWs w;
    w.pair_cnt = c.take<unsigned>(static_cast<size_t>(npairs));
    w.part_ml = c.take<float2>(slots * kRows);
    w.part_o = c.take<float>(slots * kRows * d);
    w.bytes = c.bytes();
    return w;
}

}  // namespace
}  // namespace tt

extern "C" tt_status tt_block_attn_noalloc(const tt_attn_desc *d, const void *q,
                                           const void *k_ctx, const void *v_ctx,
                                           const int32_t *ctx_lens, const void *k_blk,
                                           const void *v_blk, void *out, float *lse,
                                           tt_stream_t stream) {
    using namespace tt;
    const char *fn = "tt_block_attn_noalloc";
    Geometry g;
    tt_status st = validate(d, &g, fn);
    if (st != TT_OK) return st;
    if (d->B == 0) return TT_OK;
    if (!q || !k_blk || !v_blk || !out || !ctx_lens || (d->Lmax > 0 && (!k_ctx || !v_ctx)))
        return fail(TT_ERR_INVALID_ARG, "%s: null pointer", fn);
    const void *ptrs[6] = {q, k_ctx, v_ctx, k_blk, v_blk, out};
    for (int i = 0; i < 6; ++i)
        if (reinterpret_cast<uintptr_t>(ptrs[i]) % 16)
            return fail(TT_ERR_INVALID_ARG, "%s: tensor base not 16-byte aligned", fn);
    if (reinterpret_cast<uintptr_t>(ctx_lens) % 4 || (lse && reinterpret_cast<uintptr_t>(lse) % 4))
        return fail(TT_ERR_INVALID_ARG, "%s: ctx_lens/lse misaligned", fn);
    // slots that fit: one per pair plus at least one partition
    const size_t per_slot = carve_static(nullptr, 0, 1, d->d).bytes;
    size_t slots = kStaticScratchBytes / per_slot;
    while (slots > 0 && carve_static(nullptr, g.npairs, slots, d->d).bytes > kStaticScratchBytes)
        --slots;
    if (slots < static_cast<size_t>(g.npairs) + 1)
        return fail(TT_ERR_UNSUPPORTED,
                    "%s: B*Hkv*ceil(S*Hq/Hkv/256) = %d pairs need more than the %zu-byte static "
                    "scratch (at most %zu pairs at d=%d); use tt_block_attn with a workspace",
                    fn, g.npairs, kStaticScratchBytes, slots > 0 ? slots - 1 : 0, d->d);
    const size_t parts = slots - g.npairs;
    if (static_cast<size_t>(g.P) > parts) g.P = static_cast<int>(parts);
    void *base = nullptr;
    if ((st = static_scratch(&base, fn)) != TT_OK) return st;
    AttnWs w = carve_static(base, g.npairs, static_cast<size_t>(g.P) + g.npairs, d->d);
    // the arrival counters must start at zero whatever an earlier call left behind
    st = cuda_status(cudaMemsetAsync(w.pair_cnt, 0, sizeof(unsigned) * g.npairs,
                                     (cudaStream_t)stream), fn);
    if (st != TT_OK) return st;

    AttnArgs a;
    a.q = static_cast<const uint16_t *>(q);
    a.kctx = static_cast<const uint16_t *>(k_ctx ? k_ctx : q);
    a.vctx = static_cast<const uint16_t *>(v_ctx ? v_ctx : q);
    a.kblk = static_cast<const uint16_t *>(k_blk);
    a.vblk = static_cast<const uint16_t *>(v_blk);
    a.out = static_cast<uint16_t *>(out);
    a.lse = lse;
    for (int i = 0; i < 4; ++i) {
        a.qs[i] = d->q_strides[i];
        a.kcs[i] = d->kctx_strides[i];
        a.vcs[i] = d->vctx_strides[i];
        a.kbs[i] = d->kblk_strides[i];
        a.vbs[i] = d->vblk_strides[i];
        a.os[i] = d->o_strides[i];
    }
    a.lens = ctx_lens;
    a.B = d->B;
    a.S = d->S;
    a.Hq = d->Hq;
    a.Hkv = d->Hkv;
    a.G = g.G;
    a.Lmax = d->Lmax;
    a.R = g.R;
    a.NRG = g.NRG;
    a.npairs = g.npairs;
    a.P = g.P;
    const double scale = d->scale > 0.f ? d->scale : 1.0 / sqrt(static_cast<double>(d->d));
    a.scale_log2 = static_cast<float>(scale * 1.4426950408889634);
    a.part_o = w.part_o;
    a.part_ml = w.part_ml;
    a.pair_cnt = w.pair_cnt;
    const int extra = (g.npairs + 1) * static_cast<int>(sizeof(int));
    if (d->d == 128) return launch<128>(a, Layout<128>::kBytes + extra, (cudaStream_t)stream);
    return launch<64>(a, Layout<64>::kBytes + extra, (cudaStream_t)stream);
}
