// attn.cu -- block-query attention of one denoiser attention layer on sm_103a
// (tcgen05 tensor cores with TMEM accumulators, TMA-staged K/V).
//
// Method (dothoosh.com "فرآیند انتشار در برابر رمزگشایی متوالی در مدل جدید انویدیا",
// section "two-tower mechanism"; aitrends.kr "Nemotron-Labs-TwoTower-30B-A3B-Base-BF16",
// section "technical features"): the S block queries of denoiser layer i attend,
// through one softmax, to context-tower layer i's K/V of the committed prefix
// followed by the block's own S keys; every block query sees every block key.
// Grouped-query heads: query head h reads KV head h / (Hq/Hkv).
//
// Work decomposition (on the device, from ctx_lens):
//  * a "pair" is (sequence b, KV head g, row group rg): the R = S*Hq/Hkv query
//    rows (s, h in group g) that share one K/V stream, cut into groups of 256;
//    each group runs as two 128-row halves (one tcgen05 M=128 tile each);
//  * pair p owns ceil(L_b/64) context tiles of 64 keys plus one block tile;
//  * the tiles of all pairs are laid end to end and cut into P equal ranges, one
//    per CTA (P = min(#SMs, tiles/4)); a CTA walks its range segment by segment
//    (a segment = the part of one pair inside the range);
//  * a pair whose tiles fall in one CTA is finished there; otherwise each CTA
//    writes an fp32 partial (O / l, running max m, sum l) and a second kernel,
//    launched as a programmatic dependent, merges them: M = max m_c,
//    O = sum 2^(m_c-M) l_c O_c / sum 2^(m_c-M) l_c.  No CTA waits on another.
//
// Inside a CTA (352 threads, one CTA per SM, 512 TMEM columns):
//  warp 8     TMA producer: K and V tiles (64 keys x d, 128-byte swizzle) into a
//             ring of shared-memory stages (full/empty mbarriers);
//  warps 9,10 MMA issuers, one per half: S_h = Q_h K^T (A = Q_h in shared memory,
//             B = K tile, M=128 N=64) into one of two S buffers of the half, then
//             O_h += P_h V (A = P_h in TMEM, B = V tile read MN-major, M=128 N=d);
//             completion via tcgen05.commit;
//  warps 0-7  softmax, warpgroup h owns half h, one query row per thread: reads
//             its S row from TMEM, keeps the running max (in log2 units, raised
//             only when it grows by more than 8, so O is rescaled rarely) and
//             sum, writes P = 2^(x - m) as bf16 pairs over the first 32 columns of
//             the same S buffer, and at the end of a segment reads O, normalises
//             and stores it.
// With two S buffers per half the MMA warp computes the scores of tile j+1 while
// the softmax works on tile j.  An S buffer is rewritten by Q K^T of tile j+2 only
// after P V of tile j, which reads the P stored there, has been issued by the same
// warp; tcgen05 operations of one thread run in issue order.
// TMEM columns (d=128): O_0 O_1 [128 each] | S/P_0 [2 x 64] | S/P_1 [2 x 64].
// Every wait on an mbarrier gives up after 2 s (globaltimer), records a flag in
// the workspace and lets the CTA drain its copies and free TMEM.
#include <cuda.h>
#include <math.h>
#include <string.h>

#include <mutex>

#include "common.cuh"

namespace tt {
namespace {

constexpr int kRows = 256;  // query rows per pair (two halves of 128)
constexpr int kTN = 64;     // keys per tile
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;  // warps 9 and 10: MMA issuers of half 0 and half 1
constexpr int kThreads = 352;
constexpr int kMaxPairs = 4096;
constexpr int kMinTiles = 4;  // smallest tile range worth a partial
// Cost of starting a segment (Q load, pipeline refill, epilogue), in tile units: every
// pair is charged this many extra units at its start when the tile ranges are cut.
// Measured with the first Q by TMA (us per call, default / ragged16k / uniform 16K / long):
// 5 gave 25.8 / 79.6 / 50.5 / 122.3, 7 gave 25.8 / 77.4 / 48.4 / 122.3, 10 gave
// 26.9 / 78.5 / 48.7 / 121.4.
constexpr int kSegCost = 7;
constexpr float kLn2 = 0.69314718055994531f;
constexpr float kRescaleLog2 = 8.f;  // lazy rescale: O is rescaled when the max grows by > 2^8
constexpr int kTmemCols = 512;
// Bits of the workspace error word: a role that gave up on a wait (bit role-1:
// 1 TMA producer, 2 MMA issuer, 4 softmax warps), a context length outside [0, Lmax],
// and a page of a paged cache outside the pool.
constexpr int kErrCtxLen = 8;
constexpr int kErrPage = 16;

template <int D>
struct Cfg {
    static constexpr int kChunks = D / 64;            // 64-column (128-byte) chunks of a row
    static constexpr int kRegionBytes = kTN * 128;    // one chunk of a 64-key tile
    static constexpr int kStageBytes = 2 * kChunks * kRegionBytes;  // K chunks then V chunks
    static constexpr int kStages = D == 128 ? 4 : 6;
    static constexpr int kQRegion = 128 * 128;  // one 64-column chunk of a half's 128 Q rows
    static constexpr int kQHalfBytes = kChunks * kQRegion;
    static constexpr int kQOffset = kStages * kStageBytes;  // Q[half][chunk][128 rows][128 B]
    __host__ __device__ static constexpr uint32_t colO(int h) { return h * D; }
    __host__ __device__ static constexpr uint32_t colS(int h, int b) { return 2 * D + (2 * h + b) * kTN; }
    // instruction descriptors (kind::f16): D fp32, A/B bf16, M=128.  S = Q K^T: A = Q
    // and B = K tile, both K-major, N=64.  O += P V: A = P (TMEM), B = V MN-major, N=d.
    static constexpr uint32_t kIdescQK = (1u << 4) | (1u << 7) | (1u << 10) |
                                         (uint32_t(kTN >> 3) << 17) | (uint32_t(128 >> 4) << 24);
    static constexpr uint32_t kIdescPV = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) |
                                         (uint32_t(D >> 3) << 17) | (uint32_t(128 >> 4) << 24);
    // barriers: full[S] empty[S] s_full[2][2] p_full[2][2] pv_done[2][2]
    //           q_ready[2] fin[2] turn[2] q_tma[2]
    static constexpr int kNumBars = 2 * kStages + 20;
    static constexpr int kBarOffset = kQOffset + 2 * kQHalfBytes;
    static constexpr int kMiscOffset = kBarOffset + kNumBars * 8;  // tmem base, err, last[2]
    static constexpr int kPrefixOffset = kMiscOffset + 16;
    // prefix: int[npairs + 1]; then tail: uint8[npairs] (keys in the last context tile)
    static constexpr int smem_bytes(int npairs) { return 1024 + kPrefixOffset + (npairs + 1) * 4 + npairs; }
    static_assert(2 * D + 4 * kTN <= kTmemCols, "TMEM budget");
};

struct AttnArgs {
    const uint16_t *q;
    uint16_t *out;
    float *lse;
    int64_t qs[4], os[4];
    const int32_t *lens;
    int B, S, Hq, Hkv, G, Lmax, R, NRG, npairs, P;
    float scale_log2;
    float *part_o;    // [slots][D][256], O / l of the CTA's tiles
    float2 *part_ml;  // [slots][256]
    int2 *pair_split;  // [npairs]: first and last CTA of each pair's tile range
    int *err_word;
    int keys;                  // TT_KEYS_ALL / _PREFIX / _BLOCK
    const int32_t *page_of;    // paged cache: [B, max_pages] page of each 64-key tile, or null
    int max_pages, n_pages;
    const float *q_scale;      // modulation: q' = q (1 + scale) + shift, [B, Hq, D] fp32, or null
    const float *q_shift;
    const float *o_gate;       // out = gate * attention, [B, Hq, D] fp32, or null
    int q_tma;                 // the CTA's first segment's Q comes by TMA from the producer
};

// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, int c3, uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar),
        "l"(policy)
        : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Warp-converged issue: every lane of the MMA warp executes these, one elected
// lane (the same one each time) issues the instruction.
__device__ __forceinline__ void tc_mma_ts_e(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void tc_mma_ss_e(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void tc_commit_e(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}\n" ::"r"(
            bar)
        : "memory");
}
// Shared-memory matrix descriptor, 128-byte swizzle (sm_100 format, version 1).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return uint64_t((addr & 0x3FFFFu) >> 4) | (uint64_t(lbo >> 4) << 16) |
           (uint64_t(sbo >> 4) << 32) | (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

#define TT_R32(r)                                                                              \
    "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),       \
        "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), \
        "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]),          \
        "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]),          \
        "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
#define TT_W32(r)                                                                              \
    "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),       \
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), \
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),          \
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),          \
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
#define TT_IN32(r)                                                                             \
    "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),   \
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),      \
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),    \
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),    \
        "r"(r[29]), "r"(r[30]), "r"(r[31])
#define TT_REGLIST32                                                                           \
    "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, "   \
    "%19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}"

// 32 consecutive 32-bit TMEM columns of this thread's lane (shape 32x32b).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t *r) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 " TT_REGLIST32 ", [%32];"
                 : TT_W32(r)
                 : "r"(taddr));
}
// Completes the loads; the registers pass through so no use moves above the wait.
__device__ __forceinline__ void tmem_wait_ld(uint32_t *r) {
    asm volatile("tcgen05.wait::ld.sync.aligned;" : TT_R32(r)::"memory");
}
__device__ __forceinline__ void tmem_touch(uint32_t *r) { asm volatile("" : TT_R32(r)); }
#define TT_REGLIST32_FROM1                                                                     \
    "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, "  \
    "%20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32}"
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t *r) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], " TT_REGLIST32_FROM1 ";" ::"r"(
                     taddr),
                 TT_IN32(r)
                 : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- softmax arithmetic
// A 3-input maximum.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Row maximum of 64 raw scores (bit patterns in v).
__device__ __forceinline__ float tile_max(const uint32_t *v) {
    float m[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
    for (int j = 0; j < kTN; j += 8) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
            m[q] = fmax3(m[q], __uint_as_float(v[j + 2 * q]), __uint_as_float(v[j + 2 * q + 1]));
    }
    return fmax3(m[0], m[1], fmaxf(m[2], m[3]));
}

// P = 2^(x * c - m) for 64 scores: packed into bf16 pairs (pk), fp32 sum returned.
__device__ __forceinline__ float exp_tile(const uint32_t *v, float c, float m, uint32_t *pk) {
    const uint64_t cc = pk2(c, c), nm = pk2(-m, -m);
    uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
    for (int j = 0; j < kTN / 2; ++j) {
        const uint64_t y = ffma2(pk2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1])), cc, nm);
        float y0, y1;
        upk2(y, y0, y1);
        const uint64_t p = pk2(ex2_approx(y0), ex2_approx(y1));
        acc[j & 3] = fadd2(acc[j & 3], p);
        float p0, p1;
        upk2(p, p0, p1);
        pk[j] = pack_bf16x2(p0, p1);
    }
    const uint64_t s = fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3]));
    float s0, s1;
    upk2(s, s0, s1);
    return s0 + s1;
}

// ---------------------------------------------------------------- scheduling
struct Seg {
    int p, b, g, rg, L, nctx, rows, nh, tile0, ntiles, c_first, c_last;
};

__device__ __forceinline__ int owner_of(int64_t t, int P, int64_t T) {
    return static_cast<int>(((t + 1) * P - 1) / T);
}

struct Sched {
    const int *prefix;
    const uint8_t *tail;  // keys in each pair's last context tile (0 when L_b = 0)
    int P;
    int64_t T, tcur, tend;

    // Next segment of this CTA's range.  Units [prefix[p], prefix[p] + kSegCost) of a
    // pair carry no work; a range that holds only such units of a pair skips it.
    __device__ bool next(const AttnArgs &a, Seg &s) {
        while (tcur < tend) {
            int lo = 0, hi = a.npairs;  // prefix[lo] <= tcur < prefix[hi]
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (prefix[mid] <= tcur) lo = mid; else hi = mid;
            }
            const int p = lo;
            const int64_t rs = prefix[p] + kSegCost, pe = prefix[p + 1];
            const int64_t t0 = tcur > rs ? tcur : rs;
            const int64_t seg_end = pe < tend ? pe : tend;
            tcur = seg_end;
            if (t0 >= seg_end) continue;
            s.p = p;
            s.rg = p % a.NRG;
            const int bg = p / a.NRG;
            s.g = bg % a.Hkv;
            s.b = bg / a.Hkv;
            // the context length comes from shared memory (no global read here); a pair
            // attending to the prefix only has no block tile (and one empty tile when
            // its prefix is empty)
            s.nctx = static_cast<int>(pe - rs) - (a.keys == TT_KEYS_PREFIX ? 0 : 1);
            s.L = s.nctx == 0 ? 0 : (s.nctx - 1) * kTN + tail[p];
            s.rows = min(kRows, a.R - s.rg * kRows);
            s.nh = s.rows > 128 ? 2 : 1;
            s.tile0 = static_cast<int>(t0 - rs);
            s.ntiles = static_cast<int>(seg_end - t0);
            s.c_first = owner_of(rs, P, T);
            s.c_last = owner_of(pe - 1, P, T);
            return true;
        }
        return false;
    }
};

// Prefix length of pair p's sequence, clamped into [0, Lmax] (a value outside is
// recorded in the error word when `flag`), and 0 when only the block's keys count.
__device__ __forceinline__ int pair_len(const AttnArgs &a, int p, bool flag) {
    int L = a.lens[p / (a.Hkv * a.NRG)];
    if (L < 0 || L > a.Lmax) {
        if (flag) atomicOr(a.err_word, kErrCtxLen);
        L = L < 0 ? 0 : a.Lmax;
    }
    return a.keys == TT_KEYS_BLOCK ? 0 : L;
}
// 64-key tiles of a pair: the prefix tiles, plus the block tile unless only the prefix
// counts (then at least one tile, empty when the prefix is).
__device__ __forceinline__ int pair_tiles(const AttnArgs &a, int L) {
    const int nctx = (L + kTN - 1) / kTN;
    return a.keys == TT_KEYS_PREFIX ? (nctx > 0 ? nctx : 1) : nctx + 1;
}

__device__ __forceinline__ int tile_valid(const AttnArgs &a, const Seg &s, int tile) {
    return tile == s.nctx ? a.S : min(kTN, s.L - tile * kTN);
}

// ---------------------------------------------------------------- roles
template <int D>
struct Smem {
    uint32_t stages, qbuf, bars;
    int *prefix;
    volatile int *err;
    volatile int *last;
    uint32_t *tmem_slot;
    static constexpr int S2 = 2 * Cfg<D>::kStages;
    __device__ uint32_t full(int i) const { return bars + 8 * i; }
    __device__ uint32_t empty(int i) const { return bars + 8 * (Cfg<D>::kStages + i); }
    __device__ uint32_t s_full(int h, int b) const { return bars + 8 * (S2 + 2 * h + b); }
    __device__ uint32_t p_full(int h, int b) const { return bars + 8 * (S2 + 4 + 2 * h + b); }
    __device__ uint32_t pv_done(int h, int b) const { return bars + 8 * (S2 + 8 + 2 * h + b); }
    __device__ uint32_t q_ready(int h) const { return bars + 8 * (S2 + 12 + h); }
    __device__ uint32_t fin(int h) const { return bars + 8 * (S2 + 14 + h); }
    __device__ uint32_t turn(int h) const { return bars + 8 * (S2 + 16 + h); }
    __device__ uint32_t q_tma(int h) const { return bars + 8 * (S2 + 18 + h); }
    __device__ uint32_t q_tile(int h) const { return qbuf + h * Cfg<D>::kQHalfBytes; }
};

// Page of context tile `tile` of sequence b in a paged cache.  Tiles holding no key
// of the prefix (an empty prefix's one tile) need no page; a page id outside the
// pool is recorded in the error word and replaced by n_pages, past the map's end, so
// the TMA load reads the fill value instead of another sequence's keys.
__device__ __forceinline__ int page_at(const AttnArgs &a, int b, int tile, int L) {
    if (tile * kTN >= L) return a.n_pages;
    const int pg = __ldg(a.page_of + static_cast<int64_t>(b) * a.max_pages + tile);
    if (pg < 0 || pg >= a.n_pages) {
        atomicOr(a.err_word, kErrPage);
        return a.n_pages;
    }
    return pg;
}

template <int D>
__device__ void role_producer(const AttnArgs &a, Sched sch, const Smem<D> &sm,
                              const CUtensorMap *tkc, const CUtensorMap *tvc,
                              const CUtensorMap *tkb, const CUtensorMap *tvb,
                              const CUtensorMap *tq) {
    using C = Cfg<D>;
    int stage = 0, nissued = 0;
    uint32_t phase = 0, issued = 0, last_par = 0;
    // K/V tiles are read once: first in line for eviction from L2, so they do not
    // push out the partials the merge reads back
    const uint64_t policy = l2_evict_first();
    Seg s;
    bool ok = true;
    int next_page = 0;  // paged cache: page of the next context tile, read one tile ahead
    uint32_t q_sent = 0;  // halves whose first Q came by TMA (drained at the end)
    bool first = true;
    while (ok && sch.next(a, s)) {
        if (first && a.q_tma) {
            // The first segment's Q, ahead of every K/V tile: one 128-row box per half
            // and 64-column chunk (rows (s, head) of the pair in order, s past S read as
            // zeros), in the 128-byte swizzled K-major layout the Q K^T descriptor reads.
            // The CTAs sharing a split pair load the same Q at about the same time: it
            // is kept in L2 rather than evicted first like the K/V tiles.
            const uint64_t q_policy = l2_evict_last();
            for (int h = 0; h < s.nh; ++h) {
                mbar_expect_tx(sm.q_tma(h), C::kQHalfBytes);
                const int s0 = (s.rg * kRows + h * 128) / a.G;
#pragma unroll
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_4d(sm.q_tile(h) + c * C::kQRegion, tq, c * 64, s.g * a.G, s0, s.b,
                                sm.q_tma(h), q_policy);
                q_sent |= 1u << h;
            }
        }
        first = false;
        if (a.page_of && s.tile0 < s.nctx) next_page = page_at(a, s.b, s.tile0, s.L);
        for (int it = 0; it < s.ntiles; ++it) {
            if (!mbar_wait(sm.empty(stage), phase ^ 1, sm.err, 1)) { ok = false; break; }
            const uint32_t full = sm.full(stage);
            mbar_expect_tx(full, C::kStageBytes);
            const int tile = s.tile0 + it;
            const bool blk = tile == s.nctx;
            // ctx maps: (d, Lmax, Hkv, B), or for a paged cache (d, 64, Hkv, n_pages);
            // block maps: (d, Hkv, S, B)
            const CUtensorMap *mk = blk ? tkb : tkc;
            const CUtensorMap *mv = blk ? tvb : tvc;
            int c1 = blk ? s.g : tile * kTN, c3 = s.b;
            if (!blk && a.page_of) {
                // the tile's page (a page outside the pool is flagged and read as the
                // fill value: the coordinate n_pages lies past the map)
                c1 = 0;
                c3 = next_page;
                if (it + 1 < s.ntiles && tile + 1 < s.nctx)
                    next_page = page_at(a, s.b, tile + 1, s.L);
            }
            const int c2 = blk ? 0 : s.g;
            const uint32_t sb = sm.stages + stage * C::kStageBytes;
#pragma unroll
            for (int c = 0; c < C::kChunks; ++c) {
                tma_load_4d(sb + c * C::kRegionBytes, mk, c * 64, c1, c2, c3, full, policy);
                tma_load_4d(sb + (C::kChunks + c) * C::kRegionBytes, mv, c * 64, c1, c2, c3, full,
                            policy);
            }
            issued |= 1u << stage;
            last_par = (last_par & ~(1u << stage)) | (phase << stage);
            if (++stage == C::kStages) { stage = 0; phase ^= 1; }
            // At kernel start every SM asks for its first K/V tiles at once; a first Q
            // loaded by the softmax warps would queue behind them.  Without the TMA Q,
            // wait for that Q after one tile before filling the rest of the ring.
            if (ok && !a.q_tma && ++nissued == 1 && !mbar_wait(sm.q_ready(0), 0, sm.err, 1))
                ok = false;
        }
    }
    // no copy may still be landing when the CTA exits
    for (int st = 0; st < C::kStages; ++st)
        if (issued >> st & 1u) mbar_drain(sm.full(st), last_par >> st & 1u);
    for (int h = 0; h < 2; ++h)
        if (q_sent >> h & 1u) mbar_drain(sm.q_tma(h), 0);
}

// MMA warp of half h (warp 9 + h).  At step it it issues S_h = Q_h K^T for tile it
// into S buffer it&1 and then O_h += P_h V for tile it-1 (once the softmax has
// written that P over its S buffer).  Buffer it&1 last held tile it-2, whose P V
// this warp issued one step earlier, so the scores of the next tile are computed
// while the softmax works on the current one.  The two halves run independently; a
// K/V stage is released when both MMA warps have finished with it (empty barrier
// of count 2).
template <int D>
__device__ void role_mma(const AttnArgs &a, Sched sch, const Smem<D> &sm, uint32_t tmem, int h) {
    using C = Cfg<D>;
    const int lane = threadIdx.x & 31;
    auto wait = [&](uint32_t bar, uint32_t par) -> bool { return warp_wait(bar, par, sm.err, 2); };
    // descriptor bases; a descriptor moves by (byte offset >> 4) in its address field
    const uint64_t kdesc0 = sdesc_sw128(sm.stages, 16, 1024);
    const uint64_t vdesc0 =
        sdesc_sw128(sm.stages + C::kChunks * C::kRegionBytes, C::kRegionBytes, 1024);
    const uint64_t qdesc0 = sdesc_sw128(sm.q_tile(h), 16, 1024);
    const uint32_t d_o = tmem + C::colO(h);
    int stage = 0, prev_stage = 0;
    uint32_t phase = 0, qpar = 0, s_cnt = 0, p_cnt = 0;
    bool ok = true;
    Seg s;
    int seg_idx = 0;  // segments of the CTA so far (the first one's Q may come by TMA)
    while (ok && sch.next(a, s)) {
        const bool q_by_tma = a.q_tma && seg_idx++ == 0;
        if (h >= s.nh) {  // half unused in this segment: release each stage at once
            for (int it = 0; it < s.ntiles; ++it) {
                if (!wait(sm.full(stage), phase)) { ok = false; break; }
                if (lane == 0) mbar_arrive(sm.empty(stage));
                if (++stage == C::kStages) { stage = 0; phase ^= 1; }
            }
            continue;
        }
        for (int it = 0; it <= s.ntiles && ok; ++it) {
            if (it < s.ntiles) {
                const int nvalid = tile_valid(a, s, s.tile0 + it);
                if (!wait(sm.full(stage), phase)) { ok = false; break; }
                if (nvalid < kTN) {
                    // V rows past the valid keys may hold anything (rows >= L_b of the
                    // cache); P is 0 there, and 0 * NaN must not reach O: zero them
                    // (both MMA warps write the same zeros before their own P V).
                    const uint32_t vb = sm.stages + stage * C::kStageBytes +
                                        C::kChunks * C::kRegionBytes;
#pragma unroll
                    for (int c = 0; c < C::kChunks; ++c)
                        for (uint32_t off = nvalid * 128 + lane * 16; off < C::kRegionBytes;
                             off += 512)
                            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(
                                             vb + c * C::kRegionBytes + off),
                                         "r"(0u)
                                         : "memory");
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                }
                if (it == 0) {
                    if (q_by_tma) {
                        if (!wait(sm.q_tma(h), 0)) { ok = false; break; }
                    } else {
                        if (!wait(sm.q_ready(h), qpar)) { ok = false; break; }
                        qpar ^= 1;
                    }
                }
                tc_fence_after();
                const uint32_t d_s = tmem + C::colS(h, s_cnt & 1);
                const uint64_t kd = kdesc0 + ((stage * C::kStageBytes) >> 4);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t koff = (kk >> 2) * C::kRegionBytes + (kk & 3) * 32;
                    const uint32_t qoff = (kk >> 2) * C::kQRegion + (kk & 3) * 32;
                    tc_mma_ss_e(d_s, qdesc0 + (qoff >> 4), kd + (koff >> 4), C::kIdescQK, kk > 0);
                }
                tc_commit_e(sm.s_full(h, s_cnt & 1));
                ++s_cnt;
            }
            if (it > 0) {  // O_h += P_h V for the previous tile
                const uint32_t b = p_cnt & 1;
                if (!wait(sm.p_full(h, b), (p_cnt >> 1) & 1)) { ok = false; break; }
                tc_fence_after();
                const uint64_t vd = vdesc0 + ((prev_stage * C::kStageBytes) >> 4);
                const uint32_t a_p = tmem + C::colS(h, b);  // P: 16 keys per 8 columns
#pragma unroll
                for (int kk = 0; kk < kTN / 16; ++kk)
                    tc_mma_ts_e(d_o, a_p + kk * 8, vd + ((kk * 2048) >> 4), C::kIdescPV,
                                (it > 1 || kk > 0) ? 1u : 0u);
                tc_commit_e(sm.pv_done(h, b));
                ++p_cnt;
                tc_commit_e(sm.empty(prev_stage));
            }
            if (it < s.ntiles) {
                prev_stage = stage;
                if (++stage == C::kStages) { stage = 0; phase ^= 1; }
            }
        }
    }
    // every MMA issued here completes before TMEM is freed
    tc_commit_e(sm.fin(h));
    if (lane == 0) mbar_drain(sm.fin(h), 0);
    __syncwarp();
}

template <int D>
__device__ __forceinline__ void store_row(const AttnArgs &a, const Seg &s, int rl, float *o,
                                          int col0) {
    const int rr = s.rg * kRows + rl;
    const int sq = rr / a.G, head = s.g * a.G + rr % a.G;
    uint16_t *dst = a.out + s.b * a.os[0] + sq * a.os[1] + head * a.os[2] + col0;
    if (a.o_gate) {  // adaLN-single gate of the attention output, [B, Hq, D]
        const float4 *gp = reinterpret_cast<const float4 *>(
            a.o_gate + (static_cast<int64_t>(s.b) * a.Hq + head) * D + col0);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float4 gv = __ldg(gp + j);
            o[4 * j] *= gv.x;
            o[4 * j + 1] *= gv.y;
            o[4 * j + 2] *= gv.z;
            o[4 * j + 3] *= gv.w;
        }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint4 v;
        v.x = pack_bf16x2(o[8 * j + 0], o[8 * j + 1]);
        v.y = pack_bf16x2(o[8 * j + 2], o[8 * j + 3]);
        v.z = pack_bf16x2(o[8 * j + 4], o[8 * j + 5]);
        v.w = pack_bf16x2(o[8 * j + 6], o[8 * j + 7]);
        *reinterpret_cast<uint4 *>(dst + 8 * j) = v;
    }
}

__device__ __forceinline__ void store_lse(const AttnArgs &a, const Seg &s, int rl, float m_log2,
                                          float l) {
    if (!a.lse) return;
    const int rr = s.rg * kRows + rl;
    const int sq = rr / a.G, head = s.g * a.G + rr % a.G;
    a.lse[(static_cast<int64_t>(s.b) * a.Hq + head) * a.S + sq] =
        l > 0.f ? (m_log2 + __log2f(l)) * kLn2 : -INFINITY;  // no key: empty sum
}

template <int D>
__device__ void role_softmax(const AttnArgs &a, Sched sch, const Smem<D> &sm, uint32_t tmem) {
    using C = Cfg<D>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = warp >> 2, q4 = warp & 3, r = q4 * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(q4 * 32) << 16);  // this warp's lanes
    const float c = a.scale_log2;
    auto wait = [&](uint32_t bar, uint32_t par) -> bool { return warp_wait(bar, par, sm.err, 3); };
    // O_h += P_h V of this half's tile number n has completed
    auto wait_pv = [&](uint32_t n) -> bool { return wait(sm.pv_done(h, n & 1), (n >> 1) & 1); };
    uint32_t cnt = 0;  // tiles of this half so far; tile n uses S buffer n & 1
    // When both halves are active the two warpgroups take turns at the arithmetic of
    // a tile (turn barriers): one computes while the other waits on its memory
    // traffic and barriers, instead of both doing the same phase at once.
    uint32_t tpar = h == 0 ? 1u : 0u;
    const int rl = h * 128 + r;  // row within the pair
    // this thread's Q row inside a [128 rows][128 B] chunk, 128-byte swizzle
    const uint32_t qrow = sm.q_tile(h) + (r >> 3) * 1024 + (r & 7) * 128;
    // Q row of segment q_seg -> shared memory, K-major in 64-column chunks with the
    // 128-byte swizzle of the K tiles (zeros for rows past the pair), then q_ready.
    // The caller makes sure no Q K^T still reads the previous Q.
    auto load_q = [&](const Seg &q_seg) {
        uint4 qv[D / 8];
        if (rl < q_seg.rows) {
            const int rr = q_seg.rg * kRows + rl;
            const int sq = rr / a.G, head = q_seg.g * a.G + rr % a.G;
            const uint4 *src = reinterpret_cast<const uint4 *>(a.q + q_seg.b * a.qs[0] +
                                                               sq * a.qs[1] + head * a.qs[2]);
#pragma unroll
            for (int j = 0; j < D / 8; ++j) qv[j] = __ldg(src + j);
            if (a.q_scale) {  // adaLN-single: q' = q (1 + scale) + shift, rounded to bf16
                const int64_t mo = (static_cast<int64_t>(q_seg.b) * a.Hq + head) * D;
                const float4 *sc = reinterpret_cast<const float4 *>(a.q_scale + mo);
                const float4 *sh = reinterpret_cast<const float4 *>(a.q_shift + mo);
#pragma unroll
                for (int j = 0; j < D / 8; ++j) {
                    const float4 s0 = __ldg(sc + 2 * j), s1 = __ldg(sc + 2 * j + 1);
                    const float4 h0 = __ldg(sh + 2 * j), h1 = __ldg(sh + 2 * j + 1);
                    qv[j].x = pack_bf16x2(fmaf(bf16_lo(qv[j].x), 1.f + s0.x, h0.x),
                                          fmaf(bf16_hi(qv[j].x), 1.f + s0.y, h0.y));
                    qv[j].y = pack_bf16x2(fmaf(bf16_lo(qv[j].y), 1.f + s0.z, h0.z),
                                          fmaf(bf16_hi(qv[j].y), 1.f + s0.w, h0.w));
                    qv[j].z = pack_bf16x2(fmaf(bf16_lo(qv[j].z), 1.f + s1.x, h1.x),
                                          fmaf(bf16_hi(qv[j].z), 1.f + s1.y, h1.y));
                    qv[j].w = pack_bf16x2(fmaf(bf16_lo(qv[j].w), 1.f + s1.z, h1.z),
                                          fmaf(bf16_hi(qv[j].w), 1.f + s1.w, h1.w));
                }
            }
        } else {
#pragma unroll
            for (int j = 0; j < D / 8; ++j) qv[j] = make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int j = 0; j < D / 8; ++j)
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(
                             qrow + (j >> 3) * C::kQRegion + (((j & 7) ^ (r & 7)) << 4)),
                         "r"(qv[j].x), "r"(qv[j].y), "r"(qv[j].z), "r"(qv[j].w)
                         : "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive(sm.q_ready(h));
    };
    // next segment in which this half takes part
    int pulled = 0;  // segments of the CTA pulled so far
    auto next_mine = [&](Seg &n) -> bool {
        while (sch.next(a, n)) {
            ++pulled;
            if (h < n.nh) return true;
        }
        return false;
    };
    bool ok = true;
    Seg s, nxt;
    bool have = next_mine(s);
    // the CTA's first segment's Q comes by TMA from the producer (when enabled)
    if (have && !(a.q_tma && pulled == 1)) load_q(s);
    while (ok && have) {
        const bool valid = rl < s.rows;
        float m_run = -INFINITY, l_run = 0.f;
        for (int it = 0; it < s.ntiles; ++it) {
            const int nvalid = tile_valid(a, s, s.tile0 + it);
            const uint32_t sb = C::colS(h, cnt & 1);
            if (!wait(sm.s_full(h, cnt & 1), (cnt >> 1) & 1)) { ok = false; break; }
            tc_fence_after();
            uint32_t v[kTN];
            tmem_ld32(tl + sb, v);
            tmem_ld32(tl + sb + 32, v + 32);
            tmem_wait_ld(v);
            tmem_touch(v + 32);
            if (nvalid < kTN) {
#pragma unroll
                for (int j = 0; j < kTN; ++j)
                    if (j >= nvalid) v[j] = __float_as_uint(-INFINITY);
            }
            // The running max m_run (log2 units) is raised only when a tile's max exceeds
            // it by more than kRescaleLog2; otherwise P is taken against the stale max,
            // which leaves O / l unchanged (both carry the same factor) and lets the
            // exponentials start without waiting for this tile's max.
            if (s.nh == 2) {
                if (!wait(sm.turn(h), tpar)) { ok = false; break; }
                tpar ^= 1;
            }
            const float mx = tile_max(v);
            if (it == 0) m_run = mx * c;
            uint32_t pk[kTN / 2];
            // a tile without a key (an empty prefix attended alone) has max -inf: its
            // P is 0 whatever the reference, and 0 keeps the arithmetic finite
            float lsum = exp_tile(v, c, m_run == -INFINITY ? 0.f : m_run, pk);
            if (s.nh == 2) mbar_arrive_after(sm.turn(h ^ 1), lsum);
            if (it > 0) {
                const float m_tile = mx * c;
                const bool need = m_tile > m_run + kRescaleLog2;
                if (__any_sync(0xFFFFFFFFu, need)) {
                    // O_h must hold every earlier tile before it is rescaled
                    if (!wait_pv(cnt - 1)) { ok = false; break; }
                    tc_fence_after();
                    const float f = need ? ex2_approx(m_run - m_tile) : 1.f;
                    if (need) { l_run *= f; m_run = m_tile; }
#pragma unroll 1
                    for (int j = 0; j < D / 32; ++j) {
                        uint32_t o[32];
                        tmem_ld32(tl + C::colO(h) + 32 * j, o);
                        tmem_wait_ld(o);
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
                        tmem_st32(tl + C::colO(h) + 32 * j, o);
                    }
                    tmem_wait_st();
                    lsum = exp_tile(v, c, m_run, pk);
                }
            }
            l_run += lsum;
            // P (bf16 pairs) over the first 32 columns of this tile's S buffer
            tmem_st32(tl + sb, pk);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(sm.p_full(h, cnt & 1));
            ++cnt;
        }
        if (!ok) break;
        // The next segment's Q goes into shared memory before this segment's epilogue
        // (every Q K^T of this segment has completed: the last S was read), so the MMA
        // warp can start on the next segment while O is read out and stored.
        const bool have_next = next_mine(nxt);
        if (have_next) load_q(nxt);
        // ---- segment epilogue: O_h is final once the last P_h V is done
        if (!wait_pv(cnt - 1)) { ok = false; break; }
        tc_fence_after();
        if (s.c_first == s.c_last) {
            const float inv = l_run > 0.f ? 1.f / l_run : 0.f;  // no key at all: output 0
#pragma unroll 1
            for (int j = 0; j < D / 32; ++j) {
                uint32_t o[32];
                tmem_ld32(tl + C::colO(h) + 32 * j, o);
                tmem_wait_ld(o);
                if (valid) {
                    float f[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) f[e] = __uint_as_float(o[e]) * inv;
                    store_row<D>(a, s, rl, f, 32 * j);
                }
            }
            if (valid) store_lse(a, s, rl, m_run, l_run);
        } else {
            // ---- split pair: write this CTA's partial (O / l, m, l); block_attn_merge_kernel
            // combines the partials once the whole grid has finished
            const size_t slot = static_cast<size_t>(blockIdx.x + s.p);
            const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll 1
            for (int j = 0; j < D / 32; ++j) {
                uint32_t o[32];
                tmem_ld32(tl + C::colO(h) + 32 * j, o);
                tmem_wait_ld(o);
                if (valid) {
                    float *dst = a.part_o + (slot * D + 32 * j) * kRows + rl;
#pragma unroll
                    for (int e = 0; e < 32; ++e) __stcg(dst + e * kRows, __uint_as_float(o[e]) * inv);
                }
            }
            if (valid) __stcg(a.part_ml + slot * kRows + rl, make_float2(m_run, l_run));
        }
        s = nxt;
        have = have_next;
    }
}


template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    block_attn_tc_kernel(const __grid_constant__ CUtensorMap tm_kc,
                         const __grid_constant__ CUtensorMap tm_vc,
                         const __grid_constant__ CUtensorMap tm_kb,
                         const __grid_constant__ CUtensorMap tm_vb,
                         const __grid_constant__ CUtensorMap tm_q, const AttnArgs a) {
    using C = Cfg<D>;
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    unsigned char *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);  // 1024-byte aligned
    int *prefix = reinterpret_cast<int *>(smem + C::kPrefixOffset);
    uint8_t *tail = reinterpret_cast<uint8_t *>(prefix + a.npairs + 1);
    int *misc = reinterpret_cast<int *>(smem + C::kMiscOffset);
    __shared__ int warp_sums[kThreads / 32];

    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    constexpr int kWarps = kThreads / 32;

    // ---- tile counts per pair and their exclusive prefix sum
    {
        const int per = (a.npairs + kThreads - 1) / kThreads;
        const int p0 = min(a.npairs, t * per), p1 = min(a.npairs, p0 + per);
        int local = 0;
        for (int p = p0; p < p1; ++p) {
            const int L = pair_len(a, p, blockIdx.x == 0);
            local += pair_tiles(a, L) + kSegCost;
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
            if (lane < kWarps) warp_sums[lane] = w;
        }
        __syncthreads();
        int run = incl - local + (warp > 0 ? warp_sums[warp - 1] : 0);
        for (int p = p0; p < p1; ++p) {
            prefix[p] = run;
            const int L = pair_len(a, p, false);
            const int nctx = (L + kTN - 1) / kTN;
            tail[p] = static_cast<uint8_t>(nctx == 0 ? 0 : L - (nctx - 1) * kTN);
            run += pair_tiles(a, L) + kSegCost;
        }
        if (t == kThreads - 1) prefix[a.npairs] = run;
        __syncthreads();
    }
    const int64_t T = prefix[a.npairs];
    int64_t parts = T / kMinTiles;
    parts = parts < 1 ? 1 : (parts > a.P ? a.P : parts);
    const int P = static_cast<int>(parts);
    const int cta = blockIdx.x;
    // the merge kernel (programmatic dependent launch) may be scheduled now; it
    // waits for this grid to finish before it reads anything
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (cta >= P) return;
    if (cta == 0)
        for (int p = t; p < a.npairs; p += kThreads)
            a.pair_split[p] = make_int2(owner_of(prefix[p] + kSegCost, P, T),
                                        owner_of(prefix[p + 1] - 1, P, T));

    Smem<D> sm;
    sm.stages = smem_u32(smem);
    sm.qbuf = smem_u32(smem + C::kQOffset);
    sm.bars = smem_u32(smem + C::kBarOffset);
    sm.prefix = prefix;
    sm.tmem_slot = reinterpret_cast<uint32_t *>(misc);
    sm.err = misc + 1;
    sm.last = misc + 2;
    if (t == 0) {
        for (int i = 0; i < C::kStages; ++i) {
            mbar_init(sm.full(i), 1);
            mbar_init(sm.empty(i), 2);
        }
        for (int h = 0; h < 2; ++h) {
            for (int b = 0; b < 2; ++b) {
                mbar_init(sm.s_full(h, b), 1);
                mbar_init(sm.p_full(h, b), 128);
                mbar_init(sm.pv_done(h, b), 1);
            }
            mbar_init(sm.q_ready(h), 128);
            mbar_init(sm.turn(h), 128);
        }
        mbar_init(sm.fin(0), 1);
        mbar_init(sm.fin(1), 1);
        mbar_init(sm.q_tma(0), 1);
        mbar_init(sm.q_tma(1), 1);
        *sm.err = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(sm.tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *sm.tmem_slot;

    Sched sch;
    sch.prefix = prefix;
    sch.tail = tail;
    sch.P = P;
    sch.T = T;
    sch.tcur = static_cast<int64_t>(cta) * T / P;
    sch.tend = static_cast<int64_t>(cta + 1) * T / P;

    if (warp == kProducerWarp) {
        if (lane == 0) role_producer<D>(a, sch, sm, &tm_kc, &tm_vc, &tm_kb, &tm_vb, &tm_q);
        __syncwarp();
    } else if (warp >= kMmaWarp) {
        role_mma<D>(a, sch, sm, tmem, warp - kMmaWarp);
    } else {
        role_softmax<D>(a, sch, sm, tmem);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
    if (t == 0 && *sm.err) atomicOr(a.err_word, 1 << (*sm.err - 1));
}

// Combines the partials of every pair whose tiles were split across CTAs:
//   M = max_c m_c,  out = sum_c 2^(m_c-M) l_c (O_c/l_c) / sum_c 2^(m_c-M) l_c,
//   lse = (M + log2 sum_c 2^(m_c-M) l_c) ln 2.
// Block = (pair, 32-row chunk of the pair's 256 rows, 64-column chunk), 8 warps;
// warp w owns 8 columns and lane i row i of the chunk, so every load of a partial is
// a coalesced 128-byte line.  The loads of kMergeBatch partials are issued together
// before they are folded in with a running maximum: the kernel is bound by load
// latency, and this keeps the round trips per row at ceil(parts / kMergeBatch).
// Launched as a programmatic dependent of the attention kernel: griddepcontrol.wait
// returns once that grid has completed and its writes are visible.
constexpr int kMergeThreads = 256;
constexpr int kMergeCols = 8;   // columns per warp
constexpr int kMergeBatch = 4;  // partials in flight per thread
template <int D>
__global__ void __launch_bounds__(kMergeThreads, 4) block_attn_merge_kernel(const AttnArgs a) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    constexpr int kColChunks = D / (8 * kMergeCols);
    const int p = blockIdx.x / (8 * kColChunks);
    const int chunk = (blockIdx.x / kColChunks) & 7, cc = blockIdx.x % kColChunks;
    const int2 cs = a.pair_split[p];
    if (cs.x == cs.y) return;  // finished inside one CTA
    const int rg = p % a.NRG;
    const int rows = min(kRows, a.R - rg * kRows);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int rl = chunk * 32 + lane;
    if (rl >= rows) return;
    const int col0 = (cc * 8 + warp) * kMergeCols;
    // the partial of CTA c for pair p sits in slot c + p
    const float2 *mlp = a.part_ml + static_cast<size_t>(p) * kRows + rl;  // + c * kRows
    const float *op = a.part_o + (static_cast<size_t>(p) * D + col0) * kRows + rl;
    float M = -INFINITY, den = 0.f;
    float acc[kMergeCols];
#pragma unroll
    for (int e = 0; e < kMergeCols; ++e) acc[e] = 0.f;
    for (int c0 = cs.x; c0 <= cs.y; c0 += kMergeBatch) {
        float2 ml[kMergeBatch];
        float v[kMergeBatch][kMergeCols];
#pragma unroll
        for (int i = 0; i < kMergeBatch; ++i) {
            const int c = min(c0 + i, cs.y);  // past the last partial: a repeat, not folded in
            ml[i] = __ldcg(mlp + static_cast<size_t>(c) * kRows);
            const float *src = op + static_cast<size_t>(c) * D * kRows;
#pragma unroll
            for (int e = 0; e < kMergeCols; ++e) v[i][e] = __ldcg(src + e * kRows);
        }
#pragma unroll
        for (int i = 0; i < kMergeBatch; ++i) {
            if (c0 + i <= cs.y && ml[i].x != -INFINITY) {  // a partial without keys adds nothing
                const float Mn = fmaxf(M, ml[i].x);
                const float so = ex2_approx(M - Mn), w = ex2_approx(ml[i].x - Mn) * ml[i].y;
                M = Mn;
                den = den * so + w;
#pragma unroll
                for (int e = 0; e < kMergeCols; ++e) acc[e] = acc[e] * so + w * v[i][e];
            }
        }
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    const int rr = rg * kRows + rl;
    const int bg = p / a.NRG, g = bg % a.Hkv, b = bg / a.Hkv;
    const int sq = rr / a.G, head = g * a.G + rr % a.G;
    uint16_t *dst = a.out + b * a.os[0] + sq * a.os[1] + head * a.os[2] + col0;
    if (a.o_gate) {  // adaLN-single gate of the attention output, [B, Hq, D]
        const float4 *gp = reinterpret_cast<const float4 *>(
            a.o_gate + (static_cast<int64_t>(b) * a.Hq + head) * D + col0);
        const float4 g0 = __ldg(gp), g1 = __ldg(gp + 1);
        acc[0] *= g0.x; acc[1] *= g0.y; acc[2] *= g0.z; acc[3] *= g0.w;
        acc[4] *= g1.x; acc[5] *= g1.y; acc[6] *= g1.z; acc[7] *= g1.w;
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    o.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
    o.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
    o.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
    *reinterpret_cast<uint4 *>(dst) = o;
    if (col0 == 0 && a.lse)
        a.lse[(static_cast<int64_t>(b) * a.Hq + head) * a.S + sq] =
            den > 0.f ? (M + __log2f(den)) * kLn2 : -INFINITY;
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
    if (np * ((static_cast<int64_t>(d->Lmax) + kTN - 1) / kTN + 1 + kSegCost) >= (int64_t(1) << 31))
        return fail(TT_ERR_UNSUPPORTED, "%s: more than 2^31 key tiles", fn);
    geo->npairs = static_cast<int>(np);
    geo->P = sm_count();
    if (geo->P <= 0) return fail(TT_ERR_CUDA, "%s: no CUDA device", fn);
    return TT_OK;
}

struct AttnWs {
    int *err_word;
    int2 *pair_split;
    float2 *part_ml;
    float *part_o;
    size_t bytes;
};

AttnWs carve(void *base, int npairs, size_t slots, int d) {
    Carve c(base);
    AttnWs w;
    w.err_word = c.take<int>(1);
    w.pair_split = c.take<int2>(static_cast<size_t>(npairs));
    w.part_ml = c.take<float2>(slots * kRows);
    w.part_o = c.take<float>(slots * kRows * d);
    w.bytes = c.bytes();
    return w;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

// 4-D bf16 tensor map, 128-byte swizzle, box (64, b1, b2, 1); strides in elements.
tt_status make_map(CUtensorMap *m, const void *base, uint64_t d0, uint64_t d1, uint64_t d2,
                   uint64_t d3, int64_t s1, int64_t s2, int64_t s3, uint32_t b1, uint32_t b2,
                   const char *fn, const char *what) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return fail(TT_ERR_CUDA, "%s: cuTensorMapEncodeTiled unavailable", fn);
    const cuuint64_t dims[4] = {d0, d1, d2, d3};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(s1) * 2, static_cast<cuuint64_t>(s2) * 2,
                                   static_cast<cuuint64_t>(s3) * 2};
    const cuuint32_t box[4] = {64, b1, b2, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims,
                           strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(TT_ERR_UNSUPPORTED, "%s: tensor map for %s rejected (CUresult %d)", fn, what,
                    static_cast<int>(r));
    return TT_OK;
}

// The four tensor maps of a call depend only on pointers, shape and strides; a small
// per-thread cache skips re-encoding them for repeated calls on the same buffers
// (a decode loop calls every layer with the same caches step after step).
struct MapKey {
    const void *k_ctx, *v_ctx, *k_blk, *v_blk, *q;  // q null: no Q map
    int32_t B, S, Hq, Hkv, Lmax, d, n_pages;  // n_pages > 0: paged context pools
    int64_t kc[4], vc[4], kb[4], vb[4], qs[4];
    bool operator==(const MapKey &o) const { return memcmp(this, &o, sizeof(MapKey)) == 0; }
};
struct MapEntry {
    MapKey key;
    CUtensorMap kc, vc, kb, vb, q;
    bool used, has_q;
};
constexpr int kMapCache = 16;

template <int D>
tt_status encode_maps(const tt_attn_desc *d, const void *k_ctx, const void *v_ctx, const void *k_blk,
                      const void *v_blk, const void *q, int n_pages, MapEntry *e, const char *fn) {
    tt_status st;
    // Q [B, S, Hq, d] as (d, Hq, S, B) with a box of 64 columns x G heads x 128/G block
    // positions: one half's 128 rows of a pair.  A map the driver rejects only turns the
    // TMA Q off (the softmax warps load it instead).
    e->has_q = false;
    if (q) {
        const int G = d->Hq / d->Hkv;
        EncodeTiledFn enc = encode_fn();
        if (enc) {
            const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(d->Hq),
                                        static_cast<cuuint64_t>(d->S), static_cast<cuuint64_t>(d->B)};
            const cuuint64_t strides[3] = {static_cast<cuuint64_t>(d->q_strides[2]) * 2,
                                           static_cast<cuuint64_t>(d->q_strides[1]) * 2,
                                           static_cast<cuuint64_t>(d->q_strides[0]) * 2};
            const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(G),
                                       static_cast<cuuint32_t>(128 / G), 1};
            const cuuint32_t estr[4] = {1, 1, 1, 1};
            e->has_q = enc(&e->q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(q), dims,
                           strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
        }
    }
    const uint64_t B = d->B, S = d->S, Hkv = d->Hkv;
    // a paged cache is a pool [n_pages, Hkv, 64, d]: the map's rows are a page's 64 keys
    // and its outer dimension the page; otherwise [B, Hkv, Lmax, d]
    const uint64_t Lmax = n_pages > 0 ? kTN : d->Lmax;
    const uint64_t outer = n_pages > 0 ? static_cast<uint64_t>(n_pages) : B;
    if ((st = make_map(&e->kb, k_blk, D, Hkv, S, B, d->kblk_strides[2], d->kblk_strides[1],
                       d->kblk_strides[0], 1, 64, fn, "k_blk")) != TT_OK)
        return st;
    if ((st = make_map(&e->vb, v_blk, D, Hkv, S, B, d->vblk_strides[2], d->vblk_strides[1],
                       d->vblk_strides[0], 1, 64, fn, "v_blk")) != TT_OK)
        return st;
    if (d->Lmax > 0) {
        if ((st = make_map(&e->kc, k_ctx, D, Lmax, Hkv, outer, d->kctx_strides[2],
                           d->kctx_strides[1], d->kctx_strides[0], 64, 1, fn, "k_ctx")) != TT_OK)
            return st;
        if ((st = make_map(&e->vc, v_ctx, D, Lmax, Hkv, outer, d->vctx_strides[2],
                           d->vctx_strides[1], d->vctx_strides[0], 64, 1, fn, "v_ctx")) != TT_OK)
            return st;
    } else {  // no context rows: the context maps are never used
        e->kc = e->kb;
        e->vc = e->vb;
    }
    return TT_OK;
}


template <int D>
tt_status launch(const tt_attn_desc *d, AttnArgs a, const void *k_ctx, const void *v_ctx,
                 const void *k_blk, const void *v_blk, cudaStream_t stream, const char *fn) {
    const int n_pages = a.page_of ? a.n_pages : 0;
    // the first Q by TMA: unmodulated queries whose group size G divides 128 (a half's
    // 128 rows are whole block positions)
    const int G = d->Hq / d->Hkv;
    const void *q_tma = (a.q_scale == nullptr && G <= 128 && 128 % G == 0) ? a.q : nullptr;
    thread_local MapEntry cache[kMapCache] = {};
    thread_local int next_slot = 0;
    MapKey key;
    memset(&key, 0, sizeof key);
    key.k_ctx = k_ctx; key.v_ctx = v_ctx; key.k_blk = k_blk; key.v_blk = v_blk; key.q = q_tma;
    key.B = d->B; key.S = d->S; key.Hq = d->Hq; key.Hkv = d->Hkv; key.Lmax = d->Lmax; key.d = d->d;
    if (q_tma) memcpy(key.qs, d->q_strides, sizeof key.qs);
    key.n_pages = n_pages;
    memcpy(key.kc, d->kctx_strides, sizeof key.kc);
    memcpy(key.vc, d->vctx_strides, sizeof key.vc);
    memcpy(key.kb, d->kblk_strides, sizeof key.kb);
    memcpy(key.vb, d->vblk_strides, sizeof key.vb);
    MapEntry *hit = nullptr;
    for (int i = 0; i < kMapCache && !hit; ++i)
        if (cache[i].used && cache[i].key == key) hit = &cache[i];
    if (!hit) {
        tt_status st =
            encode_maps<D>(d, k_ctx, v_ctx, k_blk, v_blk, q_tma, n_pages, &cache[next_slot], fn);
        if (st != TT_OK) return st;
        cache[next_slot].key = key;
        cache[next_slot].used = true;
        hit = &cache[next_slot];
        next_slot = (next_slot + 1) % kMapCache;
    }
    const CUtensorMap &kc = hit->kc, &vc = hit->vc, &kb = hit->kb, &vb = hit->vb;
    a.q_tma = hit->has_q ? 1 : 0;
    const CUtensorMap &tq = hit->has_q ? hit->q : hit->kb;  // unused without the TMA Q
    static std::mutex mu;
    static bool configured[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev < 64 && !configured[dev]) {
            cudaError_t e = cudaFuncSetAttribute(block_attn_tc_kernel<D>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 Cfg<D>::smem_bytes(kMaxPairs));
            if (e != cudaSuccess) return cuda_status(e, "tt_block_attn: smem attribute");
            configured[dev] = true;
        }
    }
    block_attn_tc_kernel<D><<<a.P, kThreads, Cfg<D>::smem_bytes(a.npairs), stream>>>(kc, vc, kb,
                                                                                    vb, tq, a);
    tt_status st2 = cuda_status(cudaGetLastError(), "tt_block_attn launch");
    if (st2 != TT_OK) return st2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.npairs) * 8 * (D / (8 * kMergeCols)));
    cfg.blockDim = dim3(kMergeThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cuda_status(cudaLaunchKernelEx(&cfg, block_attn_merge_kernel<D>, a),
                       "tt_block_attn merge launch");
}

tt_status check_ptrs(const tt_attn_desc *d, const void *q, const void *k_ctx, const void *v_ctx,
                     const int32_t *ctx_lens, const void *k_blk, const void *v_blk,
                     const void *out, const float *lse, const char *fn) {
    if (!q || !k_blk || !v_blk || !out || !ctx_lens || (d->Lmax > 0 && (!k_ctx || !v_ctx)))
        return fail(TT_ERR_INVALID_ARG, "%s: null pointer", fn);
    const void *ptrs[6] = {q, k_ctx, v_ctx, k_blk, v_blk, out};
    for (int i = 0; i < 6; ++i)
        if (reinterpret_cast<uintptr_t>(ptrs[i]) % 16)
            return fail(TT_ERR_INVALID_ARG, "%s: tensor base not 16-byte aligned", fn);
    if (reinterpret_cast<uintptr_t>(ctx_lens) % 4 || (lse && reinterpret_cast<uintptr_t>(lse) % 4))
        return fail(TT_ERR_INVALID_ARG, "%s: ctx_lens/lse misaligned", fn);
    return TT_OK;
}

tt_status check_opts(const tt_attn_desc *d, const tt_attn_opts *o, const char *fn) {
    if (!o) return TT_OK;
    if (o->keys != TT_KEYS_ALL && o->keys != TT_KEYS_PREFIX && o->keys != TT_KEYS_BLOCK)
        return fail(TT_ERR_INVALID_ARG, "%s: unknown key set %d", fn, o->keys);
    if (o->block_table) {
        if (o->max_pages < 1 || o->n_pages < 1)
            return fail(TT_ERR_INVALID_ARG, "%s: paged cache needs max_pages and n_pages >= 1", fn);
        if (static_cast<int64_t>(o->max_pages) * kTN != d->Lmax)
            return fail(TT_ERR_INVALID_ARG, "%s: paged cache needs Lmax = max_pages * 64", fn);
        if (reinterpret_cast<uintptr_t>(o->block_table) % 4)
            return fail(TT_ERR_INVALID_ARG, "%s: block table not 4-byte aligned", fn);
    }
    if ((o->q_scale == nullptr) != (o->q_shift == nullptr))
        return fail(TT_ERR_INVALID_ARG, "%s: q_scale and q_shift go together", fn);
    const void *m[3] = {o->q_scale, o->q_shift, o->o_gate};
    for (int i = 0; i < 3; ++i)
        if (m[i] && reinterpret_cast<uintptr_t>(m[i]) % 16)
            return fail(TT_ERR_INVALID_ARG, "%s: modulation vectors not 16-byte aligned", fn);
    return TT_OK;
}

tt_status run(const tt_attn_desc *d, const tt_attn_opts *o, const Geometry &g, const AttnWs &w,
              const void *q, const void *k_ctx, const void *v_ctx, const int32_t *ctx_lens,
              const void *k_blk, const void *v_blk, void *out, float *lse, cudaStream_t stream,
              const char *fn) {
    AttnArgs a;
    a.keys = o ? o->keys : TT_KEYS_ALL;
    a.page_of = o ? o->block_table : nullptr;
    a.max_pages = o ? o->max_pages : 0;
    a.n_pages = o ? o->n_pages : 0;
    a.q_scale = o ? o->q_scale : nullptr;
    a.q_shift = o ? o->q_shift : nullptr;
    a.o_gate = o ? o->o_gate : nullptr;
    a.q = static_cast<const uint16_t *>(q);
    a.out = static_cast<uint16_t *>(out);
    a.lse = lse;
    for (int i = 0; i < 4; ++i) {
        a.qs[i] = d->q_strides[i];
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
    a.pair_split = w.pair_split;
    a.err_word = w.err_word;
    if (d->d == 128) return launch<128>(d, a, k_ctx, v_ctx, k_blk, v_blk, stream, fn);
    return launch<64>(d, a, k_ctx, v_ctx, k_blk, v_blk, stream, fn);
}

}  // namespace
}  // namespace tt

using namespace tt;

extern "C" {

size_t tt_block_attn_workspace_size(const tt_attn_desc *d) {
    Geometry g;
    if (validate(d, &g, "tt_block_attn_workspace_size") != TT_OK) return 0;
    return carve(nullptr, g.npairs, static_cast<size_t>(g.P) + g.npairs, d->d).bytes;
}

tt_status tt_block_attn(const tt_attn_desc *d, const void *q, const void *k_ctx, const void *v_ctx,
                        const int32_t *ctx_lens, const void *k_blk, const void *v_blk, void *out,
                        float *lse, void *workspace, size_t workspace_bytes, tt_stream_t stream) {
    const char *fn = "tt_block_attn";
    Geometry g;
    tt_status st = validate(d, &g, fn);
    if (st != TT_OK) return st;
    if (d->B == 0) return TT_OK;
    if ((st = check_ptrs(d, q, k_ctx, v_ctx, ctx_lens, k_blk, v_blk, out, lse, fn)) != TT_OK)
        return st;
    AttnWs w = carve(workspace, g.npairs, static_cast<size_t>(g.P) + g.npairs, d->d);
    if (!workspace || workspace_bytes < w.bytes)
        return fail(TT_ERR_WORKSPACE, "%s: workspace of %zu bytes, %zu needed", fn, workspace_bytes,
                    w.bytes);
    if (reinterpret_cast<uintptr_t>(workspace) % 256)
        return fail(TT_ERR_WORKSPACE, "%s: workspace not 256-byte aligned", fn);
    return run(d, nullptr, g, w, q, k_ctx, v_ctx, ctx_lens, k_blk, v_blk, out, lse,
               (cudaStream_t)stream, fn);
}

tt_status tt_block_attn_ex(const tt_attn_desc *d, const tt_attn_opts *opts, const void *q,
                           const void *k_ctx, const void *v_ctx, const int32_t *ctx_lens,
                           const void *k_blk, const void *v_blk, void *out, float *lse,
                           void *workspace, size_t workspace_bytes, tt_stream_t stream) {
    const char *fn = "tt_block_attn_ex";
    Geometry g;
    tt_status st = validate(d, &g, fn);
    if (st != TT_OK) return st;
    if ((st = check_opts(d, opts, fn)) != TT_OK) return st;
    if (d->B == 0) return TT_OK;
    if ((st = check_ptrs(d, q, k_ctx, v_ctx, ctx_lens, k_blk, v_blk, out, lse, fn)) != TT_OK)
        return st;
    AttnWs w = carve(workspace, g.npairs, static_cast<size_t>(g.P) + g.npairs, d->d);
    if (!workspace || workspace_bytes < w.bytes)
        return fail(TT_ERR_WORKSPACE, "%s: workspace of %zu bytes, %zu needed", fn, workspace_bytes,
                    w.bytes);
    if (reinterpret_cast<uintptr_t>(workspace) % 256)
        return fail(TT_ERR_WORKSPACE, "%s: workspace not 256-byte aligned", fn);
    return run(d, opts, g, w, q, k_ctx, v_ctx, ctx_lens, k_blk, v_blk, out, lse,
               (cudaStream_t)stream, fn);
}

tt_status tt_block_attn_error(const void *workspace, int32_t *flag_out, tt_stream_t stream) {
    if (!workspace || !flag_out) return fail(TT_ERR_INVALID_ARG, "tt_block_attn_error: null pointer");
    cudaError_t e = cudaMemcpyAsync(flag_out, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost,
                                    (cudaStream_t)stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
    return cuda_status(e, "tt_block_attn_error");
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
    if ((st = check_ptrs(d, q, k_ctx, v_ctx, ctx_lens, k_blk, v_blk, out, lse, fn)) != TT_OK)
        return st;
    // partial slots that fit: one per pair plus at least one partition
    size_t slots = kStaticScratchBytes / carve(nullptr, 0, 1, d->d).bytes;
    while (slots > 0 && carve(nullptr, g.npairs, slots, d->d).bytes > kStaticScratchBytes) --slots;
    if (slots < static_cast<size_t>(g.npairs) + 1)
        return fail(TT_ERR_UNSUPPORTED,
                    "%s: B*Hkv*ceil(S*Hq/Hkv/256) = %d pairs need more than the %zu-byte static "
                    "scratch (at most %zu pairs at d=%d); use tt_block_attn with a workspace",
                    fn, g.npairs, kStaticScratchBytes, slots > 0 ? slots - 1 : 0, d->d);
    const size_t parts = slots - g.npairs;
    if (static_cast<size_t>(g.P) > parts) g.P = static_cast<int>(parts);
    void *base = nullptr;
    if ((st = static_scratch(&base, fn)) != TT_OK) return st;
    AttnWs w = carve(base, g.npairs, static_cast<size_t>(g.P) + g.npairs, d->d);
    // the error word and the per-pair split table start at zero whatever an earlier call left
    const size_t head = reinterpret_cast<char *>(w.part_ml) - reinterpret_cast<char *>(base);
    st = cuda_status(cudaMemsetAsync(base, 0, head, (cudaStream_t)stream), fn);
    if (st != TT_OK) return st;
    return run(d, nullptr, g, w, q, k_ctx, v_ctx, ctx_lens, k_blk, v_blk, out, lse,
               (cudaStream_t)stream, fn);
}
