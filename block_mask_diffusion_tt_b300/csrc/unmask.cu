// unmask.cu -- confidence unmasking (one kernel) and the in-block loop driver.
//
// Method (keyframe.defihacklabs.io "Diffusion Nemotron", key point 3; 889990.xyz
// "NVIDIA发布Nemotron两塔模型", code example): per still-masked block position the
// argmax token and the confidence max softmax(l/T); commit positions with
// confidence >= gamma, at least the most confident one; re-mask the rest.
//
// Design (HBM-bound: every logit of every masked row is read exactly once):
//  * the vocabulary of every row is cut into units of 32 KB (16 or 8 KB only when
//    a batch has fewer units than CTAs); three persistent CTAs per SM walk the
//    units u = blockIdx.x + i * gridDim.x;
//  * in each CTA one producer thread streams the units through a ring of
//    shared-memory stages with TMA bulk copies (cp.async.bulk, full/empty
//    mbarriers), 64 KB per CTA in flight; a unit of a row that is not masked is
//    posted without data (rows that are not masked cost one byte of traffic);
//  * each of eight consumer warps takes an eighth of every unit from its stage
//    into registers (16-byte shared-memory loads, eight per lane), finds its
//    maximum M from a packed bf16x2 maximum (four max.bf16x2 per 8 logits, no
//    unpacking) and warp shuffles, then sums 2^((l - M) * log2(e)/T) and finds the
//    first index of M.  A vector whose maximum lies more than kSkipLog2 log2-units
//    below M adds under 2^-kSkipLog2 per element and is skipped after a packed
//    maximum; the few vectors near M are compacted into a list and exponentiated
//    one per lane.  The logits of a row that start off a 16-byte boundary are read
//    directly.  Each warp writes its own partial (M, index, sum) and moves on: no
//    barrier between warps, and no atomics, fences or counters, which would put a
//    round trip to L2 on every unit's path;
//  * a second kernel, launched as a programmatic dependent (its launch overlaps
//    the streaming kernel), runs one CTA per sequence: it merges each masked row's
//    partials into (token, conf) and applies the commit rule in one warp.  No CTA
//    waits for another.
#include <math.h>
#include <stdlib.h>

#include <chrono>
#include <mutex>
#include <thread>

#include "common.cuh"

namespace tt {
namespace {

constexpr int kMaxS = 64;
// A unit is cut into eighths, one per consumer warp.  Every consumer warp takes every
// unit of the CTA, in order: a warp must never wait on a stage more than one phase
// ahead of the one it last consumed there (a parity wait cannot tell phase n from
// phase n + 2), which groups of warps taking alternate units over an odd number of
// stages would break.
constexpr int kConsumerWarps = 8;
constexpr int kParts = kConsumerWarps;  // partials per unit
constexpr int kConsumers = 32 * kConsumerWarps;
constexpr int kUThreads = kConsumers + 32;  // + one producer warp
// Ring shape by measurement on ragged16k (512 rows x 131072 bf16): three CTAs per SM
// with two 32 KB stages each took 31.8 us per call, two CTAs with three stages 33.3,
// one CTA with three 64 KB stages 32.5, three CTAs with four 16 KB stages 41.4.
constexpr int kRingBytes = 64 * 1024;       // shared-memory ring of one CTA
constexpr int kMaxUnitBytes = 32 * 1024;
constexpr int kMinUnitBytes = 8 * 1024;
constexpr int kMaxStages = kRingBytes / kMinUnitBytes;
constexpr int kCtasPerSm = 3;
// 16-byte vectors of a unit's eighth per lane (at the largest unit)
constexpr int kVecPerLane = kMaxUnitBytes / 16 / kParts / 32;
// Terms 2^((l - M) k) below 2^-kSkipLog2 are not added: a vector of logits whose
// largest element is that far below the unit maximum M contributes nothing.  The
// unit's own maximum term is 1, so the skipped mass is at most V * 2^-kSkipLog2 of
// the row's sum (1.2e-7 relative at V = 131072).
constexpr float kSkipLog2 = 40.f;
// Error word (first int of the workspace): a role that gave up on a wait.
constexpr int kErrProducer = 1, kErrConsumer = 2;

struct UnmaskArgs {
    const char *logits;
    int64_t row_bytes;  // bytes between consecutive (b,s) rows
    int B, S, V;
    int esize;   // 2 (bf16) or 4 (fp32)
    int unit;    // elements per unit
    int nch;     // units per row (each leaves kParts partials, one per consumer warp)
    int qv;      // 16-byte vectors per eighth of a unit
    int nunits;  // B*S*nch
    int step_r, step_c;  // a step of gridDim.x units: whole rows and remaining units
    int nst;     // ring stages (kRingBytes / unit bytes)
    float k;     // log2(e) / T
    float skip;  // kSkipLog2 / k: logits this far below a maximum add under 2^-kSkipLog2
    float threshold;
    int mask_id;
    int force;
    int32_t *tokens;
    uint8_t *is_masked;
    float *conf;
    uint8_t *committed_now;
    int32_t *remaining;
    float *part_m;  // [B*S][nch][kParts] partials: maximum, first index, sum
    int32_t *part_i;
    float *part_s;
    int *err_word;
    int step;
    int32_t *steps_used;      // nullable (loop only)
    int32_t *committed_step;  // nullable (loop only)
};

struct Acc {
    float m;  // raw maximum
    int i;    // first index attaining it
    float s;  // sum of 2^((l - m) * k)
};

__device__ __forceinline__ Acc acc_empty() { return Acc{-INFINITY, 0x7FFFFFFF, 0.f}; }

__device__ __forceinline__ Acc acc_merge(Acc a, Acc b, float k) {
    float M = fmaxf(a.m, b.m);
    Acc r;
    r.m = M;
    r.i = (a.m > b.m) ? a.i : ((b.m > a.m) ? b.i : min(a.i, b.i));
    if (M == -INFINITY) {
        r.s = 0.f;
    } else {
        float sa = a.s > 0.f ? a.s * ex2_approx((a.m - M) * k) : 0.f;
        float sb = b.s > 0.f ? b.s * ex2_approx((b.m - M) * k) : 0.f;
        r.s = sa + sb;
    }
    return r;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
__device__ __forceinline__ uint32_t hmax2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ int4 lds128(uint32_t addr) {
    int4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}
// The two element types of a logits row: 8 bf16 or 4 fp32 per 16-byte vector.
template <int ESIZE>
struct Elt;
template <>
struct Elt<2> {
    static constexpr int E = 8;
    static constexpr uint32_t kNegInf = 0xFF80FF80u;  // two bf16 -inf
    __device__ static float scalar(const char *row, int v) {
        const uint16_t b = __ldcs(reinterpret_cast<const unsigned short *>(row) + v);
        return __uint_as_float(static_cast<uint32_t>(b) << 16);
    }
    // packed running maximum: four max.bf16x2, no unpacking
    __device__ static void acc_max(uint32_t &m2, const int4 &q) {
        m2 = hmax2(m2, hmax2(hmax2(q.x, q.y), hmax2(q.z, q.w)));
    }
    __device__ static float finish_max(uint32_t m2) { return fmaxf(bf16_lo(m2), bf16_hi(m2)); }
    __device__ static float vec_max(const int4 &q) {
        return finish_max(hmax2(hmax2(q.x, q.y), hmax2(q.z, q.w)));
    }
    __device__ static void unpack(const int4 &q, float (&x)[8]) {
        x[0] = bf16_lo(q.x); x[1] = bf16_hi(q.x);
        x[2] = bf16_lo(q.y); x[3] = bf16_hi(q.y);
        x[4] = bf16_lo(q.z); x[5] = bf16_hi(q.z);
        x[6] = bf16_lo(q.w); x[7] = bf16_hi(q.w);
    }
};
template <>
struct Elt<4> {
    static constexpr int E = 4;
    static constexpr uint32_t kNegInf = 0xFF800000u;  // fp32 -inf
    __device__ static float scalar(const char *row, int v) {
        return __ldcs(reinterpret_cast<const float *>(row) + v);
    }
    __device__ static void acc_max(uint32_t &m2, const int4 &q) {
        m2 = __float_as_uint(fmax3(__uint_as_float(m2),
                                   fmax3(__int_as_float(q.x), __int_as_float(q.y),
                                         __int_as_float(q.z)),
                                   __int_as_float(q.w)));
    }
    __device__ static float finish_max(uint32_t m2) { return __uint_as_float(m2); }
    __device__ static float vec_max(const int4 &q) {
        return fmax3(__int_as_float(q.x), __int_as_float(q.y),
                     fmaxf(__int_as_float(q.z), __int_as_float(q.w)));
    }
    __device__ static void unpack(const int4 &q, float (&x)[8]) {
        x[0] = __int_as_float(q.x); x[1] = __int_as_float(q.y);
        x[2] = __int_as_float(q.z); x[3] = __int_as_float(q.w);
    }
};

// Where the logits of unit u lie: row, unit in the row, the element range
// [lo, hi), and the 16-byte-aligned body [v0, v0 + nvec*E) that the bulk copy
// brings into shared memory; elements [lo, v0) (head) and [tail0, hi) (tail), at
// most E-1 each, are read directly.
struct Unit {
    int row, c, lo, hi, v0, nvec, tail0;
    const char *rp;
};

// The units of one walk (u, u + step, u + 2*step ...) as (row, unit in row), kept
// by carries instead of a division per unit.
struct UnitWalk {
    int row, c;
    __device__ void start(const UnmaskArgs &p, int u) {
        row = u / p.nch;
        c = u - row * p.nch;
    }
    __device__ void advance(const UnmaskArgs &p, int dr, int dc) {
        row += dr;
        c += dc;
        if (c >= p.nch) {
            c -= p.nch;
            ++row;
        }
    }
};

template <int ESIZE>
__device__ __forceinline__ Unit unit_at(const UnmaskArgs &p, const UnitWalk &w) {
    constexpr int E = Elt<ESIZE>::E;
    Unit x;
    x.row = w.row;
    x.c = w.c;
    x.lo = x.c * p.unit;
    x.hi = min(p.V, x.lo + p.unit);
    x.rp = p.logits + static_cast<int64_t>(x.row) * p.row_bytes;
    const uintptr_t a = reinterpret_cast<uintptr_t>(x.rp) + static_cast<uintptr_t>(x.lo) * ESIZE;
    x.v0 = min(x.lo + static_cast<int>(((16 - (a & 15)) & 15) / ESIZE), x.hi);
    x.nvec = (x.hi - x.v0) / E;
    x.tail0 = x.v0 + x.nvec * E;
    return x;
}

// Commit rule for sequence b, run by one warp once every row's (conf, token) is in
// shared memory (sconf / stok, indexed by position).  Lane l holds positions l and
// l + 32.
__device__ void commit_sequence_warp(const UnmaskArgs &p, int b, const float *sconf,
                                     const int *stok, const uint8_t *smask) {
    const int lane = threadIdx.x & 31;
    const size_t base = static_cast<size_t>(b) * p.S;
    int msk[2], pass[2], tok[2];
    float cf[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int s = lane + 32 * h;
        msk[h] = pass[h] = tok[h] = 0;
        cf[h] = __int_as_float(0x7FC00000);
        if (s < p.S) {
            msk[h] = smask[s] ? 1 : 0;
            if (msk[h]) {
                cf[h] = sconf[s];
                tok[h] = stok[s];
                pass[h] = (p.force || cf[h] >= p.threshold) ? 1 : 0;
            }
        }
    }
    const int n_masked = __popc(__ballot_sync(~0u, msk[0])) + __popc(__ballot_sync(~0u, msk[1]));
    const int n_pass = __popc(__ballot_sync(~0u, pass[0])) + __popc(__ballot_sync(~0u, pass[1]));
    if (n_masked > 0 && n_pass == 0) {
        // the masked position of highest confidence, lowest position on ties
        float bc = -INFINITY;
        int bs = 0x7FFFFFFF;
#pragma unroll
        for (int h = 0; h < 2; ++h)
            if (msk[h] && (cf[h] > bc || (cf[h] == bc && lane + 32 * h < bs))) {
                bc = cf[h];
                bs = lane + 32 * h;
            }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float oc = __shfl_xor_sync(~0u, bc, off);
            const int os = __shfl_xor_sync(~0u, bs, off);
            if (oc > bc || (oc == bc && os < bs)) {
                bc = oc;
                bs = os;
            }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h)
            if (lane + 32 * h == bs) pass[h] = 1;
    }
    int n_commit = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int s = lane + 32 * h;
        if (s < p.S) {
            p.committed_now[base + s] = static_cast<uint8_t>(pass[h]);
            p.conf[base + s] = cf[h];
            if (msk[h]) {
                if (pass[h]) {
                    p.tokens[base + s] = tok[h];
                    p.is_masked[base + s] = 0;
                    if (p.committed_step) p.committed_step[base + s] = p.step;
                } else {
                    p.tokens[base + s] = p.mask_id;
                }
            }
        }
        n_commit += __popc(__ballot_sync(~0u, s < p.S && msk[h] && pass[h]));
    }
    if (lane == 0) {
        p.remaining[b] = n_masked - n_commit;
        if (p.steps_used && n_masked > 0) p.steps_used[b] += 1;
    }
}

// One CTA per sequence, launched as a programmatic dependent of unmask_kernel: once
// that grid has finished (griddepcontrol.wait), sixteen threads per row merge the
// row's kParts*nch partials (each a sixteenth of them, loads issued together, then
// four shuffle steps) into (conf, token), and warp 0 applies the commit rule.
constexpr int kCommitTpr = 16;  // threads per row
constexpr int kCommitThreads = kCommitTpr * kMaxS;
constexpr int kCommitBatch = 8;  // partials loaded together per thread
__global__ void __launch_bounds__(kCommitThreads) unmask_commit_kernel(const UnmaskArgs p) {
    __shared__ float sconf[kMaxS];
    __shared__ int stok[kMaxS];
    __shared__ uint8_t smask[kMaxS];
    const int b = blockIdx.x;
    const int s = threadIdx.x / kCommitTpr, sub = threadIdx.x % kCommitTpr;
    const int row = b * p.S + s;
    // is_masked is read before the wait: the streaming kernel does not write it, and
    // every earlier kernel on the stream finished before the streaming kernel began
    const bool live = s < p.S && p.is_masked[row];
    if (s < p.S && sub == 0) smask[s] = live ? 1 : 0;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int np = kParts * p.nch;
    Acc r = acc_empty();
    if (live) {
        const size_t base = static_cast<size_t>(row) * np;
        for (int c0 = sub; c0 < np; c0 += kCommitTpr * kCommitBatch) {
            Acc v[kCommitBatch];
#pragma unroll
            for (int i = 0; i < kCommitBatch; ++i) {
                const int c = c0 + kCommitTpr * i;
                v[i] = c < np ? Acc{p.part_m[base + c], p.part_i[base + c], p.part_s[base + c]}
                              : acc_empty();
            }
#pragma unroll
            for (int i = 0; i < kCommitBatch; ++i) r = acc_merge(r, v[i], p.k);
        }
    }
#pragma unroll
    for (int off = 1; off < kCommitTpr; off <<= 1) {
        Acc o;
        o.m = __shfl_xor_sync(~0u, r.m, off);
        o.i = __shfl_xor_sync(~0u, r.i, off);
        o.s = __shfl_xor_sync(~0u, r.s, off);
        r = acc_merge(r, o, p.k);
    }
    if (live && sub == 0) {
        sconf[s] = 1.0f / r.s;
        stok[s] = r.i;
    }
    __syncthreads();
    if (threadIdx.x < 32) commit_sequence_warp(p, b, sconf, stok, smask);
}

struct Ring {
    uint32_t data, bars;
    int *unit_of;  // per stage: the unit it holds (>= 0), or -1 for a unit of a row not masked
    volatile int *err;
    __device__ uint32_t stage(int i, int unit_bytes) const { return data + i * unit_bytes; }
    __device__ uint32_t full(int i) const { return bars + 8 * i; }
    __device__ uint32_t empty(int i) const { return bars + 8 * (kMaxStages + i); }
};

template <int ESIZE>
__device__ void unmask_producer(const UnmaskArgs &p, const Ring &rg) {
    const int lane = threadIdx.x & 31;
    const int unit_bytes = p.unit * ESIZE;
    const uint64_t policy = l2_evict_first();  // logits are read once
    int stage = 0;
    uint32_t phase = 0, issued = 0, last_par = 0;
    bool ok = true;
    // The masked flags of 32 units at a time, one load per lane, so the issuing
    // thread never waits on a global load before a copy.
    UnitWalk walk;
    walk.start(p, blockIdx.x);
    for (int i0 = 0; ok && blockIdx.x + i0 * gridDim.x < static_cast<unsigned>(p.nunits);
         i0 += 32) {
        const int u_lane = blockIdx.x + (i0 + lane) * gridDim.x;
        const int m = u_lane < p.nunits ? p.is_masked[u_lane / p.nch] : 0;
        const unsigned masked = __ballot_sync(~0u, m != 0);
        if (lane == 0) {
            for (int l = 0; l < 32; ++l, walk.advance(p, p.step_r, p.step_c)) {
                const int u = blockIdx.x + (i0 + l) * gridDim.x;
                if (u >= p.nunits) break;
                if (!mbar_wait_sleep(rg.empty(stage), phase ^ 1, rg.err, kErrProducer)) {
                    ok = false;
                    break;
                }
                const uint32_t full = rg.full(stage);
                const Unit x = unit_at<ESIZE>(p, walk);
                const uint32_t bytes = static_cast<uint32_t>(x.nvec) * 16u;
                const bool is_m = (masked >> l) & 1u;
                rg.unit_of[stage] = is_m ? u : -1;
                if (is_m && bytes > 0) {
                    mbar_expect_tx(full, bytes);
                    bulk_load(rg.stage(stage, unit_bytes),
                              x.rp + static_cast<size_t>(x.v0) * ESIZE, bytes, full, policy);
                } else {
                    mbar_arrive(full);
                }
                // the phase posted last on each stage, with data or not: a later post
                // without data moves the barrier on, so the drain below must wait for
                // the last post's parity, not the last copy's
                issued |= 1u << stage;
                last_par = (last_par & ~(1u << stage)) | (phase << stage);
                if (++stage == p.nst) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
        ok = __shfl_sync(~0u, ok ? 1 : 0, 0) != 0;
    }
    // no copy may still be landing when the CTA exits: wait for the last phase posted
    // on each stage (a phase posted without data is already complete)
    if (lane == 0)
        for (int st = 0; st < p.nst; ++st)
            if ((issued >> st & 1u) && !mbar_drain(rg.full(st), last_par >> st & 1u))
                atomicCAS(const_cast<int *>(rg.err), 0, kErrProducer);
}

// Consumer warp w takes eighth w of every unit of the CTA.  It waits for the unit's
// stage, loads its eighth into registers (kVecPerLane 16-byte vectors per lane) and
// reduces it on its own: a packed maximum and shuffles give its maximum M, then the
// sum of 2^((x - M) k) and the first index of M, which lane 0 stores as the unit's
// partial w; the stage is released (empty barrier of count 8) once the few vectors
// near M have been read again.  No barrier between warps: a warp whose wait gives
// up just leaves.
template <int ESIZE>
__device__ void unmask_consumer(const UnmaskArgs &p, const Ring &rg) {
    using T = Elt<ESIZE>;
    constexpr int E = T::E;
    const int lane = threadIdx.x & 31, q = threadIdx.x >> 5;
    const int unit_bytes = p.unit * ESIZE;
    const int4 ninf = make_int4(T::kNegInf, T::kNegInf, T::kNegInf, T::kNegInf);
    // indices (within the eighth) of the vectors this warp exponentiates
    __shared__ uint16_t flagged_all[kConsumerWarps][32 * kVecPerLane];
    uint16_t *flagged = flagged_all[q];
    const unsigned lt_mask = (1u << lane) - 1u;
    int stage = 0;
    uint32_t phase = 0;
    UnitWalk walk;
    walk.start(p, blockIdx.x);
    for (int u = blockIdx.x; u < p.nunits; u += gridDim.x, walk.advance(p, p.step_r, p.step_c)) {
        if (!warp_wait_sleep(rg.full(stage), phase, rg.err, kErrConsumer)) return;
        const bool work = rg.unit_of[stage] >= 0;  // a masked row's unit
        const uint32_t base = rg.stage(stage, unit_bytes);
        const Unit x = unit_at<ESIZE>(p, walk);
        const int j0 = q * p.qv;  // first vector of this eighth
        int4 v4[kVecPerLane];
#pragma unroll
        for (int k = 0; k < kVecPerLane; ++k) {
            const int jj = lane + 32 * k;
            v4[k] = (work && jj < p.qv && j0 + jj < x.nvec) ? lds128(base + 16 * (j0 + jj)) : ninf;
        }
        const int cur = stage;
        if (++stage == p.nst) {
            stage = 0;
            phase ^= 1;
        }
        if (!work) {
            __syncwarp();
            if (lane == 0) mbar_arrive(rg.empty(cur));
            continue;
        }
        // elements before the first 16-byte boundary go with eighth 0, those after
        // the last whole vector with eighth 7
        float xh = -INFINITY, xt = -INFINITY;
        if (q == 0 && x.lo + lane < x.v0) xh = T::scalar(x.rp, x.lo + lane);
        if (q == kParts - 1 && x.tail0 + lane < x.hi) xt = T::scalar(x.rp, x.tail0 + lane);
        uint32_t m2 = T::kNegInf;
#pragma unroll
        for (int k = 0; k < kVecPerLane; ++k) T::acc_max(m2, v4[k]);
        const float tmax = fmax3(T::finish_max(m2), xh, xt);
        float M = tmax;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(~0u, M, off));
        // sum of 2^((x - M) k) over the elements that matter and the first index of M
        // (an eighth that is all -inf adds nothing).  Only vectors whose maximum is at
        // least thr are exponentiated; they are compacted first (their indices into a
        // per-warp list), so that the warp exponentiates them together, one vector per
        // lane, instead of once for every vector slot in which some lane has one.
        float sum = 0.f;
        int idx = 0x7FFFFFFF;
        const float thr = M - p.skip;  // elements below thr add under 2^-kSkipLog2
        if (M != -INFINITY) {
            if (xh >= thr) {
                sum += ex2_approx((xh - M) * p.k);
                if (xh == M) idx = x.lo + lane;
            }
            if (xt >= thr) {
                sum += ex2_approx((xt - M) * p.k);
                if (xt == M) idx = min(idx, x.tail0 + lane);
            }
            int nflag = 0;
#pragma unroll
            for (int k = 0; k < kVecPerLane; ++k) {
                const bool f = T::vec_max(v4[k]) >= thr;
                const unsigned bal = __ballot_sync(~0u, f);
                if (f) flagged[nflag + __popc(bal & lt_mask)] = static_cast<uint16_t>(lane + 32 * k);
                nflag += __popc(bal);
            }
            __syncwarp();
            // (x - M) k for pairs of logits as x k - hi - lo, with hi + lo = M k exactly
            // (hi = M k rounded, lo its rounding error): one rounding, on a result
            // near 0, where a product M k rounded once would shift every exponent
            const float mk_hi = M * p.k;
            const float mk_lo = fmaf(M, p.k, -mk_hi);
            const uint64_t kk = pk2(p.k, p.k), nhi = pk2(-mk_hi, -mk_hi),
                           nlo = pk2(-mk_lo, -mk_lo);
            uint64_t acc2 = pk2(0.f, 0.f);
            for (int r = lane; r < nflag; r += 32) {
                const int jv = j0 + flagged[r];
                const int4 qv = lds128(base + 16 * jv);
                float v[8];
                T::unpack(qv, v);
#pragma unroll
                for (int e = 0; e < E; e += 2) {
                    float y0, y1;
                    upk2(fadd2(ffma2(pk2(v[e], v[e + 1]), kk, nhi), nlo), y0, y1);
                    acc2 = fadd2(acc2, pk2(ex2_approx(y0), ex2_approx(y1)));
                }
                if (T::vec_max(qv) == M) {
                    int e0 = E - 1;
#pragma unroll
                    for (int e = E - 1; e >= 0; --e)
                        if (v[e] == M) e0 = e;
                    idx = min(idx, x.v0 + jv * E + e0);
                }
            }
            float a0, a1;
            upk2(acc2, a0, a1);
            sum += a0 + a1;
        }
        // this warp is done with the stage
        __syncwarp();
        if (lane == 0) mbar_arrive(rg.empty(cur));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            sum += __shfl_xor_sync(~0u, sum, off);
            idx = min(idx, __shfl_xor_sync(~0u, idx, off));
        }
        if (lane == 0) {  // merged by unmask_commit_kernel
            const size_t slot = (static_cast<size_t>(x.row) * p.nch + x.c) * kParts + q;
            p.part_m[slot] = M;
            p.part_i[slot] = idx;
            p.part_s[slot] = sum;
        }
    }
}

template <int ESIZE>
__global__ void __launch_bounds__(kUThreads, kCtasPerSm) unmask_kernel(const UnmaskArgs p) {
    // the commit kernel (programmatic dependent launch) may be scheduled now; it waits
    // for this grid to finish before it reads anything
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t bars[2 * kMaxStages];
    __shared__ int unit_of[kMaxStages];
    __shared__ int err;
    Ring rg;
    rg.data = smem_u32(smem);
    rg.bars = smem_u32(bars);
    rg.unit_of = unit_of;
    rg.err = &err;
    if (threadIdx.x == 0) {
        for (int i = 0; i < p.nst; ++i) {
            mbar_init(rg.full(i), 1);
            mbar_init(rg.empty(i), kConsumerWarps);
        }
        err = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x >= kConsumers)
        unmask_producer<ESIZE>(p, rg);
    else
        unmask_consumer<ESIZE>(p, rg);
    __syncthreads();
    if (threadIdx.x == 0 && err) atomicOr(p.err_word, err);
}

__global__ void block_init_kernel(int n, int S, int mask_id, int32_t *tokens, uint8_t *is_masked,
                                  int32_t *steps_used, int32_t *committed_step,
                                  const uint8_t *active) {
    int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    tokens[i] = mask_id;
    is_masked[i] = (active == nullptr || active[i / S] != 0) ? 1 : 0;
    if (committed_step) committed_step[i] = -1;
    if (steps_used && i % S == 0) steps_used[i / S] = 0;
}

__global__ void count_masked_kernel(int B, int S, const uint8_t *is_masked, int32_t *remaining) {
    int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    int n = 0;
    for (int s = 0; s < S; ++s) n += is_masked[static_cast<size_t>(b) * S + s] ? 1 : 0;
    remaining[b] = n;
}

// ---------------------------------------------------------------- host
struct Plan {
    int unit;  // elements per unit
    int nch;   // units per row
    int nst;   // ring stages
    int grid;  // CTAs
};

// Units of 32 KB, or 16 / 8 KB when a batch has fewer units than CTAs (three per
// SM).  Larger units win even for small batches: one CUDA-graph call on 128 rows x
// 131072 bf16 took 10.5 us with 32 KB units against 14.6 us with the 8 KB units that
// giving every CTA four units would take (64 rows: 8.0 against 15.3 us).
Plan plan_for(const tt_unmask_desc *d) {
    const int es = d->logits_dtype == TT_F32 ? 4 : 2;
    const int64_t rows = static_cast<int64_t>(d->B) * d->S;
    int sms = sm_count();
    if (sms <= 0) sms = 148;
    const int64_t ctas = static_cast<int64_t>(kCtasPerSm) * sms;
    int bytes = kMaxUnitBytes;
    while (bytes > kMinUnitBytes) {
        const int64_t unit = bytes / es;
        if (rows * ((d->V + unit - 1) / unit) >= ctas) break;
        bytes >>= 1;
    }
    Plan pl;
    pl.unit = bytes / es;
    pl.nch = static_cast<int>((static_cast<int64_t>(d->V) + pl.unit - 1) / pl.unit);
    pl.nst = kRingBytes / bytes;
    const int64_t units = rows * pl.nch;
    pl.grid = static_cast<int>(units < ctas ? units : ctas);
    return pl;
}

struct UnmaskWs {
    int *err_word;
    float *part_m;
    int32_t *part_i;
    float *part_s;
    size_t bytes;
};

// The error word comes first, so that a loop workspace (which starts with an
// unmask workspace) has it at the same place.
UnmaskWs carve_unmask(void *ws, int B, int S, int nch) {
    Carve c(ws);
    UnmaskWs w;
    const size_t rows = static_cast<size_t>(B) * S;
    w.err_word = c.take<int>(1);
    w.part_m = c.take<float>(rows * nch * kParts);
    w.part_i = c.take<int32_t>(rows * nch * kParts);
    w.part_s = c.take<float>(rows * nch * kParts);
    w.bytes = c.bytes();
    return w;
}

tt_status validate_desc(const tt_unmask_desc *d, const char *fn) {
    if (!d) return fail(TT_ERR_INVALID_ARG, "%s: null desc", fn);
    if (d->B < 0) return fail(TT_ERR_INVALID_ARG, "%s: B=%d < 0", fn, d->B);
    if (d->S < 1 || d->S > kMaxS)
        return fail(d->S < 1 ? TT_ERR_INVALID_ARG : TT_ERR_UNSUPPORTED, "%s: S=%d outside 1..%d", fn,
                    d->S, kMaxS);
    if (d->V < 1) return fail(TT_ERR_INVALID_ARG, "%s: V=%d < 1", fn, d->V);
    if (d->logits_dtype != TT_F32 && d->logits_dtype != TT_BF16)
        return fail(TT_ERR_INVALID_ARG, "%s: unknown logits dtype %d", fn, (int)d->logits_dtype);
    if (!(d->temperature > 0.f) || !isfinite(d->temperature))
        return fail(TT_ERR_INVALID_ARG, "%s: temperature must be finite and > 0", fn);
    if (isnan(d->threshold)) return fail(TT_ERR_INVALID_ARG, "%s: threshold is NaN", fn);
    if (d->logits_row_stride != 0 && d->logits_row_stride < d->V)
        return fail(TT_ERR_INVALID_ARG, "%s: logits_row_stride < V", fn);
    const double units = static_cast<double>(d->B) * d->S * plan_for(d).nch;
    if (units > 2147483647.0) return fail(TT_ERR_UNSUPPORTED, "%s: B*S too large", fn);
    return TT_OK;
}

template <int ESIZE>
tt_status launch_kernel(const UnmaskArgs &a, const Plan &pl, cudaStream_t stream) {
    static std::once_flag once[64];
    static cudaError_t set_err[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64) {
        std::call_once(once[dev], [dev] {
            set_err[dev] = cudaFuncSetAttribute(
                unmask_kernel<ESIZE>, cudaFuncAttributeMaxDynamicSharedMemorySize, kRingBytes);
        });
        if (set_err[dev] != cudaSuccess)
            return cuda_status(set_err[dev], "tt_confidence_unmask: smem attribute");
    }
    if (a.nunits > 0) {
        unmask_kernel<ESIZE><<<pl.grid, kUThreads, kRingBytes, stream>>>(a);
        tt_status st = cuda_status(cudaGetLastError(), "tt_confidence_unmask launch");
        if (st != TT_OK) return st;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.B));
    cfg.blockDim = dim3(kCommitThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cuda_status(cudaLaunchKernelEx(&cfg, unmask_commit_kernel, a),
                       "tt_confidence_unmask commit launch");
}

tt_status launch_unmask(const tt_unmask_desc *d, const void *logits, int32_t *tokens,
                        uint8_t *is_masked, float *conf, uint8_t *committed_now,
                        int32_t *remaining, int force, const UnmaskWs &w, int step,
                        int32_t *steps_used, int32_t *committed_step, cudaStream_t stream) {
    const Plan pl = plan_for(d);
    UnmaskArgs a;
    a.logits = static_cast<const char *>(logits);
    a.esize = d->logits_dtype == TT_F32 ? 4 : 2;
    a.row_bytes = (d->logits_row_stride ? d->logits_row_stride : d->V) * a.esize;
    a.B = d->B;
    a.S = d->S;
    a.V = d->V;
    a.unit = pl.unit;
    a.nch = pl.nch;
    a.qv = pl.unit * a.esize / 16 / kParts;
    a.step_r = pl.grid / pl.nch;
    a.step_c = pl.grid % pl.nch;
    a.nunits = d->B * d->S * pl.nch;
    a.nst = pl.nst;
    a.k = static_cast<float>(1.4426950408889634 / static_cast<double>(d->temperature));
    a.skip = static_cast<float>(kSkipLog2 * static_cast<double>(d->temperature) / 1.4426950408889634);
    a.threshold = d->threshold;
    a.mask_id = d->mask_token_id;
    a.force = force ? 1 : 0;
    a.tokens = tokens;
    a.is_masked = is_masked;
    a.conf = conf;
    a.committed_now = committed_now;
    a.remaining = remaining;
    a.part_m = w.part_m;
    a.part_i = w.part_i;
    a.part_s = w.part_s;
    a.err_word = w.err_word;
    a.step = step;
    a.steps_used = steps_used;
    a.committed_step = committed_step;
    return a.esize == 2 ? launch_kernel<2>(a, pl, stream) : launch_kernel<4>(a, pl, stream);
}

tt_status check_ptrs_unmask(const tt_unmask_desc *d, const void *logits, const void *tokens,
                            const void *is_masked, const char *fn) {
    if (d->B == 0) return TT_OK;
    if (!logits || !tokens || !is_masked) return fail(TT_ERR_INVALID_ARG, "%s: null pointer", fn);
    const size_t es = d->logits_dtype == TT_F32 ? 4 : 2;
    if (reinterpret_cast<uintptr_t>(logits) % es)
        return fail(TT_ERR_INVALID_ARG, "%s: logits not aligned to its element size", fn);
    if (reinterpret_cast<uintptr_t>(tokens) % 4)
        return fail(TT_ERR_INVALID_ARG, "%s: tokens not 4-byte aligned", fn);
    return TT_OK;
}

struct PinnedInts {
    int32_t *p = nullptr;
    size_t n = 0;
    ~PinnedInts() {
        if (p) cudaFreeHost(p);
    }
};

size_t loop_ws_bytes(const tt_unmask_desc *d) {
    Carve c(nullptr);
    const size_t rows = static_cast<size_t>(d->B) * d->S;
    c.take<char>(carve_unmask(nullptr, d->B, d->S, plan_for(d).nch).bytes);
    c.take<float>(rows);
    c.take<uint8_t>(rows);
    c.take<int32_t>(static_cast<size_t>(d->B));
    return c.bytes();
}

}  // namespace

// The in-block iteration behind tt_denoise_block_loop and tt_generate_blocks.
tt_status run_block_loop(const tt_unmask_desc *d, int32_t steps_per_block, int32_t start_step,
                         int32_t stop_step, const LoopProducer &prod, void *logits_buf,
                         int32_t *tokens, uint8_t *is_masked, int32_t *steps_used,
                         int32_t *committed_step, const uint8_t *init_active, void *workspace,
                         size_t workspace_bytes, cudaStream_t stream, int32_t timeout_ms,
                         int32_t *steps_run, const char *fn) {
    if (steps_run) *steps_run = 0;
    tt_status st = validate_desc(d, fn);
    if (st != TT_OK) return st;
    if (steps_per_block < 1) return fail(TT_ERR_INVALID_ARG, "%s: steps_per_block < 1", fn);
    if (start_step < 0 || start_step > steps_per_block)
        return fail(TT_ERR_INVALID_ARG, "%s: start_step outside [0, steps_per_block]", fn);
    if (!prod.fn) return fail(TT_ERR_INVALID_ARG, "%s: null producer", fn);
    if ((st = check_ptrs_unmask(d, logits_buf, tokens, is_masked, fn)) != TT_OK) return st;
    if (d->B == 0) return TT_OK;
    if (!steps_used || reinterpret_cast<uintptr_t>(steps_used) % 4)
        return fail(TT_ERR_INVALID_ARG, "%s: steps_used null or misaligned", fn);
    const int stop = (stop_step <= 0 || stop_step > steps_per_block) ? steps_per_block : stop_step;
    const size_t rows = static_cast<size_t>(d->B) * d->S;
    Carve c(workspace);
    const int nch = plan_for(d).nch;
    char *uw = c.take<char>(carve_unmask(nullptr, d->B, d->S, nch).bytes);
    float *conf = c.take<float>(rows);
    uint8_t *now = c.take<uint8_t>(rows);
    int32_t *remaining = c.take<int32_t>(static_cast<size_t>(d->B));
    if (!workspace || workspace_bytes < c.bytes())
        return fail(TT_ERR_WORKSPACE, "%s: workspace of %zu bytes, %zu needed", fn, workspace_bytes,
                    c.bytes());
    if (reinterpret_cast<uintptr_t>(workspace) % 256)
        return fail(TT_ERR_WORKSPACE, "%s: workspace not 256-byte aligned", fn);
    UnmaskWs w = carve_unmask(uw, d->B, d->S, nch);

    // per-thread pinned host buffer for the per-step remaining counts and error word
    thread_local PinnedInts host;
    const size_t need = static_cast<size_t>(d->B) + 1;
    if (host.n < need) {
        if (host.p) cudaFreeHost(host.p);
        host.p = nullptr;
        host.n = 0;
        if ((st = cuda_status(cudaMallocHost(&host.p, sizeof(int32_t) * need), fn)) != TT_OK)
            return st;
        host.n = need;
    }
    cudaEvent_t ev;
    if ((st = cuda_status(cudaEventCreateWithFlags(&ev, cudaEventDisableTiming), fn)) != TT_OK)
        return st;
    const int64_t limit_us = static_cast<int64_t>(timeout_ms > 0 ? timeout_ms : 60000) * 1000;

    // waits for the step, then returns the number of masked positions left
    auto wait_remaining = [&](int64_t *left) -> tt_status {
        tt_status s2 = cuda_status(cudaMemcpyAsync(host.p, remaining, sizeof(int32_t) * d->B,
                                                   cudaMemcpyDeviceToHost, stream), fn);
        if (s2 != TT_OK) return s2;
        s2 = cuda_status(cudaMemcpyAsync(host.p + d->B, w.err_word, sizeof(int32_t),
                                         cudaMemcpyDeviceToHost, stream), fn);
        if (s2 != TT_OK) return s2;
        if ((s2 = cuda_status(cudaEventRecord(ev, stream), fn)) != TT_OK) return s2;
        const auto t0 = std::chrono::steady_clock::now();
        for (int spin = 0;; ++spin) {
            cudaError_t q = cudaEventQuery(ev);
            if (q == cudaSuccess) break;
            if (q != cudaErrorNotReady) return cuda_status(q, fn);
            const int64_t us = std::chrono::duration_cast<std::chrono::microseconds>(
                                   std::chrono::steady_clock::now() - t0).count();
            if (us > limit_us)
                return fail(TT_ERR_TIMEOUT, "%s: device step not finished after %d ms", fn,
                            timeout_ms > 0 ? timeout_ms : 60000);
            if (spin > 64) std::this_thread::sleep_for(std::chrono::microseconds(20));
            else std::this_thread::yield();
        }
        if (host.p[d->B] != 0)
            return fail(TT_ERR_INTERNAL, "%s: the unmask kernel gave up on a wait (error word %d)",
                        fn, host.p[d->B]);
        int64_t n = 0;
        for (int b = 0; b < d->B; ++b) n += host.p[b];
        *left = n;
        return TT_OK;
    };

    int32_t done_steps = 0;
    int64_t left = 0;
    if (start_step == 0) {
        const int n = static_cast<int>(rows);
        block_init_kernel<<<(n + 255) / 256, 256, 0, stream>>>(n, d->S, d->mask_token_id, tokens,
                                                               is_masked, steps_used,
                                                               committed_step, init_active);
        st = cuda_status(cudaGetLastError(), fn);
        left = static_cast<int64_t>(rows);
        if (st == TT_OK && init_active) {  // sequences that take no part start with nothing masked
            count_masked_kernel<<<(d->B + 127) / 128, 128, 0, stream>>>(d->B, d->S, is_masked,
                                                                         remaining);
            st = cuda_status(cudaGetLastError(), fn);
            if (st == TT_OK) st = wait_remaining(&left);
        }
    } else {
        count_masked_kernel<<<(d->B + 127) / 128, 128, 0, stream>>>(d->B, d->S, is_masked,
                                                                     remaining);
        st = cuda_status(cudaGetLastError(), fn);
        if (st == TT_OK) st = wait_remaining(&left);
    }
    for (int k = start_step; st == TT_OK && k < stop && left > 0; ++k) {
        tt_status ps = prod.fn(prod.ctx, k, tokens, is_masked, logits_buf, (tt_stream_t)stream);
        if (ps != TT_OK) {
            st = fail(TT_ERR_CALLBACK, "%s: producer returned %s at step %d", fn,
                      tt_status_string(ps), k);
            break;
        }
        st = launch_unmask(d, logits_buf, tokens, is_masked, conf, now, remaining,
                           k == steps_per_block - 1, w, k, steps_used, committed_step, stream);
        if (st != TT_OK) break;
        st = wait_remaining(&left);
        if (st == TT_OK) ++done_steps;
    }
    cudaEventDestroy(ev);
    if (steps_run) *steps_run = done_steps;
    return st;
}

size_t block_loop_workspace_bytes(const tt_unmask_desc *d) {
    return validate_desc(d, "block loop workspace") == TT_OK ? loop_ws_bytes(d) : 0;
}

}  // namespace tt

using namespace tt;

namespace {
struct UserProducer {
    tt_logits_fn fn;
    void *user;
};
tt_status call_user_producer(void *ctx, int32_t step, const int32_t *tokens,
                             const uint8_t *is_masked, void *logits, tt_stream_t stream) {
    const UserProducer *u = static_cast<const UserProducer *>(ctx);
    return u->fn(u->user, step, tokens, is_masked, logits, stream);
}
}  // namespace

extern "C" {

size_t tt_confidence_unmask_workspace_size(const tt_unmask_desc *d) {
    if (validate_desc(d, "tt_confidence_unmask_workspace_size") != TT_OK) return 0;
    return carve_unmask(nullptr, d->B, d->S, plan_for(d).nch).bytes;
}

tt_status tt_confidence_unmask(const tt_unmask_desc *d, const void *logits, int32_t *tokens,
                               uint8_t *is_masked, float *conf, uint8_t *committed_now,
                               int32_t *remaining, int32_t force_commit_all, void *workspace,
                               size_t workspace_bytes, tt_stream_t stream) {
    const char *fn = "tt_confidence_unmask";
    tt_status st = validate_desc(d, fn);
    if (st != TT_OK) return st;
    if ((st = check_ptrs_unmask(d, logits, tokens, is_masked, fn)) != TT_OK) return st;
    if (d->B == 0) return TT_OK;
    if (!conf || !committed_now || !remaining) return fail(TT_ERR_INVALID_ARG, "%s: null output", fn);
    if (reinterpret_cast<uintptr_t>(conf) % 4 || reinterpret_cast<uintptr_t>(remaining) % 4)
        return fail(TT_ERR_INVALID_ARG, "%s: conf/remaining not 4-byte aligned", fn);
    const int nch = plan_for(d).nch;
    UnmaskWs w = carve_unmask(workspace, d->B, d->S, nch);
    if (!workspace || workspace_bytes < w.bytes)
        return fail(TT_ERR_WORKSPACE, "%s: workspace of %zu bytes, %zu needed", fn, workspace_bytes,
                    w.bytes);
    if (reinterpret_cast<uintptr_t>(workspace) % 256)
        return fail(TT_ERR_WORKSPACE, "%s: workspace not 256-byte aligned", fn);
    return launch_unmask(d, logits, tokens, is_masked, conf, committed_now, remaining,
                         force_commit_all, w, 0, nullptr, nullptr, (cudaStream_t)stream);
}

tt_status tt_confidence_unmask_error(const void *workspace, int32_t *flag_out,
                                     tt_stream_t stream) {
    if (!workspace || !flag_out)
        return fail(TT_ERR_INVALID_ARG, "tt_confidence_unmask_error: null pointer");
    cudaError_t e = cudaMemcpyAsync(flag_out, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost,
                                    (cudaStream_t)stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
    return cuda_status(e, "tt_confidence_unmask_error");
}

tt_status tt_block_init(const tt_unmask_desc *d, int32_t *tokens, uint8_t *is_masked,
                        int32_t *steps_used, int32_t *committed_step, tt_stream_t stream) {
    const char *fn = "tt_block_init";
    if (!d) return fail(TT_ERR_INVALID_ARG, "%s: null desc", fn);
    if (d->B < 0 || d->S < 1) return fail(TT_ERR_INVALID_ARG, "%s: bad B or S", fn);
    if (d->B == 0) return TT_OK;
    if (!tokens || !is_masked) return fail(TT_ERR_INVALID_ARG, "%s: null pointer", fn);
    const int64_t n = static_cast<int64_t>(d->B) * d->S;
    if (n > 2147483647LL) return fail(TT_ERR_UNSUPPORTED, "%s: B*S too large", fn);
    block_init_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, (cudaStream_t)stream>>>(
        static_cast<int>(n), d->S, d->mask_token_id, tokens, is_masked, steps_used, committed_step,
        nullptr);
    return cuda_status(cudaGetLastError(), fn);
}

size_t tt_denoise_block_loop_workspace_size(const tt_unmask_desc *d) {
    if (validate_desc(d, "tt_denoise_block_loop_workspace_size") != TT_OK) return 0;
    return loop_ws_bytes(d);
}

tt_status tt_denoise_block_loop(const tt_unmask_desc *d, int32_t steps_per_block,
                                int32_t start_step, int32_t stop_step, tt_logits_fn producer,
                                void *user, void *logits_buf, int32_t *tokens,
                                uint8_t *is_masked, int32_t *steps_used, int32_t *committed_step,
                                void *workspace, size_t workspace_bytes, tt_stream_t stream,
                                int32_t timeout_ms, int32_t *steps_run) {
    UserProducer up{producer, user};
    LoopProducer prod{producer ? call_user_producer : nullptr, &up};
    return run_block_loop(d, steps_per_block, start_step, stop_step, prod, logits_buf, tokens,
                          is_masked, steps_used, committed_step, nullptr, workspace,
                          workspace_bytes, (cudaStream_t)stream, timeout_ms, steps_run,
                          "tt_denoise_block_loop");
}

}  // extern "C"
