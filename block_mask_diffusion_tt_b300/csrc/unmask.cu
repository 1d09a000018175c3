// unmask.cu -- confidence unmasking (one kernel) and the in-block loop driver.
//
// Method (keyframe.defihacklabs.io "Diffusion Nemotron", key point 3; 889990.xyz
// "NVIDIA发布Nemotron两塔模型", code example): per still-masked block position the
// argmax token and the confidence max softmax(l/T); commit positions with
// confidence >= gamma, at least the most confident one; re-mask the rest.
//
// Design (HBM-bound: every logit of every masked row is read exactly once):
//  * grid = (B*S rows) x (nch vocabulary chunks), 256 threads per CTA; a CTA
//    whose row is not masked returns after one arrival (rows that are not masked
//    cost one byte of traffic);
//  * one pass over the chunk with 16-byte streaming loads, four in flight per
//    thread; per thread a running raw-logit maximum, its first index and
//    sum 2^((l - max) * log2(e)/T), rescaled when the maximum grows; a vector of
//    8 logits whose maximum lies 2^40 below the running maximum's term adds
//    nothing and costs no exponentials (bounded below, at kSkipLog2);
//  * warp-shuffle then shared-memory merge to one partial per CTA; the last CTA
//    of a row (arrival counter) merges the row's nch partials into (token, conf);
//  * the last row of a sequence to arrive (counter over all S rows, masked or
//    not) applies the commit rule for that sequence.  No CTA ever waits for
//    another; counters are reset by the CTA that consumes them.
#include <math.h>
#include <stdlib.h>

#include <chrono>
#include <thread>

#include "common.cuh"

namespace tt {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxS = 64;
// Loads in flight per thread.  Four keep the kernel at 40 registers, so six CTAs fit
// on an SM; measured faster than eight, twelve or sixteen, which fit fewer CTAs.
constexpr int kUnroll = 4;
// Terms 2^((l - m) k) below 2^-kSkipLog2 of the running maximum's term are not
// added: a vector of logits whose largest element is that far below the running
// maximum contributes nothing.  The maximum is only ever raised, so every skipped
// term is below 2^-kSkipLog2 of the final sum's largest term, and the skipped mass
// is at most V * 2^-kSkipLog2 of the sum (1.2e-7 relative at V = 131072).
constexpr float kSkipLog2 = 40.f;

struct UnmaskArgs {
    const char *logits;
    int64_t row_stride;  // elements
    int B, S, V;
    int esize;  // 2 (bf16) or 4 (fp32)
    int nch, chunk;
    float k;  // log2(e) / T
    float threshold;
    int mask_id;
    int force;
    int32_t *tokens;
    uint8_t *is_masked;
    float *conf;
    uint8_t *committed_now;
    int32_t *remaining;
    float *part_m;
    int32_t *part_i;
    float *part_s;
    float *row_conf;
    int32_t *row_tok;
    unsigned *row_cnt;
    unsigned *seq_cnt;
    int step;
    int32_t *steps_used;      // nullable (loop only)
    int32_t *committed_step;  // nullable (loop only)
};

struct Acc {
    float m;  // running raw maximum
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

// Adds one element (index idx, value x) in increasing index order.
__device__ __forceinline__ void acc_add(Acc &a, float x, int idx, float k) {
    if (x > a.m) {
        a.s = (a.m == -INFINITY) ? 0.f : a.s * ex2_approx((a.m - x) * k);
        a.m = x;
        a.i = idx;
    }
    if (a.m != -INFINITY) a.s += ex2_approx((x - a.m) * k);
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Adds N (4 or 8) consecutive elements starting at index idx.
template <int N>
__device__ __forceinline__ void acc_add_vec(Acc &a, const float (&x)[N], int idx, float k) {
    float lm;
    if constexpr (N == 8)
        lm = fmax3(fmax3(x[0], x[1], x[2]), fmax3(x[3], x[4], x[5]), fmaxf(x[6], x[7]));
    else
        lm = fmax3(x[0], x[1], fmaxf(x[2], x[3]));
    if (lm > a.m) {
        int j0 = N - 1;
#pragma unroll
        for (int j = N - 1; j >= 0; --j)
            if (x[j] == lm) j0 = j;
        a.s = (a.m == -INFINITY) ? 0.f : a.s * ex2_approx((a.m - lm) * k);
        a.m = lm;
        a.i = idx + j0;
    }
    if (a.m != -INFINITY && (lm - a.m) * k > -kSkipLog2) {
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int j = 0; j < N; j += 2) {
            s0 += ex2_approx((x[j] - a.m) * k);
            s1 += ex2_approx((x[j + 1] - a.m) * k);
        }
        a.s += s0 + s1;
    }
}

__device__ __forceinline__ float load_scalar(const char *row, int v, int esize) {
    if (esize == 4) return __ldcs(reinterpret_cast<const float *>(row) + v);
    uint16_t b = __ldcs(reinterpret_cast<const unsigned short *>(row) + v);
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ void unpack(const int4 &q, int esize, float (&x)[8]) {
    if (esize == 2) {
        x[0] = bf16_lo(q.x); x[1] = bf16_hi(q.x);
        x[2] = bf16_lo(q.y); x[3] = bf16_hi(q.y);
        x[4] = bf16_lo(q.z); x[5] = bf16_hi(q.z);
        x[6] = bf16_lo(q.w); x[7] = bf16_hi(q.w);
    } else {
        x[0] = __int_as_float(q.x); x[1] = __int_as_float(q.y);
        x[2] = __int_as_float(q.z); x[3] = __int_as_float(q.w);
    }
}

template <int ESIZE>
__device__ Acc reduce_chunk(const UnmaskArgs &p, const char *row, int lo, int hi) {
    constexpr int E = 16 / ESIZE;  // elements per 16-byte vector
    Acc a = acc_empty();
    const int t = threadIdx.x;
    // head: elements before the first 16-byte boundary
    uintptr_t addr = reinterpret_cast<uintptr_t>(row) + static_cast<uintptr_t>(lo) * ESIZE;
    int head = static_cast<int>(((16 - (addr & 15)) & 15) / ESIZE);
    if (head > hi - lo) head = hi - lo;
    if (t < head) acc_add(a, load_scalar(row, lo + t, ESIZE), lo + t, p.k);
    const int v0 = lo + head;
    const int nvec = (hi - v0) / E;
    const int4 *vec = reinterpret_cast<const int4 *>(row + static_cast<size_t>(v0) * ESIZE);
    int j = t;
    for (; j + (kUnroll - 1) * kThreads < nvec; j += kUnroll * kThreads) {
        int4 q[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) q[u] = __ldcs(vec + j + u * kThreads);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            float x[8];
            unpack(q[u], ESIZE, x);
            if (ESIZE == 2) {
                acc_add_vec<8>(a, x, v0 + (j + u * kThreads) * E, p.k);
            } else {
                float y[4] = {x[0], x[1], x[2], x[3]};
                acc_add_vec<4>(a, y, v0 + (j + u * kThreads) * E, p.k);
            }
        }
    }
    for (; j < nvec; j += kThreads) {
        float x[8];
        unpack(__ldcs(vec + j), ESIZE, x);
        if (ESIZE == 2) {
            acc_add_vec<8>(a, x, v0 + j * E, p.k);
        } else {
            float y[4] = {x[0], x[1], x[2], x[3]};
            acc_add_vec<4>(a, y, v0 + j * E, p.k);
        }
    }
    // tail: the elements after the last whole vector
    const int vt = v0 + nvec * E;
    if (vt + t < hi) acc_add(a, load_scalar(row, vt + t, ESIZE), vt + t, p.k);
    return a;
}

__device__ __forceinline__ Acc warp_merge(Acc a, float k) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        Acc o;
        o.m = __shfl_xor_sync(0xFFFFFFFFu, a.m, off);
        o.i = __shfl_xor_sync(0xFFFFFFFFu, a.i, off);
        o.s = __shfl_xor_sync(0xFFFFFFFFu, a.s, off);
        a = acc_merge(a, o, k);
    }
    return a;
}

// Commit rule for sequence b; executed by one CTA after all S rows arrived.
__device__ void commit_sequence(const UnmaskArgs &p, int b) {
    __shared__ float sconf[kMaxS];
    __shared__ int spass[kMaxS];
    __shared__ int smask[kMaxS];
    const int t = threadIdx.x;
    const size_t base = static_cast<size_t>(b) * p.S;
    int msk = 0, pass = 0, tok = 0;
    float cf = __int_as_float(0x7FC00000);
    if (t < p.S) {
        msk = p.is_masked[base + t] ? 1 : 0;
        if (msk) {
            cf = __ldcg(p.row_conf + base + t);
            tok = __ldcg(p.row_tok + base + t);
            pass = (p.force || cf >= p.threshold) ? 1 : 0;
        }
        sconf[t] = cf;
        smask[t] = msk;
        spass[t] = pass;
    }
    const int n_masked = __syncthreads_count(msk);
    const int n_pass = __syncthreads_count(pass);
    if (n_masked > 0 && n_pass == 0 && t == 0) {
        int best = -1;
        for (int s = 0; s < p.S; ++s)
            if (smask[s] && (best < 0 || sconf[s] > sconf[best])) best = s;
        spass[best] = 1;
    }
    __syncthreads();
    if (t < p.S) {
        pass = spass[t];
        p.committed_now[base + t] = static_cast<uint8_t>(pass);
        p.conf[base + t] = cf;
        if (msk) {
            if (pass) {
                p.tokens[base + t] = tok;
                p.is_masked[base + t] = 0;
                if (p.committed_step) p.committed_step[base + t] = p.step;
            } else {
                p.tokens[base + t] = p.mask_id;
            }
        }
    }
    const int n_commit = __syncthreads_count(t < p.S && msk && pass);
    if (t == 0) {
        p.remaining[b] = n_masked - n_commit;
        if (p.steps_used && n_masked > 0) p.steps_used[b] += 1;
        p.seq_cnt[b] = 0;  // all S arrivals consumed: ready for the next launch
    }
}

// Arrival of one row of sequence b; the last of the S arrivals commits.
__device__ void arrive_sequence(const UnmaskArgs &p, int b) {
    __shared__ int last;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        unsigned old = atomicAdd(p.seq_cnt + b, 1u);
        last = (old == static_cast<unsigned>(p.S - 1));
        if (last) __threadfence();
    }
    __syncthreads();
    if (last) commit_sequence(p, b);
}

template <int ESIZE>
__global__ void __launch_bounds__(kThreads) unmask_kernel(const UnmaskArgs p) {
    const int u = blockIdx.x;
    const int row = u / p.nch;
    const int c = u - row * p.nch;
    const int b = row / p.S;
    if (!p.is_masked[row]) {
        if (c == 0) arrive_sequence(p, b);
        return;
    }
    const char *rp = p.logits + static_cast<size_t>(row) * p.row_stride * ESIZE;
    const int lo = c * p.chunk;
    const int hi = min(p.V, lo + p.chunk);
    Acc a = reduce_chunk<ESIZE>(p, rp, lo, hi);
    a = warp_merge(a, p.k);
    __shared__ Acc warp_acc[kThreads / 32];
    __shared__ int row_done;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) warp_acc[warp] = a;
    __syncthreads();
    if (warp == 0) {
        a = lane < kThreads / 32 ? warp_acc[lane] : acc_empty();
        a = warp_merge(a, p.k);
        if (p.nch == 1) {
            if (lane == 0) {
                p.row_conf[row] = 1.0f / a.s;
                p.row_tok[row] = a.i;
                row_done = 1;
            }
        } else {
            int last = 0;
            if (lane == 0) {
                const size_t slot = static_cast<size_t>(row) * p.nch + c;
                p.part_m[slot] = a.m;
                p.part_i[slot] = a.i;
                p.part_s[slot] = a.s;
                __threadfence();
                last = atomicAdd(p.row_cnt + row, 1u) == static_cast<unsigned>(p.nch - 1);
                if (last) __threadfence();
            }
            last = __shfl_sync(0xFFFFFFFFu, last, 0);
            if (last) {  // merge the row's nch partials
                Acc r = acc_empty();
                for (int cc = lane; cc < p.nch; cc += 32) {
                    const size_t slot = static_cast<size_t>(row) * p.nch + cc;
                    Acc o{__ldcg(p.part_m + slot), __ldcg(p.part_i + slot), __ldcg(p.part_s + slot)};
                    r = acc_merge(r, o, p.k);
                }
                r = warp_merge(r, p.k);
                if (lane == 0) {
                    p.row_conf[row] = 1.0f / r.s;
                    p.row_tok[row] = r.i;
                    p.row_cnt[row] = 0;
                }
            }
            if (lane == 0) row_done = last;
        }
    }
    __syncthreads();
    if (row_done) arrive_sequence(p, b);
}

__global__ void block_init_kernel(int n, int S, int mask_id, int32_t *tokens, uint8_t *is_masked,
                                  int32_t *steps_used, int32_t *committed_step) {
    int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    tokens[i] = mask_id;
    is_masked[i] = 1;
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
    int nch, chunk;
};

Plan plan_for(int V) {
    int nch = (V + 32767) / 32768;
    if (nch < 1) nch = 1;
    if (nch > 64) nch = 64;
    int chunk = (V + nch - 1) / nch;
    chunk = (chunk + 63) / 64 * 64;
    nch = (V + chunk - 1) / chunk;
    return Plan{nch, chunk};
}

struct UnmaskWs {
    float *part_m;
    int32_t *part_i;
    float *part_s;
    float *row_conf;
    int32_t *row_tok;
    unsigned *row_cnt;
    unsigned *seq_cnt;
    size_t bytes;
};

UnmaskWs carve_unmask(void *ws, int B, int S, int nch) {
    Carve c(ws);
    UnmaskWs w;
    const size_t rows = static_cast<size_t>(B) * S;
    w.row_cnt = c.take<unsigned>(rows);
    w.seq_cnt = c.take<unsigned>(static_cast<size_t>(B));
    w.part_m = c.take<float>(rows * nch);
    w.part_i = c.take<int32_t>(rows * nch);
    w.part_s = c.take<float>(rows * nch);
    w.row_conf = c.take<float>(rows);
    w.row_tok = c.take<int32_t>(rows);
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
    const double blocks = static_cast<double>(d->B) * d->S * plan_for(d->V).nch;
    if (blocks > 2147483647.0) return fail(TT_ERR_UNSUPPORTED, "%s: B*S too large", fn);
    return TT_OK;
}

tt_status launch_unmask(const tt_unmask_desc *d, const void *logits, int32_t *tokens,
                        uint8_t *is_masked, float *conf, uint8_t *committed_now,
                        int32_t *remaining, int force, const UnmaskWs &w, int step,
                        int32_t *steps_used, int32_t *committed_step, cudaStream_t stream) {
    const Plan pl = plan_for(d->V);
    UnmaskArgs a;
    a.logits = static_cast<const char *>(logits);
    a.row_stride = d->logits_row_stride ? d->logits_row_stride : d->V;
    a.B = d->B;
    a.S = d->S;
    a.V = d->V;
    a.esize = d->logits_dtype == TT_F32 ? 4 : 2;
    a.nch = pl.nch;
    a.chunk = pl.chunk;
    a.k = static_cast<float>(1.4426950408889634 / static_cast<double>(d->temperature));
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
    a.row_conf = w.row_conf;
    a.row_tok = w.row_tok;
    a.row_cnt = w.row_cnt;
    a.seq_cnt = w.seq_cnt;
    a.step = step;
    a.steps_used = steps_used;
    a.committed_step = committed_step;
    const unsigned grid = static_cast<unsigned>(d->B) * d->S * pl.nch;
    if (grid == 0) return TT_OK;
    if (a.esize == 2)
        unmask_kernel<2><<<grid, kThreads, 0, stream>>>(a);
    else
        unmask_kernel<4><<<grid, kThreads, 0, stream>>>(a);
    return cuda_status(cudaGetLastError(), "tt_confidence_unmask launch");
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

}  // namespace
}  // namespace tt

using namespace tt;

extern "C" {

size_t tt_confidence_unmask_workspace_size(const tt_unmask_desc *d) {
    if (validate_desc(d, "tt_confidence_unmask_workspace_size") != TT_OK) return 0;
    return carve_unmask(nullptr, d->B, d->S, plan_for(d->V).nch).bytes;
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
    const int nch = plan_for(d->V).nch;
    UnmaskWs w = carve_unmask(workspace, d->B, d->S, nch);
    if (!workspace || workspace_bytes < w.bytes)
        return fail(TT_ERR_WORKSPACE, "%s: workspace of %zu bytes, %zu needed", fn, workspace_bytes,
                    w.bytes);
    if (reinterpret_cast<uintptr_t>(workspace) % 256)
        return fail(TT_ERR_WORKSPACE, "%s: workspace not 256-byte aligned", fn);
    return launch_unmask(d, logits, tokens, is_masked, conf, committed_now, remaining,
                         force_commit_all, w, 0, nullptr, nullptr, (cudaStream_t)stream);
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
        static_cast<int>(n), d->S, d->mask_token_id, tokens, is_masked, steps_used, committed_step);
    return cuda_status(cudaGetLastError(), fn);
}

size_t tt_denoise_block_loop_workspace_size(const tt_unmask_desc *d) {
    if (validate_desc(d, "tt_denoise_block_loop_workspace_size") != TT_OK) return 0;
    Carve c(nullptr);
    const size_t rows = static_cast<size_t>(d->B) * d->S;
    c.take<char>(carve_unmask(nullptr, d->B, d->S, plan_for(d->V).nch).bytes);
    c.take<float>(rows);
    c.take<uint8_t>(rows);
    c.take<int32_t>(static_cast<size_t>(d->B));
    return c.bytes();
}

tt_status tt_denoise_block_loop(const tt_unmask_desc *d, int32_t steps_per_block,
                                int32_t start_step, int32_t stop_step, tt_logits_fn producer,
                                void *user, void *logits_buf, int32_t *tokens,
                                uint8_t *is_masked, int32_t *steps_used, int32_t *committed_step,
                                void *workspace, size_t workspace_bytes, tt_stream_t stream_,
                                int32_t timeout_ms, int32_t *steps_run) {
    const char *fn = "tt_denoise_block_loop";
    if (steps_run) *steps_run = 0;
    tt_status st = validate_desc(d, fn);
    if (st != TT_OK) return st;
    if (steps_per_block < 1) return fail(TT_ERR_INVALID_ARG, "%s: steps_per_block < 1", fn);
    if (start_step < 0 || start_step > steps_per_block)
        return fail(TT_ERR_INVALID_ARG, "%s: start_step outside [0, steps_per_block]", fn);
    if (!producer) return fail(TT_ERR_INVALID_ARG, "%s: null producer", fn);
    if ((st = check_ptrs_unmask(d, logits_buf, tokens, is_masked, fn)) != TT_OK) return st;
    if (d->B == 0) return TT_OK;
    if (!steps_used || reinterpret_cast<uintptr_t>(steps_used) % 4)
        return fail(TT_ERR_INVALID_ARG, "%s: steps_used null or misaligned", fn);
    const int stop = (stop_step <= 0 || stop_step > steps_per_block) ? steps_per_block : stop_step;
    const size_t rows = static_cast<size_t>(d->B) * d->S;
    Carve c(workspace);
    const int nch = plan_for(d->V).nch;
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
    cudaStream_t stream = (cudaStream_t)stream_;

    // per-thread pinned host buffer for the per-step remaining counts
    thread_local PinnedInts host;
    if (host.n < static_cast<size_t>(d->B)) {
        if (host.p) cudaFreeHost(host.p);
        host.p = nullptr;
        host.n = 0;
        if ((st = cuda_status(cudaMallocHost(&host.p, sizeof(int32_t) * d->B), fn)) != TT_OK)
            return st;
        host.n = static_cast<size_t>(d->B);
    }
    cudaEvent_t ev;
    if ((st = cuda_status(cudaEventCreateWithFlags(&ev, cudaEventDisableTiming), fn)) != TT_OK)
        return st;
    const int64_t limit_us = static_cast<int64_t>(timeout_ms > 0 ? timeout_ms : 60000) * 1000;

    // waits for `ev`, then returns the number of masked positions left
    auto wait_remaining = [&](int64_t *left) -> tt_status {
        tt_status s2 = cuda_status(cudaMemcpyAsync(host.p, remaining, sizeof(int32_t) * d->B,
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
                                                               committed_step);
        st = cuda_status(cudaGetLastError(), fn);
        left = static_cast<int64_t>(rows);
    } else {
        count_masked_kernel<<<(d->B + 127) / 128, 128, 0, stream>>>(d->B, d->S, is_masked,
                                                                     remaining);
        st = cuda_status(cudaGetLastError(), fn);
        if (st == TT_OK) st = wait_remaining(&left);
    }
    for (int k = start_step; st == TT_OK && k < stop && left > 0; ++k) {
        tt_status ps = producer(user, k, tokens, is_masked, logits_buf, stream_);
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

}  // extern "C"
