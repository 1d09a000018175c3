// generate.cu -- block-by-block generation: blocks of S positions are denoised one
// after another, and each finished block becomes context for the next.
//
// Method (dothoosh.com "فرآیند انتشار در برابر رمزگشایی متوالی در مدل جدید انویدیا",
// section "two-tower mechanism": the denoiser fills a block of masked positions step
// by step, the clean block goes to the context tower, the next block attends to the
// longer prefix; 889990.xyz "NVIDIA发布Nemotron两塔模型", section 训练与推理, code
// example: max_new_tokens, block_size, steps_per_block, eos_token_id).
//
// Per block: the in-block loop (run_block_loop, with only the sequences that are
// still generating masked), then one small kernel that keeps the block's tokens,
// finds EOS, updates lengths and the active flags and counts the sequences left,
// then -- if a next block follows -- the caller's K/V producer and tt_kv_append for
// the sequences that continue.  The host reads the count of sequences left once per
// block (the loop already waits once per step).
#include <chrono>
#include <thread>

#include "common.cuh"

namespace tt {
namespace {

constexpr int kFinishThreads = 256;

struct FinishArgs {
    int B, S, blk, max_new, eos, Lmax, more_blocks;
    const int32_t *tokens;     // [B, S] this block
    const int32_t *steps_used; // [B] this block
    int32_t *out;              // [B, max_new]
    int32_t *gen_len;          // [B]
    uint8_t *active;           // [B] in/out
    int32_t *steps_total;      // [B] or null
    const int32_t *ctx_lens;   // [B]
    int32_t *overflow;         // or null
    int32_t *n_active;         // device, written
};

// One CTA: for every sequence taking part in this block, keep the block's first
// `keep` tokens, stop at EOS, at max_new, or when the cache cannot take the block
// (overflow), and count the sequences that continue.
__global__ void __launch_bounds__(kFinishThreads) finish_block_kernel(const FinishArgs a) {
    __shared__ int left;
    if (threadIdx.x == 0) left = 0;
    __syncthreads();
    const int keep = min(a.S, a.max_new - a.blk * a.S);
    int mine = 0;
    for (int b = threadIdx.x; b < a.B; b += kFinishThreads) {
        if (!a.active[b]) continue;
        const int32_t *t = a.tokens + static_cast<size_t>(b) * a.S;
        int32_t *o = a.out + static_cast<size_t>(b) * a.max_new + static_cast<size_t>(a.blk) * a.S;
        int eos_at = -1;
        for (int s = 0; s < keep; ++s) {
            const int32_t v = t[s];
            o[s] = v;
            if (eos_at < 0 && a.eos >= 0 && v == a.eos) eos_at = s;
        }
        if (a.steps_total) a.steps_total[b] += a.steps_used[b];
        bool go = true;
        if (eos_at >= 0) {
            a.gen_len[b] = a.blk * a.S + eos_at + 1;
            go = false;
        } else {
            a.gen_len[b] = a.blk * a.S + keep;
            if (a.gen_len[b] == a.max_new) {
                go = false;
            } else if (a.more_blocks && a.ctx_lens[b] + a.S > a.Lmax) {
                go = false;  // the cache cannot take this block
                if (a.overflow) atomicAdd(a.overflow, 1);
            }
        }
        if (!go) a.active[b] = 0;
        mine += go ? 1 : 0;
    }
    if (mine) atomicAdd(&left, mine);
    __syncthreads();
    if (threadIdx.x == 0) *a.n_active = left;
}

__global__ void count_active_kernel(int B, const uint8_t *active, int32_t *n_active) {
    __shared__ int left;
    if (threadIdx.x == 0) left = 0;
    __syncthreads();
    int mine = 0;
    for (int b = threadIdx.x; b < B; b += blockDim.x) mine += active[b] ? 1 : 0;
    if (mine) atomicAdd(&left, mine);
    __syncthreads();
    if (threadIdx.x == 0) *n_active = left;
}

struct BlockProducer {
    tt_block_logits_fn fn;
    void *user;
    int32_t block;
};
tt_status call_block_producer(void *ctx, int32_t step, const int32_t *tokens,
                              const uint8_t *is_masked, void *logits, tt_stream_t stream) {
    const BlockProducer *p = static_cast<const BlockProducer *>(ctx);
    return p->fn(p->user, p->block, step, tokens, is_masked, logits, stream);
}

struct GenWs {
    char *loop;
    int32_t *tokens;
    uint8_t *is_masked;
    int32_t *steps_used;
    int32_t *n_active;
    size_t loop_bytes, bytes;
};

GenWs carve_gen(void *ws, const tt_unmask_desc *d) {
    Carve c(ws);
    GenWs w;
    const size_t rows = static_cast<size_t>(d->B) * d->S;
    w.loop_bytes = block_loop_workspace_bytes(d);
    w.loop = c.take<char>(w.loop_bytes);
    w.tokens = c.take<int32_t>(rows);
    w.is_masked = c.take<uint8_t>(rows);
    w.steps_used = c.take<int32_t>(static_cast<size_t>(d->B));
    w.n_active = c.take<int32_t>(1);
    w.bytes = c.bytes();
    return w;
}

struct PinnedInt {
    int32_t *p = nullptr;
    ~PinnedInt() {
        if (p) cudaFreeHost(p);
    }
};

}  // namespace
}  // namespace tt

using namespace tt;

extern "C" {

size_t tt_generate_blocks_workspace_size(const tt_unmask_desc *desc) {
    if (!desc || block_loop_workspace_bytes(desc) == 0) return 0;
    return carve_gen(nullptr, desc).bytes;
}

tt_status tt_generate_blocks(const tt_unmask_desc *desc, const tt_kv_desc *kv,
                             const tt_generate_params *gp, tt_block_logits_fn logits_fn,
                             void *logits_user, tt_block_kv_fn kv_fn, void *kv_user,
                             void *logits_buf, void *const *k_ctx, void *const *v_ctx,
                             int32_t *ctx_lens, void *const *k_blk, void *const *v_blk,
                             int32_t *out_tokens, int32_t *gen_len, uint8_t *active,
                             int32_t *steps_total, int32_t *overflow, void *workspace,
                             size_t workspace_bytes, tt_stream_t stream_,
                             int32_t *blocks_run) {
    const char *fn = "tt_generate_blocks";
    if (blocks_run) *blocks_run = 0;
    if (!desc || !kv || !gp) return fail(TT_ERR_INVALID_ARG, "%s: null desc or params", fn);
    if (block_loop_workspace_bytes(desc) == 0) return TT_ERR_INVALID_ARG;  // message set
    if (gp->max_new_tokens < 1) return fail(TT_ERR_INVALID_ARG, "%s: max_new_tokens < 1", fn);
    if (gp->steps_per_block < 1) return fail(TT_ERR_INVALID_ARG, "%s: steps_per_block < 1", fn);
    if (kv->B != desc->B || kv->S != desc->S)
        return fail(TT_ERR_INVALID_ARG, "%s: K/V desc B/S differ from the unmask desc", fn);
    if (!logits_fn || !kv_fn) return fail(TT_ERR_INVALID_ARG, "%s: null producer", fn);
    if (desc->B == 0) return TT_OK;
    if (!logits_buf || !ctx_lens || !out_tokens || !gen_len || !active)
        return fail(TT_ERR_INVALID_ARG, "%s: null pointer", fn);
    const int64_t out_elems = static_cast<int64_t>(desc->B) * gp->max_new_tokens;
    if (out_elems > (int64_t(1) << 40)) return fail(TT_ERR_UNSUPPORTED, "%s: output too large", fn);
    GenWs w = carve_gen(workspace, desc);
    if (!workspace || workspace_bytes < w.bytes)
        return fail(TT_ERR_WORKSPACE, "%s: workspace of %zu bytes, %zu needed", fn, workspace_bytes,
                    w.bytes);
    if (reinterpret_cast<uintptr_t>(workspace) % 256)
        return fail(TT_ERR_WORKSPACE, "%s: workspace not 256-byte aligned", fn);
    cudaStream_t stream = (cudaStream_t)stream_;
    const int n_blocks = (gp->max_new_tokens + desc->S - 1) / desc->S;
    const int64_t limit_us =
        static_cast<int64_t>(gp->timeout_ms > 0 ? gp->timeout_ms : 60000) * 1000;

    thread_local PinnedInt host;
    tt_status st = TT_OK;
    if (!host.p && (st = cuda_status(cudaMallocHost(&host.p, sizeof(int32_t)), fn)) != TT_OK)
        return st;
    cudaEvent_t ev;
    if ((st = cuda_status(cudaEventCreateWithFlags(&ev, cudaEventDisableTiming), fn)) != TT_OK)
        return st;
    // the number of sequences still generating, read on the host (bounded wait)
    auto read_active = [&](int *n) -> tt_status {
        tt_status s2 = cuda_status(cudaMemcpyAsync(host.p, w.n_active, sizeof(int32_t),
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
            if (us > limit_us) return fail(TT_ERR_TIMEOUT, "%s: device work not finished", fn);
            if (spin > 64) std::this_thread::sleep_for(std::chrono::microseconds(20));
            else std::this_thread::yield();
        }
        *n = *host.p;
        return TT_OK;
    };

    int n_active = 0;
    count_active_kernel<<<1, kFinishThreads, 0, stream>>>(desc->B, active, w.n_active);
    st = cuda_status(cudaGetLastError(), fn);
    if (st == TT_OK) st = read_active(&n_active);
    for (int blk = 0; st == TT_OK && blk < n_blocks && n_active > 0; ++blk) {
        BlockProducer bp{logits_fn, logits_user, blk};
        LoopProducer prod{call_block_producer, &bp};
        int32_t steps = 0;
        st = run_block_loop(desc, gp->steps_per_block, 0, 0, prod, logits_buf, w.tokens,
                            w.is_masked, w.steps_used, nullptr, active, w.loop, w.loop_bytes,
                            stream, gp->timeout_ms, &steps, fn);
        if (st != TT_OK) break;
        FinishArgs fa;
        fa.B = desc->B;
        fa.S = desc->S;
        fa.blk = blk;
        fa.max_new = gp->max_new_tokens;
        fa.eos = gp->eos_token_id;
        fa.Lmax = kv->Lmax;
        fa.more_blocks = blk + 1 < n_blocks ? 1 : 0;
        fa.tokens = w.tokens;
        fa.steps_used = w.steps_used;
        fa.out = out_tokens;
        fa.gen_len = gen_len;
        fa.active = active;
        fa.steps_total = steps_total;
        fa.ctx_lens = ctx_lens;
        fa.overflow = overflow;
        fa.n_active = w.n_active;
        finish_block_kernel<<<1, kFinishThreads, 0, stream>>>(fa);
        if ((st = cuda_status(cudaGetLastError(), fn)) != TT_OK) break;
        if (blocks_run) *blocks_run = blk + 1;
        if ((st = read_active(&n_active)) != TT_OK) break;
        if (n_active > 0 && blk + 1 < n_blocks) {
            tt_status ks = kv_fn(kv_user, blk, w.tokens, active, k_blk, v_blk, stream_);
            if (ks != TT_OK) {
                st = fail(TT_ERR_CALLBACK, "%s: K/V producer returned %s at block %d", fn,
                          tt_status_string(ks), blk);
                break;
            }
            st = tt_kv_append(kv, k_ctx, v_ctx, ctx_lens, k_blk, v_blk, active, nullptr, stream_);
        }
    }
    cudaEventDestroy(ev);
    return st;
}

}  // extern "C"
