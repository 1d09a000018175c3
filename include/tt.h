/*
 * tt.h -- C ABI of libtt: the denoiser-step hot path of the TwoTower block
 * mask-diffusion decoder on one NVIDIA B300 (sm_103a).
 *
 * Two operations, and the in-block loop that iterates the second:
 *
 *  tt_block_attn         block-query attention of one denoiser attention layer.
 *                        The S block queries of layer i attend, through one
 *                        softmax with grouped-query heads, to context-tower
 *                        layer i's K/V for the committed prefix plus the block's
 *                        own K/V, bidirectionally inside the block.
 *                        Pages: dothoosh.com, "فرآیند انتشار در برابر رمزگشایی
 *                        متوالی در مدل جدید انویدیا", section "two-tower mechanism"
 *                        (bidirectional within the block, causal to earlier clean
 *                        blocks, layer i coupled to layer i); aitrends.kr,
 *                        "Nemotron-Labs-TwoTower-30B-A3B-Base-BF16", section
 *                        "technical features" (layer-aligned attention to the
 *                        context tower's KV); tgviewer.app, "NVIDIA, возможно,
 *                        решила главный компромисс современных LLM" (layer-by-layer
 *                        coupling of the towers).
 *
 *  tt_confidence_unmask  one confidence-unmasking step: per still-masked block
 *                        position, the argmax token of the logits and the
 *                        confidence max softmax(logits/T); commit every position
 *                        with confidence >= gamma (at least the single most
 *                        confident one) and re-mask the rest.
 *                        Pages: keyframe.defihacklabs.io, "Diffusion Nemotron",
 *                        key point 3; 889990.xyz, "NVIDIA发布Nemotron两塔模型",
 *                        code example (temperature, confidence_threshold,
 *                        mask_token_id, block_size, steps_per_block).
 *
 *  tt_denoise_block_loop the in-block iteration: a block starts as S mask tokens
 *                        and is refined step by step until every position is
 *                        committed (dothoosh.com article, "two-tower mechanism").
 *
 * Conventions for every entry point:
 *  - All pointers named device are CUDA device pointers (global memory) that
 *    the caller allocates, owns and keeps alive until the stream work ends.
 *    Host pointers are named so.  The library allocates no device memory on any
 *    call; scratch comes from the caller through the *_workspace_size queries.
 *  - Work is enqueued asynchronously on `stream` (NULL = the legacy default
 *    stream).  Only tt_denoise_block_loop waits on the host, once per step,
 *    bounded by its timeout.
 *  - Every call returns a tt_status and never aborts the process.  Arguments
 *    are validated on the host before any launch; on TT_ERR_INVALID_ARG,
 *    TT_ERR_UNSUPPORTED or TT_ERR_WORKSPACE nothing was enqueued.
 *    tt_last_error() gives a message for the calling thread's last failure.
 *  - A workspace starts with an error word that must be zero before the
 *    workspace's first use: zero the workspace once (tt_workspace_zero or any
 *    memset) after allocating it.  The kernels keep no other state in it between
 *    calls.  Calls that share a workspace must be ordered on one stream.
 *  - bf16 is IEEE bfloat16 bit patterns (uint16).  Strides are in elements.
 */
#ifndef TT_H_
#define TT_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (CUstream) handle; NULL selects the legacy default stream. */
typedef struct CUstream_st *tt_stream_t;

typedef enum {
    TT_OK = 0,
    TT_ERR_INVALID_ARG = 1,  /* bad shape, null pointer, negative size, T <= 0 ... */
    TT_ERR_UNSUPPORTED = 2,  /* valid but outside what the kernels implement */
    TT_ERR_WORKSPACE = 3,    /* workspace missing, too small or misaligned */
    TT_ERR_CUDA = 4,         /* a CUDA runtime or launch error (message kept) */
    TT_ERR_TIMEOUT = 5,      /* the loop's bounded wait on the device ran out */
    TT_ERR_CALLBACK = 6,     /* the loop's logits producer returned non-OK */
    TT_ERR_INTERNAL = 7
} tt_status;

typedef enum { TT_F32 = 0, TT_BF16 = 1 } tt_dtype;

/* Static string naming a status. */
const char *tt_status_string(tt_status s);
/* Message of the calling thread's last non-OK status ("" if none).  Valid until
 * the thread's next call into the library. */
const char *tt_last_error(void);
/* ABI version of this header (major*1000 + minor). */
int32_t tt_abi_version(void);

/* Enqueues a zero fill of `bytes` bytes of a device workspace.  Call once after
 * allocating a workspace, before its first use. */
tt_status tt_workspace_zero(void *workspace, size_t bytes, tt_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Block-query attention                                                     */
/* ------------------------------------------------------------------------ */

/*
 * Shape and layout of one attention-layer call.
 *   B     sequences;  S  block size (1..64);  Hq query heads;  Hkv KV heads
 *         (Hq % Hkv == 0; query head h uses KV head h / (Hq/Hkv));
 *   d     head dim, 64 or 128;  Lmax  allocated prefix rows of the context cache.
 *   scale softmax scale; <= 0 selects 1/sqrt(d).
 * Tensors (element strides, innermost dimension contiguous, i.e. stride 1;
 * other strides positive multiples of 8 elements so rows start on 16 bytes):
 *   q      [B, S, Hq, d]      bf16   block queries
 *   k_ctx  [B, Hkv, Lmax, d]  bf16   context-tower layer-i keys (prefix rows
 *   v_ctx  [B, Hkv, Lmax, d]  bf16   0..L_b-1; rows >= L_b never affect the
 *                                    result, whatever they hold: the kernel
 *                                    fetches keys in tiles of 64 rows, so rows
 *                                    of the last partial tile below Lmax may be
 *                                    read, and are masked out of the softmax)
 *   k_blk  [B, S, Hkv, d]     bf16   the block's own keys and values
 *   v_blk  [B, S, Hkv, d]     bf16
 *   out    [B, S, Hq, d]      bf16   written, round-to-nearest-even of fp32
 */
typedef struct {
    int32_t B, S, Hq, Hkv, d, Lmax;
    float scale;
    int64_t q_strides[4];
    int64_t kctx_strides[4];
    int64_t vctx_strides[4];
    int64_t kblk_strides[4];
    int64_t vblk_strides[4];
    int64_t o_strides[4];
} tt_attn_desc;

/* Bytes of device workspace tt_block_attn needs for `desc` on the current
 * device (depends on B, Hkv, S*Hq/Hkv, d and the device's SM count; not on the
 * context lengths).  0 on invalid desc. */
size_t tt_block_attn_workspace_size(const tt_attn_desc *desc);

/*
 * out[b,s,h,:] = sum over keys j of softmax_j(scale * <q[b,s,h,:], key_j>) * value_j,
 * where the keys of sequence b and KV head g = h/(Hq/Hkv) are the prefix rows
 * k_ctx[b,g,0..L_b-1,:] followed by the block rows k_blk[b,0..S-1,g,:] (values
 * alike).  Every block query sees the whole prefix and all S block keys.
 *   ctx_lens  device int32[B], 0 <= L_b <= Lmax.  The lengths live on the
 *             device, so the host cannot check them: a value outside that range
 *             sets the flag 8 in the workspace error word (tt_block_attn_error); the
 *             kernel computes that sequence with the length clamped into range
 *             (no read leaves the cache); the other sequences are unaffected.
 *   lse       device float[B, Hq, S] natural-log log-sum-exp of the scaled
 *             scores, or NULL.
 *   workspace device, >= tt_block_attn_workspace_size(desc) bytes, 256-byte
 *             aligned, zeroed before first use (see conventions).
 * The kernels split long prefixes across SMs and merge the partial softmax
 * states with a log-sum-exp merge; the result does not depend on the split
 * beyond fp32 rounding.  The kernel's internal waits are bounded (2 s each): a
 * wait that runs out -- which a correct build never does -- stops the kernel
 * cleanly, leaves `out` incomplete and records a nonzero flag in the workspace
 * (see tt_block_attn_error).
 */
tt_status tt_block_attn(const tt_attn_desc *desc, const void *q, const void *k_ctx,
                        const void *v_ctx, const int32_t *ctx_lens, const void *k_blk,
                        const void *v_blk, void *out, float *lse, void *workspace,
                        size_t workspace_bytes, tt_stream_t stream);

/*
 * Options of tt_block_attn_ex (a NULL options pointer, or all fields 0, is
 * tt_block_attn):
 *   keys      which keys every block query attends to, through one softmax:
 *             TT_KEYS_ALL the prefix and the block (tt_block_attn); TT_KEYS_PREFIX
 *             the context prefix only; TT_KEYS_BLOCK the block's own keys only.  The
 *             aitrends.kr page ("Nemotron-Labs-TwoTower-30B-A3B-Base-BF16", section
 *             "technical features") names in-block self-attention and layer-aligned
 *             attention to the context separately: the two key sets attended apart,
 *             each with its log-sum-exp, combine into the one softmax over both
 *             (tt_attn_lse_combine).  A row with no key (TT_KEYS_PREFIX and L_b = 0)
 *             gets out = 0 and lse = -inf.
 *   block_table, max_pages, n_pages
 *             a paged context cache: k_ctx and v_ctx are pools of n_pages pages of 64
 *             keys, [n_pages, Hkv, 64, d] with kctx_strides/vctx_strides giving (page,
 *             head, row, 1); block_table is device int32 [B, max_pages], entry j the
 *             page that holds keys 64j .. 64j+63 of sequence b; desc->Lmax must be
 *             max_pages * 64.  Entries past a sequence's length are not read.  A page
 *             id outside [0, n_pages) is recorded (flag 16 of the error word) and read
 *             as zeros.  NULL: the contiguous [B, Hkv, Lmax, d] cache.
 *   q_scale, q_shift, o_gate
 *             adaLN-single modulation (aitrends.kr page, technical features: scale,
 *             shift and gate injected per timestep into each denoiser layer; dothoosh.com
 *             page, architecture bullets), device fp32 [B, Hq, d] each: queries become
 *             q * (1 + q_scale) + q_shift (rounded to bf16) before the scores, and the
 *             output is multiplied by o_gate.  q_scale and q_shift go together; NULL
 *             for none.  16-byte aligned.
 */
typedef enum { TT_KEYS_ALL = 0, TT_KEYS_PREFIX = 1, TT_KEYS_BLOCK = 2 } tt_attn_keys;

typedef struct {
    int32_t keys;
    const int32_t *block_table;
    int32_t max_pages;
    int32_t n_pages;
    const float *q_scale;
    const float *q_shift;
    const float *o_gate;
} tt_attn_opts;

/* tt_block_attn with options (see tt_attn_opts); same workspace. */
tt_status tt_block_attn_ex(const tt_attn_desc *desc, const tt_attn_opts *opts, const void *q,
                           const void *k_ctx, const void *v_ctx, const int32_t *ctx_lens,
                           const void *k_blk, const void *v_blk, void *out, float *lse,
                           void *workspace, size_t workspace_bytes, tt_stream_t stream);

/*
 * Combines two attention results over disjoint key sets (each with its natural-log
 * lse) into the result over their union:
 *   M = max(lse1, lse2), w_i = exp(lse_i - M) (0 where lse_i = -inf),
 *   out = (w1 o1 + w2 o2) / (w1 + w2) (0 when both are -inf),
 *   lse_out = M + log(w1 + w2) (-inf when both are), lse_out nullable.
 * o1, o2, out: device bf16 [B, S, Hq, d] contiguous (16-byte aligned); lse1, lse2,
 * lse_out: device fp32 [B, Hq, S].  out may alias o1 or o2; lse_out must not alias
 * lse1 or lse2.
 */
tt_status tt_attn_lse_combine(int32_t B, int32_t S, int32_t Hq, int32_t d, const void *o1,
                              const float *lse1, const void *o2, const float *lse2, void *out,
                              float *lse_out, tt_stream_t stream);

/*
 * Reads the device error word of an attention workspace into *flag_out (host).
 * It accumulates over every call that used the workspace since it was zeroed:
 * 0 = nothing to report; otherwise an OR of
 *   1  the TMA producer gave up on a wait,   2  an MMA issuer gave up on a wait,
 *   4  the softmax warps gave up on a wait,  8  a ctx_lens value was outside
 *      [0, Lmax] (that sequence was computed with the length clamped),
 *   16 a paged cache's block table named a page outside the pool.
 * A wait that gives up leaves `out` incomplete.  Synchronizes `stream`.
 */
tt_status tt_block_attn_error(const void *workspace, int32_t *flag_out, tt_stream_t stream);

/*
 * tt_block_attn without a caller-provided workspace.  The TwoTower pages have
 * no counterpart to this entry point: it exists for callers that cannot
 * allocate device memory, such as code embedded in a host program whose device
 * memory all belongs to another allocator's pool, or a latency-critical loop
 * that must never call cudaMalloc because it can synchronize the device.
 * Same arguments and result as tt_block_attn, minus the workspace.
 *  - Scratch is a fixed 32 MiB device array inside libtt (file-scope static);
 *    every GPU that loads the library holds it until the process exits.  No
 *    call allocates or frees memory.
 *  - Limit: B*Hkv*ceil(S*(Hq/Hkv)/256) "pairs" must leave room for at least one
 *    partial slot per pair plus one: at d=128 about 250 pairs (e.g. B=125 with
 *    Hkv=2), at d=64 about 500.  Larger shapes return TT_ERR_UNSUPPORTED with a
 *    message; when the scratch holds fewer partial slots than the device has
 *    SMs the prefix is split across fewer SMs (same result up to fp32 rounding).
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress); make that first call before any stream capture.
 *  - Every call shares the one array and clears its error word and per-pair
 *    split table on `stream` before the kernel: calls that overlap on the GPU
 *    (other streams, other host threads without ordering) race and corrupt each
 *    other's results.  Order them on one stream.
 *  - The error word lives in the shared array and is cleared by the next call,
 *    and no entry point reads it: a kernel wait that gives up or a ctx_lens value
 *    out of range (see tt_block_attn_error) is NOT reported by this variant.
 *    Callers that need those reports use tt_block_attn with a workspace.
 */
tt_status tt_block_attn_noalloc(const tt_attn_desc *desc, const void *q, const void *k_ctx,
                                const void *v_ctx, const int32_t *ctx_lens, const void *k_blk,
                                const void *v_blk, void *out, float *lse, tt_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Confidence unmasking                                                      */
/* ------------------------------------------------------------------------ */

/*
 *   B, S, V          sequences, block size (1..64), vocabulary size (>= 1)
 *   logits_dtype     TT_F32 or TT_BF16
 *   logits_row_stride elements between consecutive (b,s) rows; 0 means V
 *   temperature      T > 0; confidence = max_v softmax(logits/T)_v
 *   threshold        gamma: commit every masked position whose fp32
 *                    confidence is >= gamma.  gamma = 0 commits all; gamma > 1
 *                    commits exactly the single most confident one per step.
 *   mask_token_id    token written into positions that stay masked
 */
typedef struct {
    int32_t B, S, V;
    tt_dtype logits_dtype;
    int64_t logits_row_stride;
    float temperature;
    float threshold;
    int32_t mask_token_id;
} tt_unmask_desc;

/* Bytes of device workspace tt_confidence_unmask needs (0 on invalid desc). */
size_t tt_confidence_unmask_workspace_size(const tt_unmask_desc *desc);

/*
 * One unmasking step over device logits [B, S, V] (row stride as in desc; the
 * base and each row must start on a 4-byte boundary).  For each sequence b:
 *   for masked s: token = lowest index of the maximum raw logit;
 *                 conf  = 1 / sum_v exp((l_v - max)/T)   (fp32);
 *   commit C = { masked s : conf >= gamma }; if C is empty and a position is
 *   masked, C = { the masked s of highest conf, lowest s on ties };
 *   force_commit_all != 0 commits every masked position.
 *   s in C:        tokens[b,s] = token, is_masked[b,s] = 0, committed_now = 1
 *   masked, not C: tokens[b,s] = mask_token_id, committed_now = 0
 *   not masked:    tokens unchanged, committed_now = 0, conf = NaN
 * Device arrays:  tokens int32[B,S] and is_masked uint8[B,S] (in/out);
 * conf float[B,S], committed_now uint8[B,S], remaining int32[B] (masked
 * positions left) are written.  Only masked rows of logits are read.
 * Rows must hold finite values or -inf with at least one finite value.
 */
tt_status tt_confidence_unmask(const tt_unmask_desc *desc, const void *logits, int32_t *tokens,
                               uint8_t *is_masked, float *conf, uint8_t *committed_now,
                               int32_t *remaining, int32_t force_commit_all, void *workspace,
                               size_t workspace_bytes, tt_stream_t stream);

/*
 * Reads the error word of an unmask (or block-loop) workspace into *flag_out
 * (host): 0 = nothing to report since the workspace was zeroed; otherwise an OR
 * of 1 (the kernel's copy-issuing thread gave up on a wait) and 2 (its reducing
 * warps gave up on a wait).  A wait that gives up leaves that step's outputs
 * incomplete; tt_denoise_block_loop checks the word after every step and returns
 * TT_ERR_INTERNAL when it is set.  Synchronizes `stream`.
 */
tt_status tt_confidence_unmask_error(const void *workspace, int32_t *flag_out,
                                     tt_stream_t stream);

/* ------------------------------------------------------------------------ */
/* In-block loop                                                             */
/* ------------------------------------------------------------------------ */

/*
 * Producer of one step's logits (the denoiser forward, or a stand-in).  It
 * must enqueue on `stream` work that writes logits [B,S,V] (layout of the
 * loop's desc) into logits_out, and may read tokens / is_masked (device).  A
 * non-OK return stops the loop with TT_ERR_CALLBACK.
 */
typedef tt_status (*tt_logits_fn)(void *user, int32_t step, const int32_t *tokens,
                                  const uint8_t *is_masked, void *logits_out,
                                  tt_stream_t stream);

/*
 * Starts a block: tokens[b,s] = mask_token_id and is_masked[b,s] = 1 for every
 * position; steps_used[b] = 0 and committed_step[b,s] = -1 when those (device,
 * nullable) are given.  Uses desc's B, S and mask_token_id only.
 */
tt_status tt_block_init(const tt_unmask_desc *desc, int32_t *tokens, uint8_t *is_masked,
                        int32_t *steps_used, int32_t *committed_step, tt_stream_t stream);

/* Bytes of device workspace tt_denoise_block_loop needs (0 on invalid desc). */
size_t tt_denoise_block_loop_workspace_size(const tt_unmask_desc *desc);

/*
 * Runs steps k = start_step .. min(stop_step, steps_per_block)-1 of the
 * in-block iteration (stop_step <= 0 means steps_per_block):
 *   if start_step == 0 the block is initialised first: tokens = mask_token_id,
 *   is_masked = 1, steps_used = 0, committed_step = -1;
 *   each step: if no position of any sequence is masked, stop; else
 *   producer(user, k, ...) writes logits_buf, then one tt_confidence_unmask
 *   step runs with force_commit_all at k == steps_per_block-1, steps_used[b]
 *   grows by one for each b that had a masked position, and committed_step[b,s]
 *   = k for positions committed at step k.
 * A resumed call (start_step > 0) continues from the device state it is given,
 * so running steps [0,a) then [a,n) equals running [0,n) bit for bit.
 * Device arrays: tokens int32[B,S], is_masked uint8[B,S], steps_used int32[B],
 * committed_step int32[B,S] (nullable) -- all in/out.  logits_buf is device
 * memory for [B,S,V] logits.  After each step the host waits (polling, at most
 * timeout_ms milliseconds, <= 0 = 60000) for the step's remaining counts;
 * running out returns TT_ERR_TIMEOUT with the state of the last finished step.
 * steps_run (host, nullable) receives the number of steps executed.
 */
tt_status tt_denoise_block_loop(const tt_unmask_desc *desc, int32_t steps_per_block,
                                int32_t start_step, int32_t stop_step, tt_logits_fn producer,
                                void *user, void *logits_buf, int32_t *tokens,
                                uint8_t *is_masked, int32_t *steps_used, int32_t *committed_step,
                                void *workspace, size_t workspace_bytes, tt_stream_t stream,
                                int32_t timeout_ms, int32_t *steps_run);

/* ------------------------------------------------------------------------ */
/* Synthetic logits (a stand-in producer for benches and tests)              */
/* ------------------------------------------------------------------------ */

/*
 * Counter-based synthetic logits, the same definition as the Python input
 * generator: with SplitMix64's output function mix64 (Steele, Lea & Flood,
 * OOPSLA 2014) and GAMMA = 0x9E3779B97F4A7C15,
 *   key   = mix64(mix64(seed ^ 0x6C6F67697473) + (step+1)*GAMMA)
 *   word  = mix64(key + (n+1)*GAMMA),  n = ((b*S+s)*V + v)*3 + j,  j = 0,1,2
 *   z     = (sum of the twelve 16-bit fields of the three words - 393216)
 *           * (sigma / 65536)     (fp32, exact)
 *   spike: w = mix64(mix64(key ^ 0x7370696B65) + (b*S+s+1)*GAMMA); if
 *          (w >> 32) < spike_threshold the row gets +8 at token (w & 0xFFFFFFFF) % V
 *   bf16 output rounds the fp32 value to nearest-even.
 * sigma/65536 must be exact in fp32.  out: device [B,S,V], row stride V.
 */
tt_status tt_synth_logits(uint64_t seed, int32_t step, int32_t B, int32_t S, int32_t V,
                          tt_dtype dtype, float sigma, uint64_t spike_threshold, void *out,
                          tt_stream_t stream);

/* Parameters of tt_synth_logits_producer: the per-step spike threshold is
 * spike_threshold[min(step, TT_SYNTH_MAX_STEPS-1)]. */
#define TT_SYNTH_MAX_STEPS 256
typedef struct {
    uint64_t seed;
    int32_t B, S, V;
    tt_dtype dtype;
    float sigma;
    uint64_t spike_threshold[TT_SYNTH_MAX_STEPS];
} tt_synth_params;

/* A tt_logits_fn that calls tt_synth_logits with (tt_synth_params*)user. */
tt_status tt_synth_logits_producer(void *user, int32_t step, const int32_t *tokens,
                                   const uint8_t *is_masked, void *logits_out,
                                   tt_stream_t stream);

/* ---------------------------------------------------------------- block append
 *
 * Once every position of a block is committed, the block becomes clean context:
 * the context tower takes it in and the next block attends to a prefix S tokens
 * longer (dothoosh.com, "فرآیند انتشار در برابر رمزگشایی متوالی در مدل جدید
 * انویدیا", section "two-tower mechanism": blocks are generated one after another,
 * each attending causally to the earlier clean blocks).  tt_kv_append writes the
 * block's K/V, per layer, into that layer's context cache after the prefix and
 * advances the prefix length; the K/V values themselves come from the caller
 * (the context tower's forward on the committed tokens, outside this library).
 */
#define TT_KV_MAX_LAYERS 16

typedef struct {
    int32_t B, S, Hkv, d, Lmax;
    int32_t n_layers;        /* 1..TT_KV_MAX_LAYERS */
    int64_t ctx_strides[4];  /* every layer's k_ctx / v_ctx [B, Hkv, Lmax, d] */
    int64_t blk_strides[4];  /* every layer's k_blk / v_blk [B, S, Hkv, d] */
} tt_kv_desc;

/*
 * For every layer l < n_layers and sequence b taking part (active == NULL, or
 * active[b] != 0), with L_b = ctx_lens[b] on entry and L_b + S <= Lmax:
 *   k_ctx[l][b, g, L_b + s, :] = k_blk[l][b, s, g, :]   for s < S, g < Hkv,
 * the same for V, then ctx_lens[b] = L_b + S.  Bytes are copied unchanged.
 *   k_ctx, v_ctx  host arrays of n_layers device pointers, bf16; rows of the
 *                 cache other than [L_b, L_b + S) are not touched.
 *   ctx_lens      device int32[B], updated in place.
 *   k_blk, v_blk  host arrays of n_layers device pointers, bf16.
 *   active        device uint8[B] or NULL (every sequence).
 *   overflow      device int32 or NULL: incremented once for every sequence that
 *                 takes part but has L_b < 0 or L_b + S > Lmax; such a sequence's
 *                 cache and length are left unchanged.
 * Strides are in elements, positive multiples of 8 with the innermost one 1, and
 * every pointer 16-byte aligned; d is a multiple of 8 up to 512; B <= 65535.  Two
 * launches on `stream` (the copies, then the length update); the call returns once
 * they are enqueued.
 */
tt_status tt_kv_append(const tt_kv_desc *desc, void *const *k_ctx, void *const *v_ctx,
                       int32_t *ctx_lens, const void *const *k_blk, const void *const *v_blk,
                       const uint8_t *active, int32_t *overflow, tt_stream_t stream);

/* ------------------------------------------------------------- adaLN-single
 *
 * Time conditioning of the denoiser: every denoiser layer gets a scale, shift and
 * gate per diffusion timestep from an adaLN-single module (aitrends.kr,
 * "Nemotron-Labs-TwoTower-30B-A3B-Base-BF16", section "technical features": about
 * 1.5 M added parameters; dothoosh.com, architecture bullets).  tt_adaln_single
 * computes them; tt_block_attn_ex applies them to the attention (tt_attn_opts).
 */
typedef struct {
    int32_t B;        /* sequences */
    int32_t F;        /* timestep embedding size, even, <= 1024 */
    int32_t Dh;       /* hidden size of the shared network, <= 512 */
    int32_t N;        /* size of each modulation vector (Hq*d for the attention) */
    int32_t layer;    /* which row of `embed` */
    int32_t n_layers; /* rows of `embed` */
} tt_adaln_desc;

/*
 * For every sequence b with timestep t[b] (device fp32 [B]):
 *   e = [cos(t w_i)]_{i<F/2} ++ [sin(t w_i)]_{i<F/2},  w_i = 10000^(-i/(F/2));
 *   h = SiLU(W1 e + b1);  m = W2 h + b2 + embed[layer];
 *   shift[b] = m[0:N], scale[b] = m[N:2N], gate[b] = m[2N:3N].
 * Device fp32 arrays: w1 [Dh, F], b1 [Dh], w2 [3N, Dh], b2 [3N], embed [n_layers, 3N],
 * outputs shift, scale, gate [B, N].  One launch.
 */
tt_status tt_adaln_single(const tt_adaln_desc *desc, const float *t, const float *w1,
                          const float *b1, const float *w2, const float *b2, const float *embed,
                          float *shift, float *scale, float *gate, tt_stream_t stream);

/* ---------------------------------------------------------- Mamba-2 state seeding
 *
 * The denoiser's Mamba-2 layers start from the context tower's states: each
 * denoiser Mamba layer takes as its initial state the conv/SSM boundary state the
 * corresponding context-tower layer ends on (dothoosh.com, "فرآیند انتشار در برابر
 * رمزگشایی متوالی در مدل جدید انویدیا", architecture bullets; aitrends.kr,
 * "Nemotron-Labs-TwoTower-30B-A3B-Base-BF16", section "technical features").  The
 * pages give no recurrence; this is the seeding copy, for all layers in one launch.
 */
#define TT_STATE_MAX_LAYERS 64
#define TT_STATE_MAX_PARTS 4

typedef struct {
    int32_t B;
    int32_t n_layers;                       /* 1..TT_STATE_MAX_LAYERS */
    int32_t n_parts;                        /* state tensors per layer (e.g. conv, SSM), 1..4 */
    int64_t bytes[TT_STATE_MAX_PARTS];      /* bytes of one sequence's state of each part */
    int64_t src_stride[TT_STATE_MAX_PARTS]; /* bytes between sequences in the source */
    int64_t dst_stride[TT_STATE_MAX_PARTS]; /* bytes between sequences in the destination */
} tt_state_desc;

/*
 * For every layer l, part p and sequence b taking part (active == NULL, or
 * active[b] != 0): the bytes [0, bytes[p]) of src[l*n_parts + p] + b*src_stride[p]
 * are copied to dst[l*n_parts + p] + b*dst_stride[p].  Sequences not taking part
 * keep their destination state.
 *   src, dst  host arrays of n_layers*n_parts device pointers (16-byte aligned);
 *   bytes and strides positive multiples of 16, strides at least the size;
 *   n_layers*n_parts*B at most 65535.  One launch; sources and destinations must
 *   not overlap.
 */
tt_status tt_mamba_state_seed(const tt_state_desc *desc, const void *const *src,
                              void *const *dst, const uint8_t *active, tt_stream_t stream);

/* ------------------------------------------------------- block-by-block generation
 *
 * Blocks of S positions are generated one after another: each block is denoised by
 * the in-block loop, its tokens are kept, and -- unless generation ends -- the
 * committed block's K/V (from the caller's context-tower stand-in) joins every
 * layer's context cache, so the next block attends to a prefix S tokens longer
 * (dothoosh.com, "فرآیند انتشار در برابر رمزگشایی متوالی در مدل جدید انویدیا",
 * section "two-tower mechanism"; 889990.xyz, "NVIDIA发布Nemotron两塔模型",
 * section 训练与推理, code example: max_new_tokens, block_size, steps_per_block,
 * eos_token_id).
 */

/* Producer of one step's logits for block `block` (the denoiser forward, or a
 * stand-in): as tt_logits_fn, with the block index. */
typedef tt_status (*tt_block_logits_fn)(void *user, int32_t block, int32_t step,
                                        const int32_t *tokens, const uint8_t *is_masked,
                                        void *logits_out, tt_stream_t stream);

/* Producer of a committed block's K/V (the context tower's forward over the
 * block's tokens, or a stand-in): must enqueue on `stream` work that writes, for
 * every layer l of the K/V desc, k_blk[l] and v_blk[l] ([B, S, Hkv, d] bf16, the
 * desc's block strides) from tokens [B, S] (device).  Only sequences with
 * active[b] != 0 (device) are appended; the others' rows may hold anything.  A
 * non-OK return stops generation with TT_ERR_CALLBACK. */
typedef tt_status (*tt_block_kv_fn)(void *user, int32_t block, const int32_t *tokens,
                                    const uint8_t *active, void *const *k_blk,
                                    void *const *v_blk, tt_stream_t stream);

typedef struct {
    int32_t max_new_tokens;  /* >= 1; blocks = ceil(max_new_tokens / S) */
    int32_t eos_token_id;    /* < 0: no end-of-sequence token */
    int32_t steps_per_block; /* >= 1 */
    int32_t timeout_ms;      /* bound of each host wait; <= 0 means 60000 */
} tt_generate_params;

/* Bytes of device workspace tt_generate_blocks needs (0 on invalid desc). */
size_t tt_generate_blocks_workspace_size(const tt_unmask_desc *desc);

/*
 * Runs blocks k = 0, 1, ... while some sequence is generating (active[b] != 0),
 * at most ceil(max_new_tokens / S) of them.  For block k:
 *   1. the in-block loop (tt_denoise_block_loop's steps, logits from
 *      logits_fn(user, k, step, ...) into logits_buf) over a block that starts
 *      masked for the generating sequences only;
 *   2. for every sequence generating at the start of block k, with
 *      keep = min(S, max_new_tokens - k*S): out_tokens[b, k*S + s] = token s for
 *      s < keep; if one of those is eos_token_id, gen_len[b] = k*S + (first EOS
 *      position) + 1 and the sequence stops; otherwise gen_len[b] = k*S + keep,
 *      and the sequence stops at max_new_tokens, or when another block follows and
 *      its cache cannot take this one (ctx_lens[b] + S > Lmax; counted in
 *      *overflow); steps_total[b] grows by the steps the block took;
 *   3. if another block follows and some sequence still generates:
 *      kv_fn(kv_user, k, tokens, active, k_blk, v_blk) and tt_kv_append of this
 *      block for the sequences still generating (ctx_lens grows by S).
 * Arrays: out_tokens int32[B, max_new_tokens] (positions not generated are not
 * written), gen_len int32[B] (written for generating sequences), active uint8[B]
 * in/out, steps_total int32[B] (nullable, accumulated), overflow int32 (nullable,
 * accumulated) -- all device.  k_ctx, v_ctx, ctx_lens, k_blk, v_blk and `kv` as
 * for tt_kv_append (kv->B, kv->S equal desc->B, desc->S).  The host waits once per
 * step (the loop) and once per block, each bounded by timeout_ms.  blocks_run
 * (host, nullable) receives the number of blocks run.  A producer error returns
 * TT_ERR_CALLBACK with the blocks before it complete.
 */
tt_status tt_generate_blocks(const tt_unmask_desc *desc, const tt_kv_desc *kv,
                             const tt_generate_params *params, tt_block_logits_fn logits_fn,
                             void *logits_user, tt_block_kv_fn kv_fn, void *kv_user,
                             void *logits_buf, void *const *k_ctx, void *const *v_ctx,
                             int32_t *ctx_lens, void *const *k_blk, void *const *v_blk,
                             int32_t *out_tokens, int32_t *gen_len, uint8_t *active,
                             int32_t *steps_total, int32_t *overflow, void *workspace,
                             size_t workspace_bytes, tt_stream_t stream, int32_t *blocks_run);

#ifdef __cplusplus
}
#endif
#endif /* TT_H_ */
