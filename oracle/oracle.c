/*
 * oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct CPU reference for the denoiser-step hot path
 * of the TwoTower block mask-diffusion decoder, in fp64.  Only the tests, the
 * smoke check and the bench's CPU-baseline leg may load it.  It shares no code,
 * header, table or helper with the CUDA library; the two meet only through the
 * seeded input generators (block_mask_diffusion_tt_b300/synth.py), which hold no
 * arithmetic of the method.
 *
 * Sources (web pages on the TwoTower model; no code is printed on them):
 *  - Block-query attention: dothoosh.com, "فرآیند انتشار در برابر رمزگشایی متوالی در
 *    مدل جدید انویدیا", section "two-tower mechanism": inside a block the
 *    denoiser attends bidirectionally, and causally to the clean blocks before it;
 *    denoiser layer i is coupled to context-tower layer i.  aitrends.kr,
 *    "Nemotron-Labs-TwoTower-30B-A3B-Base-BF16", section "technical features":
 *    in-block bidirectional self-attention plus layer-aligned attention to the
 *    context tower's layer-i KV.  Read here as ONE softmax over the committed
 *    prefix's keys followed by the block's own keys, with grouped-query heads
 *    (head h uses KV head floor(h / (Hq/Hkv))), scale 1/sqrt(d) unless given.
 *  - Confidence unmasking: keyframe.defihacklabs.io, "Diffusion Nemotron", key
 *    point 3 (fill a block of 16 masked positions, commit confident tokens,
 *    re-mask the rest, iterate); 889990.xyz, "NVIDIA发布Nemotron两塔模型", the code
 *    example (temperature=0.1, confidence_threshold=0.8, mask_token_id=3,
 *    block_size=16, steps_per_block=16).  Read here as: token = argmax of the
 *    raw logits (ties to the lowest index); confidence = max softmax(l/T);
 *    commit every masked position with confidence >= gamma, and the single most
 *    confident one when none passes.
 *
 * Build: gcc -O2 -shared -fPIC -pthread oracle.c -o liboracle.so -lm
 * (no -ffast-math: the arithmetic below is evaluated as written).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ------------------------------------------------------------------ helpers */

/* bf16 bit pattern -> double, exactly (bf16 is the top half of an fp32). */
static double bf16_to_double(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int oracle_hw_threads(void)
{
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

static int resolve_threads(int requested, long work_items)
{
    int n = requested > 0 ? requested : oracle_hw_threads();
    if (work_items < n) n = (int)(work_items > 0 ? work_items : 1);
    return n;
}

/* Runs fn(ctx, i) for i in [0, n) on `threads` threads (static interleaved split). */
typedef void (*item_fn)(void *ctx, long i);
struct pool_arg { item_fn fn; void *ctx; long n; int t, nt; };

static void *pool_worker(void *p)
{
    struct pool_arg *a = (struct pool_arg *)p;
    for (long i = a->t; i < a->n; i += a->nt) a->fn(a->ctx, i);
    return NULL;
}

static int run_parallel(item_fn fn, void *ctx, long n, int threads)
{
    if (threads <= 1) {
        for (long i = 0; i < n; ++i) fn(ctx, i);
        return 1;
    }
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)threads);
    struct pool_arg *args = (struct pool_arg *)malloc(sizeof(struct pool_arg) * (size_t)threads);
    int started = 0;
    for (int t = 0; t < threads; ++t) {
        args[t] = (struct pool_arg){fn, ctx, n, t, threads};
        if (pthread_create(&tid[t], NULL, pool_worker, &args[t]) == 0) {
            ++started;
        } else { /* fall back to running this share inline */
            pool_worker(&args[t]);
            tid[t] = 0;
        }
    }
    for (int t = 0; t < threads; ++t)
        if (tid[t]) pthread_join(tid[t], NULL);
    free(tid);
    free(args);
    return started > 0 ? started : 1;
}

/* ------------------------------------------------------------ attention */

/* Which keys a block query sees: the prefix then the block (the one softmax of the
 * two-tower mechanism), the context prefix alone, or the block alone (the aitrends.kr
 * page names in-block self-attention and attention to the context separately). */
enum { KEYS_ALL = 0, KEYS_PREFIX = 1, KEYS_BLOCK = 2 };

struct attn_ctx {
    int B, S, Hq, Hkv, d, Lmax;
    double scale;
    const uint16_t *q, *k_ctx, *v_ctx, *k_blk, *v_blk;
    const double *q64;  /* queries in fp64 (modulated), overrides q when given */
    const double *gate; /* [B, Hq, d] output gate, or NULL */
    const int32_t *lens;
    int keys;
    double *out, *lse;
};

/* Number of keys a query of sequence b sees. */
static int visible(const struct attn_ctx *c, int b)
{
    int L = c->lens[b];
    return c->keys == KEYS_PREFIX ? L : (c->keys == KEYS_BLOCK ? c->S : L + c->S);
}

/* Key j of the visible sequence for (b, kv head g): the prefix rows first (context
 * tower cache row j), then the block rows (block row j - L_b); with only one of the
 * two sets visible, its rows alone. */
static const uint16_t *key_row(const struct attn_ctx *c, const uint16_t *ctx,
                               const uint16_t *blk, int b, int g, int j)
{
    int L = c->keys == KEYS_BLOCK ? 0 : c->lens[b];
    if (j < L)
        return ctx + (((size_t)b * c->Hkv + g) * c->Lmax + j) * c->d;
    return blk + (((size_t)b * c->S + (j - L)) * c->Hkv + g) * c->d;
}

/* One work item = (b, query head h): every block row s of that head. */
static void attn_item(void *p, long item)
{
    const struct attn_ctx *c = (const struct attn_ctx *)p;
    int b = (int)(item / c->Hq), h = (int)(item % c->Hq);
    int G = c->Hq / c->Hkv, g = h / G;          /* grouped-query head map */
    int n = visible(c, b);
    int d = c->d;
    double *x = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    double *acc = (double *)malloc(sizeof(double) * (size_t)d);
    double *qd = (double *)malloc(sizeof(double) * (size_t)d);

    for (int s = 0; s < c->S; ++s) {
        size_t qi = (((size_t)b * c->S + s) * c->Hq + h) * d;
        for (int e = 0; e < d; ++e) qd[e] = c->q64 ? c->q64[qi + e] : bf16_to_double(c->q[qi + e]);
        double *o = c->out + qi;
        if (n == 0) { /* no key: an empty sum */
            for (int e = 0; e < d; ++e) o[e] = 0.0;
            if (c->lse) c->lse[((size_t)b * c->Hq + h) * c->S + s] = -INFINITY;
            continue;
        }
        /* scores x_j = scale * <q, k_j> */
        double m = -INFINITY;
        for (int j = 0; j < n; ++j) {
            const uint16_t *kr = key_row(c, c->k_ctx, c->k_blk, b, g, j);
            double dot = 0.0;
            for (int e = 0; e < d; ++e) dot += qd[e] * bf16_to_double(kr[e]);
            x[j] = c->scale * dot;
            if (x[j] > m) m = x[j];
        }
        /* softmax weights and the weighted sum of values */
        double den = 0.0;
        for (int e = 0; e < d; ++e) acc[e] = 0.0;
        for (int j = 0; j < n; ++j) {
            double w = exp(x[j] - m);
            den += w;
            const uint16_t *vr = key_row(c, c->v_ctx, c->v_blk, b, g, j);
            for (int e = 0; e < d; ++e) acc[e] += w * bf16_to_double(vr[e]);
        }
        const double *gt = c->gate ? c->gate + ((size_t)b * c->Hq + h) * d : NULL;
        for (int e = 0; e < d; ++e) o[e] = (gt ? gt[e] : 1.0) * (acc[e] / den);
        if (c->lse) c->lse[((size_t)b * c->Hq + h) * c->S + s] = m + log(den);
    }
    free(x);
    free(acc);
    free(qd);
}

/*
 * out[b,s,h,:] = sum_j softmax_j(scale * <q[b,s,h], key_j>) * value_j over the
 * keys of sequence b, KV head floor(h/(Hq/Hkv)): prefix rows 0..L_b-1 of
 * k_ctx/v_ctx [B,Hkv,Lmax,d], then block rows 0..S-1 of k_blk/v_blk [B,S,Hkv,d].
 * q is [B,S,Hq,d]; all bf16 bit patterns, contiguous.  lse (nullable) is
 * [B,Hq,S], natural log.  Returns the number of threads used, or -1 on bad
 * arguments.  Context rows at or beyond L_b are never read.
 */
int oracle_block_attn2(int B, int S, int Hq, int Hkv, int d, int Lmax, double scale,
                       const uint16_t *q, const double *q64, const uint16_t *k_ctx,
                       const uint16_t *v_ctx, const int32_t *ctx_lens, const uint16_t *k_blk,
                       const uint16_t *v_blk, int keys, const double *gate, double *out,
                       double *lse, int nthreads);

int oracle_block_attn(int B, int S, int Hq, int Hkv, int d, int Lmax, double scale,
                      const uint16_t *q, const uint16_t *k_ctx, const uint16_t *v_ctx,
                      const int32_t *ctx_lens, const uint16_t *k_blk, const uint16_t *v_blk,
                      double *out, double *lse, int nthreads)
{
    return oracle_block_attn2(B, S, Hq, Hkv, d, Lmax, scale, q, NULL, k_ctx, v_ctx, ctx_lens,
                              k_blk, v_blk, KEYS_ALL, NULL, out, lse, nthreads);
}

/*
 * oracle_block_attn with the key set chosen (keys: 0 prefix then block, 1 prefix
 * only, 2 block only; a row that sees no key gets out = 0 and lse = -inf), the
 * queries optionally given in fp64 (q64 [B,S,Hq,d], e.g. modulated; then q is not
 * read) and an optional output gate (gate [B,Hq,d] multiplies the result).
 */
int oracle_block_attn2(int B, int S, int Hq, int Hkv, int d, int Lmax, double scale,
                       const uint16_t *q, const double *q64, const uint16_t *k_ctx,
                       const uint16_t *v_ctx, const int32_t *ctx_lens, const uint16_t *k_blk,
                       const uint16_t *v_blk, int keys, const double *gate, double *out,
                       double *lse, int nthreads)
{
    if (keys < KEYS_ALL || keys > KEYS_BLOCK) return -1;
    if (!q && !q64) return -1;
    if (B < 0 || S < 1 || Hq < 1 || Hkv < 1 || d < 1 || Lmax < 0 || Hq % Hkv != 0) return -1;
    if (!k_blk || !v_blk || !out || !ctx_lens || (Lmax > 0 && (!k_ctx || !v_ctx))) return -1;
    for (int b = 0; b < B; ++b)
        if (ctx_lens[b] < 0 || ctx_lens[b] > Lmax) return -1;
    struct attn_ctx c = {B, S, Hq, Hkv, d, Lmax, scale > 0.0 ? scale : 1.0 / sqrt((double)d),
                         q, k_ctx, v_ctx, k_blk, v_blk, q64, gate, ctx_lens, keys, out, lse};
    long items = (long)B * Hq;
    return run_parallel(attn_item, &c, items, resolve_threads(nthreads, items));
}

/* ------------------------------------------------------------ unmasking */

#define ORACLE_AMBIG_REL 1e-5

/* A confidence within 2^-26 of 1 is exactly 1.0f in any fp32 evaluation whose
 * relative error stays below 2^-25: the probability mass outside the top token
 * is then under half an fp32 unit of the sum's leading 1.  Decisions between
 * such confidences (exact fp32 ties, or a threshold of 1) are not ambiguous. */
static int conf_is_one_in_f32(double c) { return c >= 1.0 - ldexp(1.0, -26); }

struct unmask_ctx {
    int S, V, dtype;
    const void *logits;
    double temperature;
    const uint8_t *is_masked;
    int32_t *tok;
    double *conf;
};

static double logit_at(const struct unmask_ctx *c, size_t row, int v)
{
    if (c->dtype == 0) return (double)((const float *)c->logits)[row * (size_t)c->V + v];
    return bf16_to_double(((const uint16_t *)c->logits)[row * (size_t)c->V + v]);
}

/* Row reduction for one masked position: token = lowest index of the raw-logit
 * maximum; confidence = max_v softmax(l/T)_v = 1 / sum_v exp((l_v - max)/T). */
static void unmask_row(void *p, long row)
{
    const struct unmask_ctx *c = (const struct unmask_ctx *)p;
    if (!c->is_masked[row]) {
        c->conf[row] = NAN;
        c->tok[row] = -1;
        return;
    }
    double best = -INFINITY;
    int arg = 0;
    for (int v = 0; v < c->V; ++v) {
        double l = logit_at(c, (size_t)row, v);
        if (l > best) { best = l; arg = v; }  /* strict: first occurrence wins */
    }
    double sum = 0.0;
    for (int v = 0; v < c->V; ++v) sum += exp((logit_at(c, (size_t)row, v) - best) / c->temperature);
    c->tok[row] = arg;
    c->conf[row] = 1.0 / sum;
}

/*
 * One confidence-unmasking step over logits [B,S,V] (dtype 0 = fp32, 1 = bf16
 * bits).  For every sequence b independently:
 *   masked positions s get (token, confidence) from unmask_row;
 *   C = { masked s : (float)conf >= threshold }     (decision taken in fp32);
 *   if C is empty and some s is masked: C = { the masked s of highest (float)
 *   confidence, lowest s on ties };  if force_commit_all: C = all masked s;
 *   s in C: tokens = token, is_masked = 0, committed_now = 1;
 *   other masked s: tokens = mask_token_id (re-masked), committed_now = 0;
 *   already-committed s: unchanged, committed_now = 0, conf = NaN.
 * remaining[b] = masked positions left.  ambiguous[b,s] (nullable) flags a
 * decision that a relative perturbation of 1e-5 in a confidence could flip:
 * |conf - threshold| <= 1e-5*threshold, or a fallback choice whose two best
 * confidences are within 1e-5 relative -- except between confidences that are
 * 1.0f in any fp32 evaluation (conf_is_one_in_f32).  Returns threads used, -1
 * on bad args.
 */
int oracle_confidence_unmask(int B, int S, int V, int dtype, const void *logits,
                             double temperature, float threshold, int32_t mask_token_id,
                             int force_commit_all, int32_t *tokens, uint8_t *is_masked,
                             double *conf, uint8_t *committed_now, int32_t *remaining,
                             uint8_t *ambiguous, int nthreads)
{
    if (B < 0 || S < 1 || V < 1 || (dtype != 0 && dtype != 1) || !(temperature > 0.0)) return -1;
    if (!logits || !tokens || !is_masked || !conf || !committed_now || !remaining) return -1;
    int32_t *tok = (int32_t *)malloc(sizeof(int32_t) * (size_t)B * S + 1);
    struct unmask_ctx c = {S, V, dtype, logits, temperature, is_masked, tok, conf};
    long rows = (long)B * S;
    int used = run_parallel(unmask_row, &c, rows, resolve_threads(nthreads, rows));

    for (int b = 0; b < B; ++b) {
        size_t base = (size_t)b * S;
        int n_masked = 0, n_pass = 0;
        for (int s = 0; s < S; ++s) {
            committed_now[base + s] = 0;
            if (ambiguous) ambiguous[base + s] = 0;
            if (!is_masked[base + s]) continue;
            ++n_masked;
            float cf = (float)conf[base + s];
            if (force_commit_all || cf >= threshold) {
                committed_now[base + s] = 1;
                ++n_pass;
            }
            if (ambiguous && !force_commit_all && !conf_is_one_in_f32(conf[base + s]) &&
                fabs(conf[base + s] - (double)threshold) <= ORACLE_AMBIG_REL * fabs((double)threshold))
                ambiguous[base + s] = 1;
        }
        if (n_masked > 0 && n_pass == 0) {  /* at least the single most confident one */
            int best = -1, second = -1;
            for (int s = 0; s < S; ++s) {
                if (!is_masked[base + s]) continue;
                float cf = (float)conf[base + s];
                if (best < 0 || cf > (float)conf[base + best]) { second = best; best = s; }
                else if (second < 0 || cf > (float)conf[base + second]) second = s;
            }
            committed_now[base + best] = 1;
            if (ambiguous && second >= 0 &&
                !(conf_is_one_in_f32(conf[base + best]) && conf_is_one_in_f32(conf[base + second])) &&
                fabs(conf[base + best] - conf[base + second]) <= ORACLE_AMBIG_REL * conf[base + best]) {
                ambiguous[base + best] = 1;
                ambiguous[base + second] = 1;
            }
        }
        int left = 0;
        for (int s = 0; s < S; ++s) {
            if (!is_masked[base + s]) continue;
            if (committed_now[base + s]) {
                tokens[base + s] = tok[base + s];
                is_masked[base + s] = 0;
            } else {
                tokens[base + s] = mask_token_id;
                ++left;
            }
        }
        remaining[b] = left;
    }
    free(tok);
    return used;
}
