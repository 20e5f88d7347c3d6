/*
 * kvd_oracle.c -- plain, slow fp64 CPU reference of the KV-cached decoder step.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product library calls, links or includes
 * this file; only the tests, the smoke check and the CPU-baseline leg of the benchmark
 * use it. It shares no code, header, table or constant with the CUDA library.
 *
 * Every function is the plain definition of the result, written loop by loop:
 * no blocking, no fusion, no online softmax, no split. 16-bit inputs are decoded
 * exactly to double; all arithmetic on them is double precision; comparisons of
 * fp32 logits happen in their own precision (exactly, since comparing two floats
 * as doubles gives the same answer).
 *
 * Sources (web pages, cited by title and section):
 *  [W]  readoss.com, "Whisper のデコーダー内部：Beam Search、Logit フィルター、KV キャッシュ"
 *  [S]  agentlenshq.com, "추측 디코딩으로 Whisper 추론 속도 2배 향상"
 *  [N]  agentlenshq.com, "nanoVLM における KV キャッシュ実装"
 *  [A]  aitime.ge, Whisper speculative-decoding article (single-paragraph body with the
 *       "The quick brown sock / fox" example)
 *
 * Element types (argument `dtype`): 0 = IEEE binary16 stored as uint16 bits,
 * 1 = bfloat16 stored as uint16 bits, 2 = IEEE binary64.
 *
 * Error results are bit masks: bit (code - 16) for code 16 = length overflow,
 * 17 = bad parent index, 18 = draft id outside the vocabulary, 19 = NaN logit.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define KVO_ERR_LEN_OVERFLOW (1u << 0)
#define KVO_ERR_BAD_INDEX    (1u << 1)
#define KVO_ERR_BAD_TOKEN    (1u << 2)
#define KVO_ERR_NAN          (1u << 3)

/* ---- number formats ---------------------------------------------------------------- */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double kvo_decode_f16(uint16_t bits)
{
    int sign = (bits >> 15) & 1;
    int expo = (bits >> 10) & 0x1F;
    int frac = bits & 0x3FF;
    double mag;
    if (expo == 0)
        mag = ldexp((double)frac, -24);              /* subnormal: frac * 2^(1-15-10) */
    else if (expo == 31)
        mag = frac ? NAN : INFINITY;
    else
        mag = ldexp((double)(1024 + frac), expo - 25); /* (1 + frac/2^10) * 2^(expo-15) */
    return sign ? -mag : mag;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
double kvo_decode_bf16(uint16_t bits)
{
    int sign = (bits >> 15) & 1;
    int expo = (bits >> 7) & 0xFF;
    int frac = bits & 0x7F;
    double mag;
    if (expo == 0)
        mag = ldexp((double)frac, -133);             /* subnormal: frac * 2^(1-127-7) */
    else if (expo == 255)
        mag = frac ? NAN : INFINITY;
    else
        mag = ldexp((double)(128 + frac), expo - 134); /* (1 + frac/2^7) * 2^(expo-127) */
    return sign ? -mag : mag;
}

static size_t elem_size(int dtype) { return dtype == 2 ? 8 : 2; }

static double load(int dtype, const void *base, int64_t idx)
{
    if (dtype == 0) return kvo_decode_f16(((const uint16_t *)base)[idx]);
    if (dtype == 1) return kvo_decode_bf16(((const uint16_t *)base)[idx]);
    return ((const double *)base)[idx];
}

static void copy_elem(int dtype, void *dst, int64_t di, const void *src, int64_t si)
{
    size_t n = elem_size(dtype);
    memcpy((char *)dst + (size_t)di * n, (const char *)src + (size_t)si * n, n);
}

/* ---- append the new tokens' K/V to the cache ---------------------------------------
 *
 * [N] "KV キャッシュが推論を最適化する方法", steps 2-3: after the first pass only the newest
 * token's K and V are computed, and they are added to the stored per-layer K/V whose
 * shape is (batch, heads, seq_len_cached, head_dim). [W] "Inference 抽象と KV キャッシュ":
 * the self-attention projections of the new token are concatenated onto the cached
 * sequence along the sequence axis.
 *
 * K, V: [batch, heads, capacity, head_dim] with element strides sb, sh, st (1 over D).
 * k_new, v_new: contiguous [batch, heads, q, head_dim].
 * K[b,h,lens_in[b]+j,:] = k_new[b,h,j,:] for j < q; lens_out[b] = lens_in[b] + q.
 * A row with lens_in[b] + q > capacity (or lens_in[b] < 0) is left untouched,
 * lens_out[b] = lens_in[b], and the length-overflow bit is returned.
 */
unsigned kvo_kv_append(int dtype, int batch, int heads, int capacity, int head_dim, int q,
                       void *K, void *V, int64_t sb, int64_t sh, int64_t st,
                       const void *k_new, const void *v_new,
                       const int32_t *lens_in, int32_t *lens_out)
{
    unsigned err = 0;
    for (int b = 0; b < batch; ++b) {
        int32_t len = lens_in[b];
        if (len < 0 || (int64_t)len + q > capacity) {
            err |= KVO_ERR_LEN_OVERFLOW;
            if (lens_out) lens_out[b] = len;
            continue;
        }
        for (int h = 0; h < heads; ++h)
            for (int j = 0; j < q; ++j)
                for (int d = 0; d < head_dim; ++d) {
                    int64_t dst = b * sb + h * sh + (int64_t)(len + j) * st + d;
                    int64_t src = (((int64_t)b * heads + h) * q + j) * head_dim + d;
                    copy_elem(dtype, K, dst, k_new, src);
                    copy_elem(dtype, V, dst, v_new, src);
                }
        if (lens_out) lens_out[b] = len + q;
    }
    return err;
}

/* ---- attention of a query block over cached K/V --------------------------------
 *
 * [N] "KV キャッシュが推論を最適化する方法", step 4: the current token's query is combined
 * with the cached K and V to produce the output. [W] "Inference 抽象と KV キャッシュ": the
 * attention layer sees the whole concatenated key/value sequence, the token just
 * appended included; cross-attention K/V come from the encoder output, are computed
 * on the first pass and then reused. [S] "추측 디코딩이란?" and [A]: the main model checks
 * all candidate tokens in a single forward pass -- query i of a block of nq new tokens
 * sits at absolute position len - nq + i and (causal) sees positions 0 .. len - nq + i.
 * [N] "nanoVLM における技術的実装", item 1: grouped attention, several query heads read
 * one K/V head.
 *
 * q:   contiguous [batch, n_q_heads, nq, head_dim]
 * K,V: [kv_batch, n_kv_heads, capacity, head_dim] with strides sb, sh, st
 * row r reads cache row r / rows_per_kv; query head hq reads KV head hq / (n_q/n_kv).
 * len = lens ? lens[r / rows_per_kv] : fixed_len.
 * out[r,hq,i,:] = sum_{t < limit} softmax_t(scale * q.K_t) V_t in double, where
 * limit = len (non-causal) or len - nq + 1 + i (causal). limit <= 0 gives zeros.
 * Two passes over the positions: max of the scores, then sum of exp(score - max),
 * then the weighted sum of V divided by that sum.
 */
unsigned kvo_attention(int dtype, int batch, int n_q_heads, int nq, int head_dim,
                       const void *q, int n_kv_heads, int capacity,
                       const void *K, const void *V, int64_t sb, int64_t sh, int64_t st,
                       const int32_t *lens, int fixed_len, int rows_per_kv, int causal,
                       double scale, double *out)
{
    unsigned err = 0;
    int group = n_q_heads / n_kv_heads;
    for (int r = 0; r < batch; ++r) {
        int bk = r / rows_per_kv;
        int32_t len = lens ? lens[bk] : fixed_len;
        for (int hq = 0; hq < n_q_heads; ++hq) {
            int h = hq / group;
            for (int i = 0; i < nq; ++i) {
                double *o = out + (((int64_t)r * n_q_heads + hq) * nq + i) * head_dim;
                const int64_t qoff = (((int64_t)r * n_q_heads + hq) * nq + i) * head_dim;
                for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
                if (len < 0 || len > capacity) {
                    err |= KVO_ERR_LEN_OVERFLOW;
                    continue;
                }
                int limit = causal ? len - nq + 1 + i : len;
                if (limit > len) limit = len;
                if (limit <= 0) continue;

                double m = -INFINITY;
                for (int t = 0; t < limit; ++t) {
                    double s = 0.0;
                    for (int d = 0; d < head_dim; ++d)
                        s += load(dtype, q, qoff + d) *
                             load(dtype, K, bk * sb + h * sh + (int64_t)t * st + d);
                    s *= scale;
                    if (s > m) m = s;
                }
                double l = 0.0;
                for (int t = 0; t < limit; ++t) {
                    double s = 0.0;
                    for (int d = 0; d < head_dim; ++d)
                        s += load(dtype, q, qoff + d) *
                             load(dtype, K, bk * sb + h * sh + (int64_t)t * st + d);
                    s *= scale;
                    double w = exp(s - m);
                    l += w;
                    for (int d = 0; d < head_dim; ++d)
                        o[d] += w * load(dtype, V, bk * sb + h * sh + (int64_t)t * st + d);
                }
                for (int d = 0; d < head_dim; ++d) o[d] /= l;
            }
        }
    }
    return err;
}

/* ---- greedy verification -- accept up to the first mismatch ------------------------
 *
 * [W] "Inference 抽象と KV キャッシュ" (GreedyDecoder): at temperature 0 the next token is
 * the argmax of the logits. [S] "추측 디코딩이란?" and [A]: the main model's token at each
 * candidate position is compared with the candidate; candidates are accepted up to the
 * first mismatch, the mismatching candidate is replaced by the main model's token and
 * the rest are dropped. [S] "배치 크기 고려사항": in a batch, every row's candidates must
 * match for the batch to advance together -- n_min is the per-batch minimum.
 *
 * logits: [batch, k+1, vocab] fp32; draft: [batch, k] int32.
 * a_i = argmax_v logits[b,i,v]: the first (lowest) index on ties; a NaN ranks above
 * every number and the first NaN wins; -inf is an ordinary value.
 * n_b = first i < k with draft[b,i] != a_i (an id outside [0, vocab) never matches),
 * or k when all k match; next_b = a_{n_b}. Outputs that are NULL are skipped.
 */
static int beats(float cand, float best)
{
    if (isnan(best)) return 0;
    if (isnan(cand)) return 1;
    return cand > best;
}

unsigned kvo_greedy_accept(int batch, int k, int vocab, const float *logits,
                           const int32_t *draft, int32_t *n_accepted, int32_t *next_token,
                           int32_t *n_min, int32_t *argmax_out)
{
    unsigned err = 0;
    int32_t running_min = k;
    int32_t *amax = (int32_t *)malloc(sizeof(int32_t) * (size_t)(k + 1));
    if (!amax) return ~0u;
    for (int b = 0; b < batch; ++b) {
        for (int i = 0; i <= k; ++i) {
            const float *row = logits + ((int64_t)b * (k + 1) + i) * vocab;
            int32_t best = 0;
            for (int v = 0; v < vocab; ++v) {
                if (isnan(row[v])) err |= KVO_ERR_NAN;
                if (v > 0 && beats(row[v], row[best])) best = v;
            }
            amax[i] = best;
            if (argmax_out) argmax_out[b * (k + 1) + i] = best;
        }
        int32_t n = k;
        for (int i = 0; i < k; ++i) {
            int32_t d = draft[(int64_t)b * k + i];
            if (d < 0 || d >= vocab) err |= KVO_ERR_BAD_TOKEN;
        }
        for (int i = 0; i < k; ++i) {
            int32_t d = draft[(int64_t)b * k + i];
            if (d < 0 || d >= vocab || d != amax[i]) {
                n = i;
                break;
            }
        }
        if (n_accepted) n_accepted[b] = n;
        if (next_token) next_token[b] = amax[n];
        if (n < running_min) running_min = n;
    }
    if (n_min) *n_min = running_min;
    free(amax);
    return err;
}

/* ---- beam-search cache reorder ----------------------------------------------------
 *
 * [W] "Inference 抽象と KV キャッシュ" (BeamSearchDecoder.update and rearrange_kv_cache):
 * after the beams are re-ranked the stored key/value tensors must be put in the new
 * beam order; otherwise a beam would continue from another beam's cache.
 *
 * One layer's K or V: src, dst [rows, heads, capacity, head_dim] with strides sb, sh,
 * st (same for both). Row r belongs to window r / beam; its parent must lie in that
 * window's block [w*beam, (w+1)*beam), else the bad-index bit is set and the row keeps
 * its own data. dst[r,h,t,:] = src[parent[r],h,t,:] for t < len; positions t >= len
 * keep dst[r] = src[r]. len outside [0, capacity] sets the length bit and copies src.
 * Written out-of-place on purpose: dst and src must not overlap.
 */
unsigned kvo_beam_reorder(int dtype, int rows, int beam, int heads, int capacity,
                          int head_dim, int len, const int32_t *parent,
                          const void *src, void *dst, int64_t sb, int64_t sh, int64_t st)
{
    unsigned err = 0;
    if (len < 0 || len > capacity) {
        err |= KVO_ERR_LEN_OVERFLOW;
        len = 0;
    }
    for (int r = 0; r < rows; ++r) {
        int w = r / beam;
        int p = parent[r];
        if (p < w * beam || p >= (w + 1) * beam) {
            err |= KVO_ERR_BAD_INDEX;
            p = r;
        }
        for (int h = 0; h < heads; ++h)
            for (int t = 0; t < capacity; ++t) {
                int from = t < len ? p : r;
                for (int d = 0; d < head_dim; ++d)
                    copy_elem(dtype, dst, r * sb + h * sh + (int64_t)t * st + d,
                              src, from * sb + h * sh + (int64_t)t * st + d);
            }
    }
    return err;
}

/* ---- rotary position encoding at absolute positions ----------------------------
 *
 * [N] "nanoVLM における KV キャッシュ実装" (the LanguageModel passes start_pos so that the
 * rotary position encoding of new tokens matches their absolute position in the
 * sequence). The page gives no formula; this is the usual rotary encoding in its
 * rotate-half form, with theta_i = base^(-2i/D) and a = pos * theta_i for i < D/2:
 *   y[i]       = x[i] cos a - x[i + D/2] sin a
 *   y[i + D/2] = x[i + D/2] cos a + x[i] sin a
 * x: [batch, heads, n, head_dim], contiguous; token j of row b is at pos0[b] + j
 * (pos0 NULL: 0). y: double, same shape. head_dim must be even.
 */
void kvo_rope(int dtype, int batch, int heads, int n, int head_dim, const void *x,
              const int32_t *pos0, double base, double *y)
{
    int half = head_dim / 2;
    for (int b = 0; b < batch; ++b)
        for (int h = 0; h < heads; ++h)
            for (int j = 0; j < n; ++j) {
                double pos = (double)((pos0 ? pos0[b] : 0) + j);
                int64_t row = (((int64_t)b * heads + h) * n + j) * head_dim;
                for (int i = 0; i < half; ++i) {
                    double theta = pow(base, -2.0 * i / head_dim);
                    double a = pos * theta;
                    double x0 = load(dtype, x, row + i);
                    double x1 = load(dtype, x, row + i + half);
                    y[row + i] = x0 * cos(a) - x1 * sin(a);
                    y[row + i + half] = x1 * cos(a) + x0 * sin(a);
                }
            }
}

/* ---- logit filters and one beam-search step ---------------------------------------
 *
 * [W] "LogitFilter チェーン": SuppressBlank sets the logits of the blank (space) ids and
 * of EOT to -inf, at the first sampling position only; SuppressTokens sets the listed
 * ids to -inf at every position. [W] "Inference 抽象と KV キャッシュ"
 * (BeamSearchDecoder.update), for each window of `beam` rows:
 *   1. per beam row, the beam+1 tokens of highest log-probability (log-softmax of the
 *      filtered logits),
 *   2. every continuation (row j, token t) scores cum[j] + logprob_j(t),
 *   3. going from the highest score down, EOT continuations are collected as finished
 *      and the others kept, until `beam` are kept,
 *   4. the kept continuations' rows are the parents the caches are reordered by.
 *
 * Readings where the page is silent: a NaN logit or a NaN cum counts as -inf and sets
 * the NaN bit; tokens of a row rank by logit, ties to the lower id; continuations of
 * equal score keep the order (row, then rank in the row); a row whose filtered logits
 * are all -inf has every log-probability -inf; a suppressed or blank id outside
 * [0, vocab) is skipped and sets the bad-token bit; the EOT continuations collected are
 * those ranked above the last kept one.
 *
 * logits: fp32 [rows, vocab], rows = windows * beam. cum: fp32 [rows] or NULL (zeros).
 * Outputs, each optional (NULL):
 *   row_token, row_logprob [rows, beam+1]: step 1, best first;
 *   parent (absolute row), token, new_cum [rows]: kept continuation s of window w at
 *   w*beam + s, best first;
 *   n_fin [windows]; fin_parent, fin_score [rows]: finished continuation f of window w
 *   at w*beam + f, best first; slots past n_fin[w] hold -1 and -inf.
 */
unsigned kvo_beam_select(int rows, int beam, int vocab, const float *logits, const float *cum,
                         const int32_t *suppress, int n_suppress, const int32_t *blank,
                         int n_blank, int eot, int first_step, int32_t *row_token,
                         double *row_logprob, int32_t *parent, int32_t *token, double *new_cum,
                         int32_t *n_fin, int32_t *fin_parent, double *fin_score)
{
    unsigned err = 0;
    const int kk = beam + 1;
    const int windows = rows / beam;
    double *x = malloc(sizeof(double) * (size_t)vocab);
    char *used = malloc((size_t)vocab);
    double *score = malloc(sizeof(double) * (size_t)beam * kk);
    int *tok = malloc(sizeof(int) * (size_t)beam * kk);
    char *taken = malloc((size_t)beam * kk);
    for (int w = 0; w < windows; ++w) {
        for (int j = 0; j < beam; ++j) {
            const int r = w * beam + j;
            /* the filters */
            for (int v = 0; v < vocab; ++v) {
                x[v] = logits[(int64_t)r * vocab + v];
                if (isnan(x[v])) {
                    err |= KVO_ERR_NAN;
                    x[v] = -INFINITY;
                }
            }
            for (int i = 0; i < n_suppress; ++i) {
                if (suppress[i] < 0 || suppress[i] >= vocab) err |= KVO_ERR_BAD_TOKEN;
                else x[suppress[i]] = -INFINITY;
            }
            if (first_step) {
                for (int i = 0; i < n_blank; ++i) {
                    if (blank[i] < 0 || blank[i] >= vocab) err |= KVO_ERR_BAD_TOKEN;
                    else x[blank[i]] = -INFINITY;
                }
                x[eot] = -INFINITY;
            }
            /* log-softmax: logprob(v) = x[v] - log(sum_u exp(x[u])) */
            double mx = -INFINITY;
            for (int v = 0; v < vocab; ++v)
                if (x[v] > mx) mx = x[v];
            double lse = -INFINITY;
            if (mx > -INFINITY) {
                double sum = 0.0;
                for (int v = 0; v < vocab; ++v) sum += exp(x[v] - mx);
                lse = mx + log(sum);
            }
            /* step 1: the beam+1 best tokens, by logit, ties to the lower id */
            double c = cum ? (double)cum[r] : 0.0;
            if (isnan(c)) {
                err |= KVO_ERR_NAN;
                c = -INFINITY;
            }
            memset(used, 0, (size_t)vocab);
            for (int k = 0; k < kk; ++k) {
                int best = -1;
                for (int v = 0; v < vocab; ++v)
                    if (!used[v] && (best < 0 || x[v] > x[best])) best = v;
                used[best] = 1;
                const double lp = mx > -INFINITY ? x[best] - lse : -INFINITY;
                if (row_token) row_token[(int64_t)r * kk + k] = best;
                if (row_logprob) row_logprob[(int64_t)r * kk + k] = lp;
                /* step 2: the continuation's score */
                score[j * kk + k] = c + lp;
                tok[j * kk + k] = best;
            }
        }
        if (!parent) continue;
        /* step 3: walk the continuations from the highest score down */
        int kept = 0, fin = 0;
        memset(taken, 0, (size_t)beam * kk);
        while (kept < beam) {
            int best = -1;
            for (int cnd = 0; cnd < beam * kk; ++cnd)
                if (!taken[cnd] && (best < 0 || score[cnd] > score[best])) best = cnd;
            taken[best] = 1;
            const int src = w * beam + best / kk;
            if (tok[best] == eot) {
                fin_parent[w * beam + fin] = src;
                fin_score[w * beam + fin] = score[best];
                ++fin;
            } else {
                parent[w * beam + kept] = src;
                token[w * beam + kept] = tok[best];
                new_cum[w * beam + kept] = score[best];
                ++kept;
            }
        }
        n_fin[w] = fin;
        for (int f = fin; f < beam; ++f) {
            fin_parent[w * beam + f] = -1;
            fin_score[w * beam + f] = -INFINITY;
        }
    }
    free(x);
    free(used);
    free(score);
    free(tok);
    free(taken);
    return err;
}

/* ---- temperature sampling and stochastic speculative acceptance -------------------
 *
 * [W] "Inference 抽象と KV キャッシュ": at a temperature above 0 GreedyDecoder samples
 * from Categorical(logits / temperature). [S] "추측 디코딩이란?" names the speculative
 * decoding of Leviathan et al. (2022); with sampling, its verification step is the
 * rejection rule of that paper, written here from its definition:
 *   p_i = softmax(target_i / T), q_i = softmax(draft_i / T), x_i the drafted token;
 *   for i = 0, 1, ...: accept x_i when r_i * q_i(x_i) < p_i(x_i) (i.e. with probability
 *   min(1, p/q)); at the first rejection n = i, the next token is drawn from the
 *   residual max(0, p_n - q_n) (normalised); if all k are accepted, n = k and the next
 *   token is drawn from p_k.
 * A draw from weights w with uniform u in [0, 1) is the inverse CDF in id order: the
 * smallest v whose running sum exceeds u * sum(w) (the last id with w > 0 if rounding
 * leaves none). Readings: the uniforms r[b, i] and u[b] are inputs (the caller's random
 * numbers); a NaN logit counts as -inf and sets the NaN bit; a drafted id outside the
 * vocabulary sets the bad-token bit and is rejected; a residual that sums to 0 falls
 * back to p_n. k = 0 is plain temperature sampling of target row 0.
 *
 * target: fp32 [batch, k+1, vocab]; draft: fp32 [batch, k, vocab] (unused when k = 0);
 * drafts: int32 [batch, k]; r: fp32 [batch, k]; u: fp32 [batch].
 * Outputs: n_acc[b] in 0..k, next[b].
 */
static void softmax_t(const float *x, int vocab, double temperature, double *p, unsigned *err)
{
    double mx = -INFINITY;
    for (int v = 0; v < vocab; ++v) {
        double y = x[v];
        if (isnan(y)) {
            *err |= KVO_ERR_NAN;
            y = -INFINITY;
        }
        p[v] = y / temperature;
        if (p[v] > mx) mx = p[v];
    }
    double s = 0.0;
    for (int v = 0; v < vocab; ++v) {
        p[v] = mx == -INFINITY ? 0.0 : exp(p[v] - mx);
        s += p[v];
    }
    for (int v = 0; v < vocab; ++v) p[v] = s > 0.0 ? p[v] / s : 0.0;
}

static int inverse_cdf(const double *w, int vocab, double u)
{
    double total = 0.0;
    for (int v = 0; v < vocab; ++v) total += w[v];
    double run = 0.0;
    int last = 0;
    for (int v = 0; v < vocab; ++v) {
        if (w[v] > 0.0) last = v;
        run += w[v];
        if (run > u * total) return v;
    }
    return last;
}

unsigned kvo_sample_accept(int batch, int k, int vocab, const float *target, const float *draft,
                           const int32_t *drafts, double temperature, const float *r,
                           const float *u, int32_t *n_acc, int32_t *next)
{
    unsigned err = 0;
    double *p = malloc(sizeof(double) * (size_t)vocab);
    double *q = malloc(sizeof(double) * (size_t)vocab);
    double *w = malloc(sizeof(double) * (size_t)vocab);
    for (int b = 0; b < batch; ++b) {
        int n = k;
        for (int i = 0; i < k; ++i) {
            softmax_t(target + ((int64_t)b * (k + 1) + i) * vocab, vocab, temperature, p, &err);
            softmax_t(draft + ((int64_t)b * k + i) * vocab, vocab, temperature, q, &err);
            const int x = drafts[b * k + i];
            const int ok = x >= 0 && x < vocab;
            if (!ok) err |= KVO_ERR_BAD_TOKEN;
            if (ok && (double)r[b * k + i] * q[x] < p[x]) continue;  /* accepted */
            n = i;
            double s = 0.0;
            for (int v = 0; v < vocab; ++v) {
                w[v] = p[v] - q[v] > 0.0 ? p[v] - q[v] : 0.0;
                s += w[v];
            }
            next[b] = inverse_cdf(s > 0.0 ? w : p, vocab, (double)u[b]);
            break;
        }
        if (n == k) {
            softmax_t(target + ((int64_t)b * (k + 1) + k) * vocab, vocab, temperature, p, &err);
            next[b] = inverse_cdf(p, vocab, (double)u[b]);
        }
        n_acc[b] = n;
    }
    free(p);
    free(q);
    free(w);
    return err;
}
