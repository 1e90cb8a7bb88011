/*
 * bloom_oracle.c -- plain CPU reference of the BLOOM decoder forward, in double.
 *
 * TEST INFRASTRUCTURE ONLY (see bloom_oracle.h).  Written for reading, not for
 * speed: loops follow the definitions one to one.  The only parallelism is an
 * OpenMP loop over output features of each linear layer and over heads.
 */
#include "bloom_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 is the top half of an IEEE binary32; widening is exact. */
double orc_bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double bfv(const uint16_t *p, size_t i) { return p ? orc_bf16_to_double(p[i]) : 0.0; }

int32_t orc_num_threads(void) {
#ifdef _OPENMP
    return (int32_t)omp_get_max_threads();
#else
    return 1;
#endif
}

/* ALiBi slopes.  For n heads let m be the largest power of two <= n.  The
 * first m heads get 2^(-8 i / m), i = 1..m (the closed form 2^(-8i/n) when n is
 * a power of two).  The other n - m heads take every other term of the
 * sequence built for 2m heads, 2^(-8 i / (2m)) with i = 1, 3, 5, ..., in that
 * order.  (Positions are added once per head, centrally, as in "Hugging Face
 * BLOOM Inference Optimization", "Efficient PyTorch Implementation".) */
void orc_alibi_slopes(int32_t n, double *out) {
    int32_t m = 1;
    while (m * 2 <= n) m *= 2;
    for (int32_t i = 1; i <= m; ++i) out[i - 1] = pow(2.0, -8.0 * (double)i / (double)m);
    for (int32_t j = 0; j < n - m; ++j) {
        int32_t i = 2 * j + 1;
        out[m + j] = pow(2.0, -8.0 * (double)i / (double)(2 * m));
    }
}

/* tanh approximation of GeLU with the BLOOM constants (the jit-fused
 * bloom_gelu_forward of "Hugging Face BLOOM Inference Optimization",
 * "Kernel Fusion with torch.jit.script"). */
double orc_gelu(double x) {
    return x * 0.5 * (1.0 + tanh(0.79788456 * x * (1.0 + 0.044715 * x * x)));
}

/* LayerNorm: biased variance over h, eps inside the square root, affine. */
void orc_layernorm(int32_t h, const double *x, const uint16_t *g, const uint16_t *b,
                   double eps, double *y) {
    double mean = 0.0;
    for (int32_t i = 0; i < h; ++i) mean += x[i];
    mean /= (double)h;
    double var = 0.0;
    for (int32_t i = 0; i < h; ++i) var += (x[i] - mean) * (x[i] - mean);
    var /= (double)h;
    double r = 1.0 / sqrt(var + eps);
    for (int32_t i = 0; i < h; ++i) {
        double gi = g ? orc_bf16_to_double(g[i]) : 1.0;
        double bi = b ? orc_bf16_to_double(b[i]) : 0.0;
        y[i] = (x[i] - mean) * r * gi + bi;
    }
}

/* Weight W[n][k] of a linear layer, widened to double. */
static double weight_at(const orc_linear *L, int32_t K, int32_t n, int32_t k) {
    size_t i = (size_t)n * (size_t)K + (size_t)k;
    if (L->w) return orc_bf16_to_double(L->w[i]);
    return (double)L->q[i] * orc_bf16_to_double(L->s[n]);
}

void orc_linear_apply(const orc_linear *L, int32_t N, int32_t K, int32_t M,
                      const double *x, double *y) {
#pragma omp parallel
    {
        double *row = (double *)malloc(sizeof(double) * (size_t)K);
#pragma omp for schedule(static)
        for (int32_t n = 0; n < N; ++n) {
            for (int32_t k = 0; k < K; ++k) row[k] = weight_at(L, K, n, k);
            double bias = bfv(L->b, (size_t)n);
            for (int32_t t = 0; t < M; ++t) {
                const double *xt = x + (size_t)t * (size_t)K;
                double acc = 0.0;
                for (int32_t k = 0; k < K; ++k) acc += row[k] * xt[k];
                y[(size_t)t * (size_t)N + (size_t)n] = acc + bias;
            }
        }
        free(row);
    }
}

/* One query against nk keys: scaled dot product, plus slope * pos_k, masked
 * keys excluded, softmax with the maximum subtracted, weighted sum of values. */
void orc_attend(int32_t d, int32_t nk, const double *q, const double *keys,
                const double *vals, const int32_t *pos, double slope,
                double *o, double *probs) {
    double *s = (double *)malloc(sizeof(double) * (size_t)(nk > 0 ? nk : 1));
    double inv_sqrt_d = 1.0 / sqrt((double)d);
    double mx = -INFINITY;
    for (int32_t k = 0; k < nk; ++k) {
        if (pos[k] < 0) continue;
        double dot = 0.0;
        for (int32_t e = 0; e < d; ++e) dot += q[e] * keys[(size_t)k * d + e];
        s[k] = dot * inv_sqrt_d + slope * (double)pos[k];
        if (s[k] > mx) mx = s[k];
    }
    for (int32_t e = 0; e < d; ++e) o[e] = 0.0;
    double l = 0.0;
    for (int32_t k = 0; k < nk; ++k) {
        double p = (pos[k] < 0) ? 0.0 : exp(s[k] - mx);
        s[k] = p;
        l += p;
    }
    for (int32_t k = 0; k < nk; ++k) {
        double p = (l > 0.0) ? s[k] / l : 0.0;
        if (probs) probs[k] = p;
        if (p == 0.0) continue;
        for (int32_t e = 0; e < d; ++e) o[e] += p * vals[(size_t)k * d + e];
    }
    free(s);
}

int32_t orc_argmax(int32_t n, const double *v) {
    int32_t best = 0;
    for (int32_t i = 1; i < n; ++i)
        if (v[i] > v[best]) best = i;
    return best;
}

orc_seq *orc_seq_new(const orc_config *c, int32_t max_seq) {
    orc_seq *s = (orc_seq *)calloc(1, sizeof(orc_seq));
    size_t n = (size_t)c->n_layer * (size_t)c->n_head * (size_t)max_seq *
               (size_t)(c->hidden / c->n_head);
    s->max_seq = max_seq;
    s->pos = (int32_t *)malloc(sizeof(int32_t) * (size_t)max_seq);
    for (int32_t i = 0; i < max_seq; ++i) s->pos[i] = -1;
    s->k = (double *)calloc(n, sizeof(double));
    s->v = (double *)calloc(n, sizeof(double));
    return s;
}

void orc_seq_free(orc_seq *s) {
    if (!s) return;
    free(s->pos);
    free(s->k);
    free(s->v);
    free(s);
}

/* Position of slot t = (number of tokens at slots <= t) - 1; pads get -1. */
void orc_seq_set_prompt(orc_seq *s, int32_t T, const uint8_t *mask) {
    int32_t count = 0;
    for (int32_t t = 0; t < T; ++t) {
        if (mask[t]) s->pos[t] = count++;
        else s->pos[t] = -1;
    }
    s->len = T;
    s->next_pos = count;
}

void orc_seq_advance(orc_seq *s) {
    s->len += 1;
    s->next_pos += 1;
}

static double *kv_at(const orc_config *c, double *base, const orc_seq *s, int32_t layer,
                     int32_t head, int32_t slot) {
    int32_t d = c->hidden / c->n_head;
    size_t i = (((size_t)layer * (size_t)c->n_head + (size_t)head) * (size_t)s->max_seq +
                (size_t)slot) * (size_t)d;
    return base + i;
}

/* MLP half of the block and the attention output projection, shared by the
 * prefill and decode forms: x += Wo o + bo; x += Wdown gelu(Wup LN2(x) + bup) + bdown. */
static void block_tail(const orc_config *c, const orc_layer *L, int32_t M, double *x,
                       const double *o) {
    int32_t h = c->hidden, F = c->ffn;
    double *y = (double *)malloc(sizeof(double) * (size_t)M * (size_t)h);
    double *m = (double *)malloc(sizeof(double) * (size_t)M * (size_t)h);
    double *u = (double *)malloc(sizeof(double) * (size_t)M * (size_t)F);
    orc_linear_apply(&L->o, h, h, M, o, y);
    for (size_t i = 0; i < (size_t)M * (size_t)h; ++i) x[i] += y[i];
    for (int32_t t = 0; t < M; ++t)
        orc_layernorm(h, x + (size_t)t * h, L->ln2_g, L->ln2_b, c->ln_eps, m + (size_t)t * h);
    orc_linear_apply(&L->up, F, h, M, m, u);
    for (size_t i = 0; i < (size_t)M * (size_t)F; ++i) u[i] = orc_gelu(u[i]);
    orc_linear_apply(&L->down, h, F, M, u, y);
    for (size_t i = 0; i < (size_t)M * (size_t)h; ++i) x[i] += y[i];
    free(y);
    free(m);
    free(u);
}

void orc_layer_prefill(const orc_config *c, const orc_layer *L, int32_t layer, int32_t T,
                       const int32_t *pos, double *x, orc_seq *seq) {
    int32_t h = c->hidden, n = c->n_head, d = h / n;
    double *slopes = (double *)malloc(sizeof(double) * (size_t)n);
    orc_alibi_slopes(n, slopes);
    double *a = (double *)malloc(sizeof(double) * (size_t)T * h);
    double *qkv = (double *)malloc(sizeof(double) * (size_t)T * 3 * h);
    double *o = (double *)malloc(sizeof(double) * (size_t)T * h);
    for (int32_t t = 0; t < T; ++t)
        orc_layernorm(h, x + (size_t)t * h, L->ln1_g, L->ln1_b, c->ln_eps, a + (size_t)t * h);
    orc_linear_apply(&L->qkv, 3 * h, h, T, a, qkv);
#pragma omp parallel for schedule(static)
    for (int32_t j = 0; j < n; ++j) {
        /* fused-QKV rows are head-interleaved: head j owns rows [3jd, 3jd+3d)
         * as q | k | v */
        double *K = (double *)malloc(sizeof(double) * (size_t)T * d);
        double *V = (double *)malloc(sizeof(double) * (size_t)T * d);
        for (int32_t t = 0; t < T; ++t)
            for (int32_t e = 0; e < d; ++e) {
                K[(size_t)t * d + e] = qkv[(size_t)t * 3 * h + (size_t)(3 * j + 1) * d + e];
                V[(size_t)t * d + e] = qkv[(size_t)t * 3 * h + (size_t)(3 * j + 2) * d + e];
            }
        if (seq) {
            for (int32_t t = 0; t < T; ++t) {
                memcpy(kv_at(c, seq->k, seq, layer, j, t), K + (size_t)t * d, sizeof(double) * d);
                memcpy(kv_at(c, seq->v, seq, layer, j, t), V + (size_t)t * d, sizeof(double) * d);
            }
        }
        for (int32_t t = 0; t < T; ++t) {
            double *ot = o + (size_t)t * h + (size_t)j * d;
            if (pos[t] < 0) { /* a pad query has no key: output 0 */
                for (int32_t e = 0; e < d; ++e) ot[e] = 0.0;
                continue;
            }
            const double *q = qkv + (size_t)t * 3 * h + (size_t)(3 * j) * d;
            orc_attend(d, t + 1, q, K, V, pos, slopes[j], ot, NULL); /* causal: keys 0..t */
        }
        free(K);
        free(V);
    }
    block_tail(c, L, T, x, o);
    free(slopes);
    free(a);
    free(qkv);
    free(o);
}

void orc_layer_decode(const orc_config *c, const orc_layer *L, int32_t layer, double *x,
                      orc_seq *seq) {
    int32_t h = c->hidden, n = c->n_head, d = h / n;
    int32_t slot = seq->len;
    seq->pos[slot] = seq->next_pos;
    double *slopes = (double *)malloc(sizeof(double) * (size_t)n);
    orc_alibi_slopes(n, slopes);
    double *a = (double *)malloc(sizeof(double) * (size_t)h);
    double *qkv = (double *)malloc(sizeof(double) * (size_t)3 * h);
    double *o = (double *)malloc(sizeof(double) * (size_t)h);
    orc_layernorm(h, x, L->ln1_g, L->ln1_b, c->ln_eps, a);
    orc_linear_apply(&L->qkv, 3 * h, h, 1, a, qkv);
    for (int32_t j = 0; j < n; ++j) {
        memcpy(kv_at(c, seq->k, seq, layer, j, slot), qkv + (size_t)(3 * j + 1) * d,
               sizeof(double) * d);
        memcpy(kv_at(c, seq->v, seq, layer, j, slot), qkv + (size_t)(3 * j + 2) * d,
               sizeof(double) * d);
        orc_attend(d, slot + 1, qkv + (size_t)(3 * j) * d, kv_at(c, seq->k, seq, layer, j, 0),
                   kv_at(c, seq->v, seq, layer, j, 0), seq->pos, slopes[j], o + (size_t)j * d,
                   NULL);
    }
    block_tail(c, L, 1, x, o);
    free(slopes);
    free(a);
    free(qkv);
    free(o);
}

void orc_embed(const orc_config *c, const orc_weights *w, int32_t n, const int32_t *tok,
               double *x) {
    int32_t h = c->hidden;
    double *row = (double *)malloc(sizeof(double) * (size_t)h);
    for (int32_t i = 0; i < n; ++i) {
        for (int32_t e = 0; e < h; ++e)
            row[e] = orc_bf16_to_double(w->word_emb[(size_t)tok[i] * h + e]);
        orc_layernorm(h, row, w->emb_ln_g, w->emb_ln_b, c->ln_eps, x + (size_t)i * h);
    }
    free(row);
}

/* Tied head: logits = E LN_f(x), no bias. */
void orc_head(const orc_config *c, const orc_weights *w, int32_t n, const double *x,
              double *logits) {
    int32_t h = c->hidden;
    double *xf = (double *)malloc(sizeof(double) * (size_t)n * h);
    for (int32_t i = 0; i < n; ++i)
        orc_layernorm(h, x + (size_t)i * h, w->lnf_g, w->lnf_b, c->ln_eps, xf + (size_t)i * h);
    orc_linear head = {w->word_emb, NULL, NULL, NULL};
    orc_linear_apply(&head, c->vocab, h, n, xf, logits);
    free(xf);
}

void orc_prefill(const orc_config *c, const orc_weights *w, int32_t B, int32_t T,
                 const int32_t *tokens, const uint8_t *mask, orc_seq **seqs,
                 double *logits, double *taps) {
    int32_t h = c->hidden;
    double *x = (double *)malloc(sizeof(double) * (size_t)T * h);
    double *last = (double *)malloc(sizeof(double) * (size_t)B * h);
    for (int32_t b = 0; b < B; ++b) {
        const int32_t *tok = tokens + (size_t)b * T;
        const uint8_t *mk = mask + (size_t)b * T;
        orc_seq_set_prompt(seqs[b], T, mk);
        orc_embed(c, w, T, tok, x);
        if (taps) memcpy(taps + ((size_t)0 * B + b) * T * h, x, sizeof(double) * (size_t)T * h);
        for (int32_t l = 0; l < c->n_layer; ++l) {
            orc_layer_prefill(c, &w->layers[l], l, T, seqs[b]->pos, x, seqs[b]);
            if (taps)
                memcpy(taps + ((size_t)(l + 1) * B + b) * T * h, x,
                       sizeof(double) * (size_t)T * h);
        }
        int32_t tl = -1;
        for (int32_t t = 0; t < T; ++t)
            if (mk[t]) tl = t;
        if (tl < 0) tl = T - 1; /* no token: caller's error; keep memory safe */
        memcpy(last + (size_t)b * h, x + (size_t)tl * h, sizeof(double) * h);
    }
    orc_head(c, w, B, last, logits);
    free(x);
    free(last);
}

void orc_decode(const orc_config *c, const orc_weights *w, int32_t B, const int32_t *tokens,
                orc_seq **seqs, double *logits, double *taps) {
    int32_t h = c->hidden;
    double *x = (double *)malloc(sizeof(double) * (size_t)B * h);
    orc_embed(c, w, B, tokens, x);
    if (taps) memcpy(taps, x, sizeof(double) * (size_t)B * h);
    for (int32_t b = 0; b < B; ++b) {
        for (int32_t l = 0; l < c->n_layer; ++l) {
            orc_layer_decode(c, &w->layers[l], l, x + (size_t)b * h, seqs[b]);
            if (taps)
                memcpy(taps + ((size_t)(l + 1) * B + b) * h, x + (size_t)b * h,
                       sizeof(double) * h);
        }
        orc_seq_advance(seqs[b]);
    }
    orc_head(c, w, B, x, logits);
    free(x);
}

void orc_forward_full(const orc_config *c, const orc_weights *w, int32_t T,
                      const int32_t *tokens, const uint8_t *mask, double *logits) {
    int32_t h = c->hidden;
    int32_t *pos = (int32_t *)malloc(sizeof(int32_t) * (size_t)T);
    int32_t count = 0;
    for (int32_t t = 0; t < T; ++t) pos[t] = mask[t] ? count++ : -1;
    double *x = (double *)malloc(sizeof(double) * (size_t)T * h);
    orc_embed(c, w, T, tokens, x);
    for (int32_t l = 0; l < c->n_layer; ++l) orc_layer_prefill(c, &w->layers[l], l, T, pos, x, NULL);
    orc_head(c, w, T, x, logits);
    free(pos);
    free(x);
}
