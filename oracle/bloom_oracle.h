/*
 * bloom_oracle.h -- plain, slow CPU reference of the BLOOM decoder forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or
 * call this library: only the tests, the package's smoke check and the CPU
 * baseline leg of the benchmark use it.  It shares no code, header, table or
 * helper with the CUDA library.
 *
 * What it computes (the pages give the method, not the block arithmetic; the
 * architecture is the BLOOM decoder-only transformer of "BLOOM: A 176B-Parameter
 * Open-Access Multilingual Language Model" as ported to transformers, cf.
 * "Optimization story: Bloom inference", section "Porting to transformers"):
 *
 *   x      = LN_emb(E[token])
 *   per layer:  a = LN1(x);  qkv = Wqkv a + bqkv  (head-interleaved rows)
 *               s_k = q.k_k / sqrt(d) + slope_head * pos_k   for valid k <= t
 *               p = softmax(s) ;  o = sum_k p_k v_k
 *               x = x + Wo o + bo
 *               m = LN2(x);  x = x + Wdown gelu(Wup m + bup) + bdown
 *   logits = E LN_f(x) ;  next = argmax (lowest index on ties)
 *
 * Greedy generation with a KV cache ("Incredibly Fast BLOOM Inference with
 * DeepSpeed and Accelerate", Benchmark Environment: greedy, do_sample=False,
 * KV cache on).  Masked scores take no part in the softmax, which is what the
 * masked_fill + float32 softmax of "Hugging Face BLOOM Inference Optimization",
 * section "Custom CUDA Kernels and Hardware Acceleration", computes.
 *
 * All arithmetic is IEEE double.  Weights arrive as bf16 bit patterns (or int8
 * codes with bf16 per-row scales) and are widened exactly.  Activations are
 * never rounded to bf16 here.
 *
 * Parity pins live in tests/ (closed forms, library routines, invariants,
 * brute force on tiny shapes).  Every function below is pinned by one of them.
 */
#ifndef BLOOM_ORACLE_H
#define BLOOM_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    int32_t n_layer;
    int32_t hidden;   /* h */
    int32_t n_head;   /* n; head_dim d = h / n */
    int32_t ffn;      /* F (4h for BLOOM) */
    int32_t vocab;    /* V */
    double  ln_eps;
    int32_t int8;     /* 1: block linears given as int8 codes + bf16 row scales */
} orc_config;

/* One linear layer y = W x + b, W is [N][K] row-major.
 * bf16 form: w != NULL.  int8 form: q != NULL and s != NULL (W = q * s[n]). */
typedef struct {
    const uint16_t *w;
    const int8_t   *q;
    const uint16_t *s;
    const uint16_t *b;   /* [N] bf16, may be NULL (zero bias) */
} orc_linear;

typedef struct {
    const uint16_t *ln1_g, *ln1_b;   /* [h] */
    orc_linear qkv;                  /* [3h][h] */
    orc_linear o;                    /* [h][h]  */
    const uint16_t *ln2_g, *ln2_b;   /* [h] */
    orc_linear up;                   /* [F][h]  */
    orc_linear down;                 /* [h][F]  */
} orc_layer;

typedef struct {
    const uint16_t *word_emb;        /* [V][h], also the tied LM head */
    const uint16_t *emb_ln_g, *emb_ln_b;
    const uint16_t *lnf_g, *lnf_b;
    const orc_layer *layers;         /* [n_layer] */
} orc_weights;

/* Per-sequence KV cache of the oracle. */
typedef struct {
    int32_t max_seq;
    int32_t len;        /* slots filled (valid and pad) */
    int32_t next_pos;   /* ALiBi position the next valid token gets */
    int32_t *pos;       /* [max_seq]; -1 marks a pad slot */
    double  *k;         /* [n_layer][n_head][max_seq][d] */
    double  *v;         /* same */
} orc_seq;

/* ---- building blocks (each pinned on its own by tests) ---- */
double orc_bf16_to_double(uint16_t b);
void   orc_alibi_slopes(int32_t n_head, double *out);
double orc_gelu(double x);
void   orc_layernorm(int32_t h, const double *x, const uint16_t *g, const uint16_t *b,
                     double eps, double *y);
/* y[M][N] = x[M][K] W^T + b */
void   orc_linear_apply(const orc_linear *L, int32_t N, int32_t K, int32_t M,
                        const double *x, double *y);
/* Attention of one query against keys 0..nk-1 of one head.
 * q[d], keys[nk][d], vals[nk][d], pos[nk] (-1 = masked).  Writes o[d] and, if
 * probs != NULL, the probabilities probs[nk].  If every key is masked, o = 0. */
void   orc_attend(int32_t d, int32_t nk, const double *q, const double *keys,
                  const double *vals, const int32_t *pos, double slope,
                  double *o, double *probs);
/* Lowest index of the maximum. */
int32_t orc_argmax(int32_t n, const double *v);

/* ---- sequences ---- */
orc_seq *orc_seq_new(const orc_config *c, int32_t max_seq);
void     orc_seq_free(orc_seq *s);

/* ---- one layer (for teacher-forced per-layer checks) ----
 * Prefill form: x[T][h] in/out, mask[T] (1 = token).  Stores K,V of the T
 * positions into slots [0,T) of seq if seq != NULL (seq positions must already
 * be set by orc_seq_set_prompt).  Decode form: x[h] in/out for the token at
 * slot seq->len with position seq->next_pos; it appends K,V at that slot but
 * does not advance seq (orc_seq_advance does). */
void orc_seq_set_prompt(orc_seq *s, int32_t T, const uint8_t *mask);
void orc_seq_advance(orc_seq *s);
void orc_layer_prefill(const orc_config *c, const orc_layer *L, int32_t layer,
                       int32_t T, const int32_t *pos, double *x, orc_seq *seq);
void orc_layer_decode(const orc_config *c, const orc_layer *L, int32_t layer,
                      double *x, orc_seq *seq);

/* ---- whole model ---- */
void orc_embed(const orc_config *c, const orc_weights *w, int32_t n, const int32_t *tok,
               double *x);
void orc_head(const orc_config *c, const orc_weights *w, int32_t n, const double *x,
              double *logits);

/* Prefill B prompts of T slots each (tokens[B][T], mask[B][T], 1 = token; each row
 * needs at least one token).  Fills the caches seqs[b] (len = T) and writes the
 * logits of each row's last valid position to logits[B][V].  taps, if not NULL,
 * receives the hidden states [n_layer+1][B][T][h] (embedding output, then the
 * output of every layer). */
void orc_prefill(const orc_config *c, const orc_weights *w, int32_t B, int32_t T,
                 const int32_t *tokens, const uint8_t *mask, orc_seq **seqs,
                 double *logits, double *taps);

/* One decode step: token[b] goes to slot seqs[b]->len; logits[B][V].
 * taps, if not NULL, receives [n_layer+1][B][h]. */
void orc_decode(const orc_config *c, const orc_weights *w, int32_t B,
                const int32_t *tokens, orc_seq **seqs, double *logits, double *taps);

/* Whole-sequence recompute without a cache (one sequence), logits of every
 * position [T][V] (pad positions get the value of an all-masked row). */
void orc_forward_full(const orc_config *c, const orc_weights *w, int32_t T,
                      const int32_t *tokens, const uint8_t *mask, double *logits);

/* Threads the library uses (OpenMP), for reporting. */
int32_t orc_num_threads(void);

#ifdef __cplusplus
}
#endif
#endif
