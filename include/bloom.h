/*
 * bloom.h -- C ABI of the GB300 (sm_103a) BLOOM decoder engine.
 *
 * One job: KV-cached greedy token generation through a BLOOM-architecture
 * decoder stack on one GPU.  A generation is one prefill of the padded prompts
 * followed by one decode step per new token, the argmax token fed back in
 * ("Incredibly Fast BLOOM Inference with DeepSpeed and Accelerate", Benchmark
 * Environment: greedy, do_sample=False, KV cache enabled; per-token cost =
 * wall time / (batch x tokens)).
 *
 * The block (BLOOM as ported to transformers, "Optimization story: Bloom
 * inference", Porting to transformers):
 *   x = LN_emb(E[tok]);  per layer:  a = LN1(x); qkv = Wqkv a + bqkv;
 *   ALiBi attention with masked keys excluded and a float32 softmax
 *   ("Hugging Face BLOOM Inference Optimization", Custom CUDA Kernels);
 *   x += Wo o + bo;  x += Wdown gelu_tanh(Wup LN2(x) + bup) + bdown
 *   ("Kernel Fusion with torch.jit.script" for the GeLU);
 *   logits = E LN_f(x) (tied head); next = argmax, lowest index on ties.
 *
 * Conventions (all entry points):
 *  - Every tensor pointer is a DEVICE pointer owned by the caller unless the
 *    argument says "host".  The library borrows weights for the model's life.
 *  - Weights use the nn.Linear layout [out][in], row-major, bf16 (IEEE
 *    binary16-brain) or int8 with one bf16 scale per output row (W = q * s).
 *    Row pointers of every matrix must be 16-byte aligned (in % 8 == 0 for
 *    bf16, in % 16 == 0 for int8, base 16-byte aligned).
 *  - Fused QKV rows are head-interleaved: row (3*j + c)*d + e holds head j,
 *    c = 0 (query) / 1 (key) / 2 (value), element e, d = hidden / n_head.
 *  - Calls are asynchronous on the given CUDA stream (a cudaStream_t; NULL =
 *    the legacy default stream) and return a status validated on the host
 *    before anything is launched.  A kernel that meets a bad value (a token
 *    id >= vocab, a slot beyond the cache) records it in a device flag that
 *    bloom_check_device() reports; kernels never trap.
 *  - A model is not thread-safe; calls on one model must be issued in order
 *    on one stream.  Models are independent of one another.
 */
#ifndef BLOOM_H
#define BLOOM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    BLOOM_OK = 0,
    BLOOM_E_INVALID = 1,      /* null / misaligned pointer, bad size or value */
    BLOOM_E_UNSUPPORTED = 2,  /* shape the kernels do not implement (see bloom_create) */
    BLOOM_E_OOM = 3,          /* device workspace allocation failed */
    BLOOM_E_CAPACITY = 4,     /* batch above the cache's, or cache full */
    BLOOM_E_CUDA = 5,         /* a CUDA runtime call failed; see bloom_last_error() */
    BLOOM_E_DEVICE_FLAG = 6   /* a kernel recorded a bad value (bloom_check_device) */
} bloom_status;

enum { BLOOM_WEIGHT_BF16 = 0, BLOOM_WEIGHT_INT8 = 1 };

/* flags */
enum {
    BLOOM_FLAG_NO_GRAPH = 1,  /* launch decode steps one kernel at a time (debug, profiling) */
    BLOOM_FLAG_NO_PDL = 2,    /* launch without programmatic dependent launch (each kernel
                                 waits for the previous one to finish before it starts) */
    BLOOM_FLAG_NO_LN_FUSION = 4, /* run every LayerNorm as its own kernel instead of inside
                                    the decode linear kernel that consumes it */
    BLOOM_FLAG_NO_TC_GEMM = 8    /* every linear on the weight-streaming kernel instead of the
                                    tensor-core (tcgen05) kernels: the prefill GEMM (>= 128
                                    tokens), the decode LM head (>= 3 sequences) and the decode
                                    block linears (bf16: every batch size where each block matrix
                                    is at most one wave of 128-row tiles, else >= 3 sequences;
                                    int8: 3..128 sequences) */
};

typedef struct {
    int32_t n_layer;
    int32_t hidden;        /* h; multiple of 256 */
    int32_t n_head;        /* n; head_dim d = h / n must be 64 or 128 */
    int32_t ffn;           /* F (4h in BLOOM); multiple of 256 */
    int32_t vocab;         /* V; the tied embedding has V rows */
    float   ln_eps;        /* LayerNorm epsilon (1e-5 in BLOOM) */
    int32_t weight_dtype;  /* BLOOM_WEIGHT_BF16 or BLOOM_WEIGHT_INT8 (block linears only;
                              the embedding / LM head is always bf16) */
    int32_t max_batch;     /* largest batch of any call */
    int32_t max_tokens;    /* largest B*T of any prefill (sizes the activation workspace) */
    int32_t max_seq;       /* largest cache length (prompt + generated) of any call */
    int32_t flags;         /* BLOOM_FLAG_* */
    int32_t wait_us;       /* bound of every wait of the tensor-core kernels in microseconds,
                              0 = about two seconds.  A wait that expires makes its launch give
                              up (stores skipped, memory it holds freed once its own copies and
                              MMAs have landed) and sets flag 8 for bloom_check_device; the model
                              stays usable.  Waits for the kernel's own copies and MMAs in
                              flight keep the default bound. */
} bloom_config;

/* One linear layer: bf16 weight, or int8 codes + bf16 row scales. */
typedef struct {
    const void *w;         /* bf16 [N][K] or int8 [N][K] */
    const void *scale;     /* bf16 [N] for int8, else NULL */
    const void *bias;      /* bf16 [N] or NULL (zero bias) */
} bloom_linear;

typedef struct {
    const void *ln1_g, *ln1_b;     /* bf16 [h] */
    bloom_linear qkv;              /* [3h][h] */
    bloom_linear o;                /* [h][h] */
    const void *ln2_g, *ln2_b;     /* bf16 [h] */
    bloom_linear up;               /* [F][h] */
    bloom_linear down;             /* [h][F] */
} bloom_layer_weights;

typedef struct {
    const void *word_emb;          /* bf16 [V][h]; also the tied LM head */
    const void *emb_ln_g, *emb_ln_b;
    const void *lnf_g, *lnf_b;
    const bloom_layer_weights *layers;   /* HOST array [n_layer] of device pointers */
} bloom_weights;

typedef struct bloom_model bloom_model;   /* opaque */

/* KV cache: one caller-owned device allocation of bloom_kv_bytes() bytes, one
 * row per sequence.  Layout (all regions 256-byte aligned): a 256-byte header,
 * int32 len[batch] (slots filled in each row), int32 active[batch] (1 = the row
 * takes part in decode steps), int32 next_pos[batch] (ALiBi position of each
 * row's next token), int32 pos[batch][max_seq] (position of each slot, -1 for a
 * pad slot), then K and V, each bf16 [n_layer][batch][n_head][max_seq][d].
 * The device copy is authoritative; the struct keeps a host mirror of the
 * per-row state, which the library updates on every call (the caller only
 * reads it).  Rows leave and join between decode steps (bloom_kv_retire,
 * bloom_kv_admit): "Hugging Face BLOOM Inference Optimization", Webserver
 * Architecture and Request Handling (dynamic batch extraction). */
#define BLOOM_MAX_BATCH 256
typedef struct {
    void   *buf;
    size_t  bytes;
    int32_t batch;
    int32_t max_seq;
    int32_t len;                              /* longest active row */
    int32_t row_len[BLOOM_MAX_BATCH];         /* slots filled, per row */
    uint8_t row_active[BLOOM_MAX_BATCH];      /* 1: the row decodes */
    void   *host_buf;                         /* K / V of layers >= offload_from (NULL: none) */
    size_t  host_bytes;
    int32_t offload_from;                     /* first layer kept in host_buf (n_layer: none) */
} bloom_kv;

/* Bytes a cache for `batch` sequences of `max_seq` slots needs (0 on bad args). */
size_t bloom_kv_bytes(const bloom_config *cfg, int32_t batch, int32_t max_seq);

/* Validate the config and weights, compute the ALiBi slopes once (largest
 * power of two m <= n heads: 2^(-8i/m), then every other term of the 2m
 * sequence), allocate the activation workspace, and pick launch shapes.
 * The current CUDA device is the model's device.  *out is NULL on failure.
 * For testing the error path, the environment variable BLOOM_INJECT_FAILURE
 * containing "workspace" makes the workspace allocation fail (BLOOM_E_OOM).
 * For testing that no kernel reads an activation before writing it, the
 * variable BLOOM_POISON_WORKSPACE fills the workspace with 0xff bytes (NaN in
 * bf16 and float32) instead of zeros, all but its tickets, argmax scratch and
 * flag word; results must not change. */
bloom_status bloom_create(const bloom_config *cfg, const bloom_weights *w, bloom_model **out);

/* Bind `buf` (device, >= bloom_kv_bytes bytes, 256-byte aligned) as an empty
 * cache and fill *kv: every row empty and idle, every slot a pad. */
bloom_status bloom_kv_init(bloom_model *m, bloom_kv *kv, void *buf, size_t bytes,
                           int32_t batch, int32_t max_seq, void *stream);

/* KV offload to host memory ("DeepSpeed Inference", IV.C.2 Offloading
 * Activations to CPU Memory: cached keys and values beyond what the GPU
 * should hold go to CPU memory, so that larger batches fit; IV.C.3 overlaps
 * the PCIe traffic with compute.  On GB300 the Grace memory is read and
 * written by the kernels themselves over NVLink-C2C, with no copies to
 * schedule): the K and V of layers [offload_from, n_layer) live in host_buf,
 * everything else in buf.  Sizes of both parts (offload_from = n_layer:
 * host_bytes = 0, device_bytes = bloom_kv_bytes).  BLOOM_E_INVALID on bad
 * arguments. */
bloom_status bloom_kv_bytes_offload(const bloom_config *cfg, int32_t batch, int32_t max_seq,
                                    int32_t offload_from, size_t *device_bytes,
                                    size_t *host_bytes);

/* bloom_kv_init with layers [offload_from, n_layer) in host_buf: page-locked
 * host memory (cudaHostAlloc / cudaMallocHost, 256-byte aligned) that the
 * device addresses with the same pointer -- checked, else BLOOM_E_INVALID.
 * The caller owns both buffers.  Decode and prefill kernels read and write the
 * offloaded layers' cache directly (zero-copy), at the host link's bandwidth. */
bloom_status bloom_kv_init_offload(bloom_model *m, bloom_kv *kv, void *buf, size_t bytes,
                                   void *host_buf, size_t host_bytes, int32_t batch,
                                   int32_t max_seq, int32_t offload_from, void *stream);

/* Prefill: run the B x T padded prompts (tokens int32 [B][T], mask uint8 [B][T],
 * 1 = token, 0 = pad; each row needs one token), write K,V of slots [0,T),
 * set slot positions (count of tokens before the slot), and emit the greedy
 * token of each row's last token slot to out_tokens int32 [B].  out_logits
 * (float [B][V]) may be NULL.  Requires B == kv->batch, T <= kv->max_seq,
 * B*T <= max_tokens.  Every row becomes active with length T. */
bloom_status bloom_prefill(bloom_model *m, bloom_kv *kv, const int32_t *tokens,
                           const uint8_t *mask, int32_t B, int32_t T, int32_t *out_tokens,
                           float *out_logits, void *stream);

/* One decode step: next_tokens int32 [B] of every active row go to the row's
 * next slot (row_len); out_tokens int32 [B] receives the greedy next token of
 * each active row and -1 for an idle one, and may alias next_tokens;
 * out_logits float [B][V] may be NULL (idle rows' logits are meaningless).
 * Unless BLOOM_FLAG_NO_GRAPH is set, the step is captured once per distinct
 * (kv, next_tokens, out_tokens, out_logits) into a CUDA graph and replayed; the
 * graph reads the rows' state on the device, so it stays valid across admit
 * and retire.  Each active row grows by one slot; BLOOM_E_CAPACITY if an active
 * row is full, BLOOM_E_INVALID if no row is active. */
bloom_status bloom_decode_step(bloom_model *m, bloom_kv *kv, const int32_t *next_tokens,
                               int32_t *out_tokens, float *out_logits, void *stream);

/* Per-member sampling (temperature + top-p) after the LM head: one decode step
 * (bloom_decode_step, logits into `logits`, float [B][V], device, required),
 * then each active row's next token drawn from its logits by bloom_op_sample
 * with its own temperature[b], top_p[b] and uniform number u[b] (device float
 * [B] each; the caller draws u, so the same inputs give the same tokens) into
 * out_tokens; idle rows get -1.  "Hugging Face BLOOM Inference
 * Optimization", Webserver Architecture and Request Handling: the custom
 * generation loop applies each batch member's own sampling parameters. */
bloom_status bloom_decode_step_sampled(bloom_model *m, bloom_kv *kv, const int32_t *next_tokens,
                                       int32_t *out_tokens, float *logits,
                                       const float *temperature, const float *top_p,
                                       const float *u, void *stream);

/* Dynamic batch: prefill n new prompts (tokens int32 [n][T], mask uint8 [n][T],
 * device) into the cache rows rows[i] (HOST int32 [n], distinct, < kv->batch),
 * leaving every other row untouched; those rows become active with length T
 * and take part in the next decode steps.  out_tokens int32 [n] (device)
 * receives each prompt's greedy token, out_logits float [n][V] may be NULL.
 * Requires n * T <= max_tokens. */
bloom_status bloom_kv_admit(bloom_model *m, bloom_kv *kv, const int32_t *rows, int32_t n,
                            const int32_t *tokens, const uint8_t *mask, int32_t T,
                            int32_t *out_tokens, float *out_logits, void *stream);

/* Dynamic batch: rows rows[i] (HOST int32 [n]) leave the batch: decode steps
 * no longer append to them (their out_tokens are -1) until an admit reuses
 * them. */
bloom_status bloom_kv_retire(bloom_model *m, bloom_kv *kv, const int32_t *rows, int32_t n,
                             void *stream);

/* Whole greedy generation with HOST buffers: copies tokens/mask (host int32 /
 * uint8 [B][T]) to the device, prefills, runs n_new - 1 decode steps feeding
 * each argmax back on the device, and copies the n_new tokens of every row to
 * out_host (host int32 [n_new][B]).  Synchronises the stream before returning
 * and reports a device flag as BLOOM_E_DEVICE_FLAG.  Requires T + n_new - 1
 * <= kv->max_seq. */
bloom_status bloom_generate(bloom_model *m, bloom_kv *kv, const int32_t *tokens_host,
                            const uint8_t *mask_host, int32_t B, int32_t T, int32_t n_new,
                            int32_t *out_host, void *stream);

/* Operations and kernels of a decode step, as bloom_decode_profile reports
 * them: code = op | (kernel << 8). */
enum {
    BLOOM_OP_EMBED = 0,       /* embedding gather + embedding LayerNorm */
    BLOOM_OP_LAYERNORM = 1,   /* LN1 / LN2 / ln_f as a kernel of its own */
    BLOOM_OP_QKV = 2,         /* fused QKV + bias + K/V append */
    BLOOM_OP_ATTN = 3,        /* ALiBi attention over the cache */
    BLOOM_OP_DENSE = 4,       /* attention output projection + bias + residual */
    BLOOM_OP_UP = 5,          /* MLP up projection + bias + GeLU */
    BLOOM_OP_DOWN = 6,        /* MLP down projection + bias + residual */
    BLOOM_OP_HEAD = 7         /* tied LM head + argmax */
};
enum {
    BLOOM_KERNEL_EMBED = 0,
    BLOOM_KERNEL_LAYERNORM = 1,
    BLOOM_KERNEL_STREAM = 2,          /* weight-streaming mma.sync linear */
    BLOOM_KERNEL_GEMV_TC = 3,         /* tensor-core (tcgen05) decode linear */
    BLOOM_KERNEL_GEMM_TC = 4,         /* tensor-core (tcgen05) prefill GEMM */
    BLOOM_KERNEL_ATTN = 5,            /* split-KV decode attention */
    BLOOM_KERNEL_ATTN_PREFILL = 6     /* prefill attention */
};

/* One decode step exactly as bloom_decode_step computes it (same kernels,
 * same results, kv->len advanced), but launched one kernel at a time, each
 * starting after the previous one has finished, with a CUDA event recorded
 * on `stream` after every launch; for measuring the share of each kernel in a
 * step.  Fills codes[i] (op | kernel << 8) and ms[i] (the launch's duration,
 * from the previous event) for the first min(cap, launches) launches, sets *n
 * to that count, and synchronises the stream.  codes, ms and n are HOST
 * pointers.  Not for use inside a stream capture. */
bloom_status bloom_decode_profile(bloom_model *m, bloom_kv *kv, const int32_t *next_tokens,
                                  int32_t *out_tokens, int32_t *codes, float *ms, int32_t cap,
                                  int32_t *n, void *stream);

/* Synchronise the stream, read and clear the device flag: BLOOM_OK or
 * BLOOM_E_DEVICE_FLAG (the flag's bits are in bloom_last_error()). */
bloom_status bloom_check_device(bloom_model *m, void *stream);

/* Free the workspace and graphs.  Caller-owned weights and caches are kept. */
bloom_status bloom_destroy(bloom_model *m);

/* Message of the last failing call on this thread ("" if none). */
const char *bloom_last_error(void);

/* Kernel launches one decode step of `batch` sequences issues (for launch
 * accounting): one per operation, less the LayerNorms fused into a linear. */
int32_t bloom_decode_launches(const bloom_model *m, int32_t batch);

/* ------------------------------------------------------------------------
 * Layer-level entry points.  They run one piece of the path on caller
 * buffers, with the same kernels the calls above use; tests use them to feed
 * each layer a reference input (teacher forcing) and to time one kernel.
 * ------------------------------------------------------------------------ */

/* The residual stream x of the layer-level calls is float32: it is the running
 * sum over layers and is kept unrounded; every other activation is bf16. */

/* One decoder layer of the decode step on x (float [kv->batch][h], in/out) for
 * the next token of every active row: it writes the layer's K,V at the row's
 * next slot and sets the slot position, but does not advance the rows. */
bloom_status bloom_layer_decode(bloom_model *m, bloom_kv *kv, int32_t layer, void *x,
                                void *stream);

/* Set the slot positions of a prompt (mask uint8 [B][T]) in the cache and
 * make every row active with length T, as the prefill does before its first
 * layer. */
bloom_status bloom_kv_set_prompt(bloom_model *m, bloom_kv *kv, const uint8_t *mask,
                                 int32_t B, int32_t T, void *stream);

/* One decoder layer of the prefill on x (float [B*T][h], in/out), writing K,V
 * of slots [0,T).  Needs bloom_kv_set_prompt first. */
bloom_status bloom_layer_prefill(bloom_model *m, bloom_kv *kv, int32_t layer, void *x,
                                 int32_t B, int32_t T, void *stream);

/* Final LayerNorm + tied LM head + argmax on x (float [B][h]): out_tokens int32
 * [B], out_logits float [B][V] or NULL. */
bloom_status bloom_head(bloom_model *m, const void *x, int32_t B, int32_t *out_tokens,
                        float *out_logits, void *stream);

/* Tied LM head + argmax alone (one kernel, the model's scratch) on rows that
 * are already normalised by ln_f: xn bf16 [B][h] -> out_tokens int32 [B],
 * out_logits float [B][V] or NULL.  Used to time the head in isolation. */
bloom_status bloom_lm_head(bloom_model *m, const void *xn, int32_t B, int32_t *out_tokens,
                           float *out_logits, void *stream);

/* Embedding gather + embedding LayerNorm: tokens int32 [n] -> x float [n][h]. */
bloom_status bloom_embed(bloom_model *m, const int32_t *tokens, int32_t n, void *x,
                         void *stream);

/* ------------------------------------------------------------------------
 * Operator entry points (no model needed), the kernels of the path on raw
 * buffers.  All bf16 tensors are row-major.
 * ------------------------------------------------------------------------ */

/* y[r] = LN(x[r]) * g + b over h features, float32 statistics, biased
 * variance, eps inside the square root; x, y bf16 [rows][h]; g, b bf16 [h]
 * (NULL: 1 and 0).  h % 8 == 0, h <= 16384. */
bloom_status bloom_op_layernorm(const void *x, const void *g, const void *b, int32_t rows,
                                int32_t h, float eps, void *y, void *stream);

enum {
    BLOOM_EPI_STORE = 0,   /* y = acc + bias */
    BLOOM_EPI_GELU = 1,    /* y = gelu_tanh(acc + bias) */
    BLOOM_EPI_RESID = 2    /* y = y + acc + bias (residual add in place) */
};

/* Weight-streaming linear layer y[M][N] (bf16) = epilogue(x[M][K] W^T + bias)
 * with float32 accumulation; W per bloom_linear.  K % 8 == 0 (bf16) or
 * K % 16 == 0 (int8). */
bloom_status bloom_op_linear(const bloom_linear *lin, int32_t int8, const void *x, int32_t M,
                             int32_t N, int32_t K, int32_t epilogue, void *y, void *stream);

/* The same linear layer on the tensor-core GEMM that prefill uses for batches
 * of >= 128 tokens ("DeepSpeed Inference", III.A and IV.C.1: prompt processing
 * is compute-bound): 128 x 256 output tiles, tcgen05.mma into TMEM, operands
 * moved by TMA.  bf16 weights only (lin->scale must be NULL); x and lin->w
 * 16-byte aligned; K % 8 == 0; any M >= 0 and N >= 1.  Same epilogues and
 * result layout as bloom_op_linear.  BLOOM_E_UNSUPPORTED if the driver cannot
 * describe the operands for TMA. */
bloom_status bloom_op_gemm(const bloom_linear *lin, const void *x, int32_t M, int32_t N,
                           int32_t K, int32_t epilogue, void *y, void *stream);

/* The same linear layer on the tensor-core decode kernel (the decode steps of
 * 3 or more sequences run their linears on it): W is the 128-row operand of
 * tcgen05.mma, the tokens its N operand, both moved by TMA, the accumulator in
 * TMEM; narrow matrices split K over a thread-block cluster whose partials are
 * summed in split order ("DeepSpeed Inference", III.A: small-batch cost is
 * reading W).  int8 = 0: bf16 weights, M <= 256, K % 8 == 0.  int8 = 1: int8
 * codes with bf16 row scales (lin->scale), widened exactly on the chip (to f16,
 * with the activations converted to f16, up to 32 rows; to bf16 above) and
 * scaled per row in the epilogue, M <= 128, K % 16 == 0 ("Incredibly Fast
 * BLOOM Inference...", Key observations: int8 halves the bytes read).  x and
 * lin->w 16-byte aligned.  Same epilogues and result layout as bloom_op_linear. */
bloom_status bloom_op_linear_tc(const bloom_linear *lin, int32_t int8, const void *x, int32_t M,
                                int32_t N, int32_t K, int32_t epilogue, void *y, void *stream);

/* Split-KV decode attention for one token per sequence.
 * q bf16 [B][n][d]; k_cache, v_cache bf16 [B][n][max_seq][d]; pos int32
 * [B][max_seq] (-1 = masked); keys are slots [0, len]; slopes float [n];
 * o bf16 [B][n*d].  d in {64, 128}.  `splits` key ranges per (b, head), 0 =
 * library choice.  q, k_cache, v_cache and o 16-byte aligned (BLOOM_E_INVALID
 * otherwise); K / V in device memory may be staged by bulk copies, K / V in
 * host memory are read directly. */
bloom_status bloom_op_attn_decode(const void *q, const void *k_cache, const void *v_cache,
                                  const int32_t *pos, const float *slopes, int32_t B,
                                  int32_t n_head, int32_t d, int32_t max_seq, int32_t len,
                                  int32_t splits, void *o, void *stream);

/* Temperature + top-p sampling of B rows of float32 logits (row b at logits +
 * b * ld, ld >= V; device).  temperature, top_p, u: device float [B]; out_tokens:
 * device int32 [B].  Row b: p_i proportional to exp((z_i - max z) / temperature);
 * the nucleus is the shortest prefix of the tokens by probability (highest
 * first, equal logits in index order) whose mass reaches top_p; the token is
 * where the nucleus's cumulative mass in vocabulary order first exceeds u times
 * its mass.  temperature <= 0 or NaN: greedy argmax (lowest index on ties);
 * top_p >= 1 or NaN: every token with non-zero mass; top_p <= 0: the most
 * probable token; u < 0 or NaN counts as 0, u >= 1 takes the last nucleus
 * token.  Masses are 2^-40 fixed point of float32 exp, summed in 64-bit
 * integers: the result does not depend on summation order.  NaN logits, and
 * logits more than 27 temperature units below the maximum (mass below 2^-38
 * of the maximum's), take no part.  One cluster of 8 CTAs per row;
 * BLOOM_E_INVALID for null pointers, B outside 1..65535, V < 1 or ld < V. */
bloom_status bloom_op_sample(const float *logits, int32_t B, int32_t V, int64_t ld,
                             const float *temperature, const float *top_p, const float *u,
                             int32_t *out_tokens, void *stream);

/* Tied LM head with fused argmax: logits[m][v] = x[m] . E[v]; out_tokens[m] =
 * lowest index of the row maximum of the float32 logits; out_logits may be
 * NULL.  x bf16 [M][K], E bf16 [V][K]. */
bloom_status bloom_op_lmhead_argmax(const void *x, const void *emb, int32_t M, int32_t V,
                                    int32_t K, int32_t *out_tokens, float *out_logits,
                                    void *stream);

/* ------------------------------------------------------------------------
 * Allocation-free variant (no counterpart on the pages: an addition of this
 * library).
 * ------------------------------------------------------------------------ */

/* Same result as bloom_op_lmhead_argmax, but the call allocates nothing: the
 * kernel's scratch (a completion ticket and one running maximum per row) is a
 * fixed array inside the library, present on every GPU that loads it until the
 * process exits.  For callers that cannot allocate device memory on the call
 * path (cudaMalloc / cudaFree may synchronise the device or fail under memory
 * pressure; a framework's caching allocator may own all GPU memory; serving
 * loops may forbid allocation between requests).
 *  - M <= 256 rows; larger M returns BLOOM_E_CAPACITY and launches nothing.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current and keeps it for the
 *    process; make that first call before any stream capture, and make no call
 *    after a cudaDeviceReset of that device (the kept address would be stale).
 *  - Each call clears the part of the array it uses (cudaMemsetAsync on
 *    `stream`) before its kernel; calls whose work overlaps on the GPU (other
 *    streams, other threads) share the array and race, so serialise them. */
bloom_status bloom_op_lmhead_argmax_noalloc(const void *x, const void *emb, int32_t M,
                                            int32_t V, int32_t K, int32_t *out_tokens,
                                            float *out_logits, void *stream);

#ifdef __cplusplus
}
#endif
#endif
