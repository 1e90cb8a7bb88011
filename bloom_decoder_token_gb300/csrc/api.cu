// C ABI of the BLOOM decode engine: validation, workspace, launch sequences,
// CUDA-graph replay of the decode step.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/bloom.h"
#include <nvtx3/nvToolsExt.h>

#include "kernels.h"

using namespace bloom;

namespace bloom {
thread_local bool g_pdl = true;
// Set while a decode step is captured into a graph: every kernel of an earlier
// step, and of the calls before it, has finished when the graph starts.
static thread_local bool g_capture = false;
}

// ----------------------------------------------------------------- errors
static thread_local std::string g_err;

static bloom_status fail(bloom_status st, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return st;
}

#define CK(call)                                                                         \
    do {                                                                                 \
        cudaError_t e_ = (call);                                                         \
        if (e_ != cudaSuccess)                                                           \
            return fail(BLOOM_E_CUDA, "%s failed: %s (%s:%d)", #call, cudaGetErrorString(e_), \
                        __FILE__, __LINE__);                                             \
    } while (0)

extern "C" const char *bloom_last_error(void) { return g_err.c_str(); }

void bloom::bloom_set_error(const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
}

static bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// NVTX ranges around the host-side phases (prefill, decode step, each layer's
// launches; named in a profiler's timeline, no cost when none is attached).
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};

// Host-side fault injection for tests: BLOOM_INJECT_FAILURE names the
// allocations to fail ("workspace").
static bool inject_failure(const char *what) {
    const char *v = getenv("BLOOM_INJECT_FAILURE");
    return v && strstr(v, what) != nullptr;
}
static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// ----------------------------------------------------------------- KV layout
struct KvLayout {
    size_t len, active, next_pos, pos, k, v, total, layer;   // layer = bytes of one layer's K (or V)
};

// [256-byte header][len int32[B]][active int32[B]][next_pos int32[B]]
// [pos int32[B][S]][K bf16[L][B][n][S][d]][V ...], every region 256-byte aligned.
// hbm_layers: the layers whose K and V live in this buffer (the first ones);
// the rest live in the host buffer of an offloaded cache (kv_host_layout).
static KvLayout kv_layout(const bloom_config &c, int batch, int max_seq, int hbm_layers = -1) {
    if (hbm_layers < 0) hbm_layers = c.n_layer;
    KvLayout L;
    const size_t d = (size_t)(c.hidden / c.n_head);
    size_t off = 256;
    L.len = off;
    off = align256(off + 4 * (size_t)batch);
    L.active = off;
    off = align256(off + 4 * (size_t)batch);
    L.next_pos = off;
    off = align256(off + 4 * (size_t)batch);
    L.pos = off;
    off = align256(off + 4 * (size_t)batch * max_seq);
    L.layer = (size_t)batch * c.n_head * max_seq * d * 2;
    L.k = off;
    off = align256(off + L.layer * hbm_layers);
    L.v = off;
    off = align256(off + L.layer * hbm_layers);
    L.total = off;
    return L;
}

// Host part of an offloaded cache: K then V of layers [offload_from, n_layer).
struct KvHostLayout {
    size_t k, v, total;
};
static KvHostLayout kv_host_layout(const bloom_config &c, int batch, int max_seq, int offload_from) {
    const KvLayout L = kv_layout(c, batch, max_seq);
    const size_t n = (size_t)(c.n_layer - offload_from);
    KvHostLayout H;
    H.k = 0;
    H.v = align256(L.layer * n);
    H.total = align256(H.v + L.layer * n);
    return H;
}

// ----------------------------------------------------------------- model
// A captured decode step.  The graph bakes in every address and stride of the
// cache layout, so it is keyed by the whole cache descriptor (buffer, bytes,
// batch, max_seq) and the step's token / logit buffers.
struct GraphEntry {
    void *kvbuf;
    size_t kvbytes;
    void *hostbuf;      // offloaded layers' K / V (null: none)
    size_t hostbytes;
    int offload_from;
    int B, max_seq;
    const void *next;
    void *out;
    void *logits;
    cudaGraphExec_t exec;
};

// One TMA descriptor (CUtensorMap: 128 bytes, 64-byte aligned).
struct TcMap {
    alignas(64) unsigned char b[128];
};
enum { TC_QKV = 0, TC_O = 1, TC_UP = 2, TC_DOWN = 3, TC_PER_LAYER = 4 };
enum { TC_X_A = 0, TC_X_O = 1, TC_X_U = 2 };
constexpr int kTcNtClasses = 5;   // decode token columns 16, 32, 64, 128, 256

struct bloom_model {
    bloom_config cfg;
    const void *word_emb, *emb_ln_g, *emb_ln_b, *lnf_g, *lnf_b;
    std::vector<bloom_layer_weights> layers;
    int dev = 0, num_sms = 0;
    int d = 0;
    long long attn_resident = 0, attn_resident_wide = 0;   // attn_decode_resident_ctas
    void *ws = nullptr;
    size_t ws_bytes = 0;
    float *x = nullptr;           // float32 residual stream [max_tokens][h]
    uint16_t *a = nullptr, *q = nullptr, *o = nullptr, *u = nullptr, *xl = nullptr;
    float *slopes = nullptr;
    unsigned long long *best = nullptr;
    int *head_ticket = nullptr;
    float *attn_part = nullptr;
    int *attn_ticket = nullptr;
    int *err = nullptr;
    int *last = nullptr;
    int32_t *tok = nullptr;       // [max_batch] device feedback token
    int32_t *gen = nullptr;       // [max_seq][max_batch]
    int32_t *ptok = nullptr;      // [max_tokens] prompt ids (bloom_generate)
    uint8_t *pmask = nullptr;     // [max_tokens]
    int *rowmap = nullptr;        // [max_batch] cache rows of the prompts of bloom_kv_admit
    cudaStream_t cap = nullptr;
    std::vector<GraphEntry> graphs;
    // tensor-core prefill GEMM: weight maps [layer][TC_*], activation maps TC_X_*
    bool tc = false;
    std::vector<TcMap> wmaps;
    TcMap xmaps[3];
    // tensor-core LM head (decode steps, see use_tc_head): the
    // embedding's map (box 128 rows) and the ln_f output's maps per token-column class
    bool tcd = false;
    TcMap head_wmap;
    TcMap head_xmaps[kTcNtClasses];
    // the bf16 block linears of decode steps (see use_tc_linear) on
    // the tensor cores: weight maps [layer][TC_*] (box 128 rows), activation maps
    // [TC_X_*][token-column class]
    bool tcb = false;
    // every block matrix is at most one wave of unsplit tensor-core decode CTAs
    // (two per SM), so one- and two-sequence steps run there too (use_tc_linear)
    bool tc_small = false;
    std::vector<TcMap> dwmaps;
    TcMap dxmaps[3][kTcNtClasses];

};

static int attn_splits(const bloom_model *m, int B, int max_seq) {
    const int want = (2 * m->num_sms + B * m->cfg.n_head - 1) / (B * m->cfg.n_head);
    int cap = (max_seq + 31) / 32;
    int s = want < cap ? want : cap;
    if (s > kMaxSplits) s = kMaxSplits;
    return s < 1 ? 1 : s;
}

static bloom_status check_linear(const bloom_linear &l, int int8, int N, int K, const char *nm,
                                 int layer) {
    (void)N;
    if (!l.w) return fail(BLOOM_E_INVALID, "layer %d %s: null weight", layer, nm);
    if (!aligned16(l.w)) return fail(BLOOM_E_INVALID, "layer %d %s: weight not 16-byte aligned", layer, nm);
    if (int8 && !l.scale) return fail(BLOOM_E_INVALID, "layer %d %s: int8 weight without scales", layer, nm);
    if (!int8 && l.scale) return fail(BLOOM_E_INVALID, "layer %d %s: scales given for bf16 weight", layer, nm);
    if (K % (int8 ? 16 : 8)) return fail(BLOOM_E_UNSUPPORTED, "layer %d %s: K=%d not a multiple of %d", layer, nm, K, int8 ? 16 : 8);
    return BLOOM_OK;
}

static bloom_status validate_config(const bloom_config *c) {
    if (!c) return fail(BLOOM_E_INVALID, "null config");
    if (c->n_layer < 1 || c->hidden < 8 || c->n_head < 1 || c->ffn < 16 || c->vocab < 1)
        return fail(BLOOM_E_INVALID, "non-positive size in config");
    if (c->hidden % c->n_head) return fail(BLOOM_E_INVALID, "hidden %% n_head != 0");
    const int d = c->hidden / c->n_head;
    if (d != 64 && d != 128) return fail(BLOOM_E_UNSUPPORTED, "head_dim %d (64 or 128 supported)", d);
    if (c->hidden % 16 || c->hidden > kMaxHidden)
        return fail(BLOOM_E_UNSUPPORTED, "hidden %d (multiple of 16, <= %d)", c->hidden, kMaxHidden);
    if (c->ffn % 16) return fail(BLOOM_E_UNSUPPORTED, "ffn %d not a multiple of 16", c->ffn);
    if (!(c->ln_eps > 0.f)) return fail(BLOOM_E_INVALID, "ln_eps must be > 0");
    if (c->weight_dtype != BLOOM_WEIGHT_BF16 && c->weight_dtype != BLOOM_WEIGHT_INT8)
        return fail(BLOOM_E_INVALID, "weight_dtype %d", c->weight_dtype);
    if (c->max_batch < 1 || c->max_batch > kMaxBatch)
        return fail(BLOOM_E_UNSUPPORTED, "max_batch %d (1..%d)", c->max_batch, kMaxBatch);
    if (c->max_tokens < c->max_batch) return fail(BLOOM_E_INVALID, "max_tokens < max_batch");
    if (c->max_seq < 1) return fail(BLOOM_E_INVALID, "max_seq < 1");
    if (c->wait_us < 0) return fail(BLOOM_E_INVALID, "wait_us < 0");
    return BLOOM_OK;
}

extern "C" size_t bloom_kv_bytes(const bloom_config *cfg, int32_t batch, int32_t max_seq) {
    if (validate_config(cfg) != BLOOM_OK || batch < 1 || max_seq < 1) return 0;
    return kv_layout(*cfg, batch, max_seq).total;
}

extern "C" bloom_status bloom_kv_bytes_offload(const bloom_config *cfg, int32_t batch,
                                               int32_t max_seq, int32_t offload_from,
                                               size_t *device_bytes, size_t *host_bytes) {
    bloom_status st = validate_config(cfg);
    if (st) return st;
    if (!device_bytes || !host_bytes) return fail(BLOOM_E_INVALID, "null argument");
    if (batch < 1 || max_seq < 1 || offload_from < 0 || offload_from > cfg->n_layer)
        return fail(BLOOM_E_INVALID, "batch %d max_seq %d offload_from %d", batch, max_seq,
                    offload_from);
    *device_bytes = kv_layout(*cfg, batch, max_seq, offload_from).total;
    *host_bytes = offload_from < cfg->n_layer
                      ? kv_host_layout(*cfg, batch, max_seq, offload_from).total : 0;
    return BLOOM_OK;
}

extern "C" bloom_status bloom_destroy(bloom_model *m) {
    if (!m) return BLOOM_OK;
    cudaSetDevice(m->dev);
    for (auto &g : m->graphs) cudaGraphExecDestroy(g.exec);
    if (m->cap) cudaStreamDestroy(m->cap);
    if (m->ws) cudaFree(m->ws);
    delete m;
    return BLOOM_OK;
}

extern "C" bloom_status bloom_create(const bloom_config *cfg, const bloom_weights *w,
                                     bloom_model **out) {
    if (!out) return fail(BLOOM_E_INVALID, "null output handle");
    *out = nullptr;
    bloom_status st = validate_config(cfg);
    if (st) return st;
    if (!w || !w->word_emb || !w->emb_ln_g || !w->emb_ln_b || !w->lnf_g || !w->lnf_b || !w->layers)
        return fail(BLOOM_E_INVALID, "null top-level weight pointer");
    if (!aligned16(w->word_emb) || !aligned16(w->emb_ln_g) || !aligned16(w->emb_ln_b) ||
        !aligned16(w->lnf_g) || !aligned16(w->lnf_b))
        return fail(BLOOM_E_INVALID, "top-level weights must be 16-byte aligned");
    const int h = cfg->hidden, F = cfg->ffn, i8 = cfg->weight_dtype == BLOOM_WEIGHT_INT8;
    for (int l = 0; l < cfg->n_layer; ++l) {
        const bloom_layer_weights &L = w->layers[l];
        if (!L.ln1_g || !L.ln1_b || !L.ln2_g || !L.ln2_b)
            return fail(BLOOM_E_INVALID, "layer %d: null LayerNorm pointer", l);
        if (!aligned16(L.ln1_g) || !aligned16(L.ln1_b) || !aligned16(L.ln2_g) || !aligned16(L.ln2_b))
            return fail(BLOOM_E_INVALID, "layer %d: LayerNorm params not 16-byte aligned", l);
        if ((st = check_linear(L.qkv, i8, 3 * h, h, "qkv", l))) return st;
        if ((st = check_linear(L.o, i8, h, h, "o", l))) return st;
        if ((st = check_linear(L.up, i8, F, h, "up", l))) return st;
        if ((st = check_linear(L.down, i8, h, F, "down", l))) return st;
    }
    bloom_model *m = new bloom_model();
    m->cfg = *cfg;
    m->word_emb = w->word_emb;
    m->emb_ln_g = w->emb_ln_g;
    m->emb_ln_b = w->emb_ln_b;
    m->lnf_g = w->lnf_g;
    m->lnf_b = w->lnf_b;
    m->layers.assign(w->layers, w->layers + cfg->n_layer);
    m->d = h / cfg->n_head;
    cudaError_t e = cudaGetDevice(&m->dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&m->num_sms, cudaDevAttrMultiProcessorCount, m->dev);
    if (e == cudaSuccess && (m->d == 64 || m->d == 128)) {
        m->attn_resident = attn_decode_resident_ctas(m->d, m->num_sms);
        m->attn_resident_wide = attn_decode_resident_ctas(m->d, m->num_sms, 1);
    }
    if (e != cudaSuccess) {
        delete m;
        return fail(BLOOM_E_CUDA, "no CUDA device: %s", cudaGetErrorString(e));
    }
    // workspace carve-up
    const size_t MT = (size_t)cfg->max_tokens, MB = (size_t)cfg->max_batch;
    const size_t n = (size_t)cfg->n_head, d = (size_t)m->d;
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off = align256(off + bytes); return o; };
    const size_t o_x = take(MT * h * 4), o_a = take(MT * h * 2), o_q = take(MT * h * 2),
                 o_o = take(MT * h * 2), o_u = take(MT * F * 2), o_xl = take(MB * h * 2),
                 o_sl = take(n * 4), o_best = take(MB * 8), o_ht = take(4),
                 o_ap = take(MB * n * kMaxSplits * (d + 2) * 4), o_at = take(MB * n * 4),
                 o_err = take(4), o_last = take(MB * 4), o_tok = take(MB * 4),
                 o_gen = take((size_t)cfg->max_seq * MB * 4), o_ptok = take(MT * 4),
                 o_pmask = take(MT), o_rowmap = take(MB * 4);
    m->ws_bytes = off;
    e = inject_failure("workspace") ? cudaErrorMemoryAllocation : cudaMalloc(&m->ws, m->ws_bytes);
    if (e != cudaSuccess) {
        delete m;
        cudaGetLastError();
        return fail(BLOOM_E_OOM, "workspace of %zu bytes: %s", off, cudaGetErrorString(e));
    }
    char *base = (char *)m->ws;
    m->x = (float *)(base + o_x);
    m->a = (uint16_t *)(base + o_a);
    m->q = (uint16_t *)(base + o_q);
    m->o = (uint16_t *)(base + o_o);
    m->u = (uint16_t *)(base + o_u);
    m->xl = (uint16_t *)(base + o_xl);
    m->slopes = (float *)(base + o_sl);
    m->best = (unsigned long long *)(base + o_best);
    m->head_ticket = (int *)(base + o_ht);
    m->attn_part = (float *)(base + o_ap);
    m->attn_ticket = (int *)(base + o_at);
    m->err = (int *)(base + o_err);
    m->last = (int *)(base + o_last);
    m->tok = (int32_t *)(base + o_tok);
    m->gen = (int32_t *)(base + o_gen);
    m->ptok = (int32_t *)(base + o_ptok);
    m->pmask = (uint8_t *)(base + o_pmask);
    m->rowmap = (int *)(base + o_rowmap);
    // ALiBi slopes, once: largest power of two p <= n heads gets 2^(-8i/p),
    // i = 1..p; the remaining heads take 2^(-8i/(2p)) for odd i = 1, 3, ...
    std::vector<float> sl(n);
    int p2 = 1;
    while (p2 * 2 <= (int)n) p2 *= 2;
    for (int i = 1; i <= p2; ++i) sl[i - 1] = (float)pow(2.0, -8.0 * i / p2);
    for (int j = 0; j < (int)n - p2; ++j) sl[p2 + j] = (float)pow(2.0, -8.0 * (2 * j + 1) / (2.0 * p2));
    bloom_status st2 = BLOOM_OK;
    // BLOOM_POISON_WORKSPACE (a debug aid for tests): every byte of the workspace
    // 0xff (NaN in bf16 and float32, -1 in int32) except the tickets, the argmax
    // scratch and the flag word, which rest at zero; a kernel that read any
    // activation before writing it would then show NaN or wrong tokens
    const bool poison = getenv("BLOOM_POISON_WORKSPACE") != nullptr;
    auto init_ws = [&]() -> bool {
        if (!poison) return cudaMemset(m->ws, 0, m->ws_bytes) == cudaSuccess;
        return cudaMemset(m->ws, 0xff, m->ws_bytes) == cudaSuccess &&
               cudaMemset(base + o_best, 0, MB * 8) == cudaSuccess &&
               cudaMemset(base + o_ht, 0, 4) == cudaSuccess &&
               cudaMemset(base + o_at, 0, MB * n * 4) == cudaSuccess &&
               cudaMemset(base + o_err, 0, 4) == cudaSuccess;
    };
    if (!init_ws() ||
        cudaMemcpy(m->slopes, sl.data(), n * 4, cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaStreamCreateWithFlags(&m->cap, cudaStreamNonBlocking) != cudaSuccess ||
        linear_prepare() != cudaSuccess) {
        st2 = fail(BLOOM_E_CUDA, "workspace init: %s", cudaGetErrorString(cudaGetLastError()));
    }
    // the LM head of decode steps on the tensor cores
    if (!st2 && !(cfg->flags & BLOOM_FLAG_NO_TC_GEMM)) {
        bool ok = gemm_map_bytes() == sizeof(TcMap) &&
                  gemm_make_map(m->head_wmap.b, w->word_emb, cfg->vocab, h, gemv_tc_box_rows_w());
        const int ntmax = gemv_tc_nt(cfg->max_batch);
        for (int ci = 0; ok && ci < kTcNtClasses && (16 << ci) <= ntmax; ++ci)
            ok = gemm_make_map(m->head_xmaps[ci].b, m->xl, cfg->max_batch, h, 16 << ci);
        if (!ok)
            st2 = fail(BLOOM_E_CUDA, "TMA descriptors for the LM head could not be encoded");
        else if (gemv_tc_prepare() != cudaSuccess)
            st2 = fail(BLOOM_E_CUDA, "LM head setup: %s", cudaGetErrorString(cudaGetLastError()));
        else
            m->tcd = true;
    }
    if (!st2 && m->tcd) {
        const int F = cfg->ffn;
        const int ntmax = gemv_tc_nt(cfg->max_batch);
        bool ok = true;
        m->dwmaps.resize((size_t)cfg->n_layer * TC_PER_LAYER);
        const int bw = gemv_tc_box_rows_w();
        for (int l = 0; ok && l < cfg->n_layer; ++l) {
            const bloom_layer_weights &L = w->layers[l];
            TcMap *wm = &m->dwmaps[(size_t)l * TC_PER_LAYER];
            auto mk = i8 ? gemm_make_map_u8 : gemm_make_map;
            ok = mk(wm[TC_QKV].b, L.qkv.w, 3 * h, h, bw) && mk(wm[TC_O].b, L.o.w, h, h, bw) &&
                 mk(wm[TC_UP].b, L.up.w, F, h, bw) && mk(wm[TC_DOWN].b, L.down.w, h, F, bw);
        }
        for (int ci = 0; ok && ci < kTcNtClasses && (16 << ci) <= ntmax; ++ci)
            ok = gemm_make_map(m->dxmaps[TC_X_A][ci].b, m->a, cfg->max_batch, h, 16 << ci) &&
                 gemm_make_map(m->dxmaps[TC_X_O][ci].b, m->o, cfg->max_batch, h, 16 << ci) &&
                 gemm_make_map(m->dxmaps[TC_X_U][ci].b, m->u, cfg->max_batch, F, 16 << ci);
        if (!ok)
            st2 = fail(BLOOM_E_CUDA, "TMA descriptors for the decode linears could not be encoded");
        else {
            m->tcb = true;
            const int widest = std::max(3 * h, F);
            m->tc_small = (widest + bw - 1) / bw <= 2 * m->num_sms;
        }
    }
    // TMA descriptors of every bf16 weight and of the activations the prefill GEMMs read
    if (!st2 && !i8 && !(cfg->flags & BLOOM_FLAG_NO_TC_GEMM) && cfg->max_tokens >= kTcMinM) {
        bool ok = gemm_map_bytes() == sizeof(TcMap);
        m->wmaps.resize((size_t)cfg->n_layer * TC_PER_LAYER);
        const int bw = gemm_box_rows_w(), bx = gemm_box_rows_x();
        for (int l = 0; ok && l < cfg->n_layer; ++l) {
            const bloom_layer_weights &L = w->layers[l];
            TcMap *wm = &m->wmaps[(size_t)l * TC_PER_LAYER];
            ok = gemm_make_map(wm[TC_QKV].b, L.qkv.w, 3 * h, h, bw) &&
                 gemm_make_map(wm[TC_O].b, L.o.w, h, h, bw) &&
                 gemm_make_map(wm[TC_UP].b, L.up.w, F, h, bw) &&
                 gemm_make_map(wm[TC_DOWN].b, L.down.w, h, F, bw);
        }
        ok = ok && gemm_make_map(m->xmaps[TC_X_A].b, m->a, (long long)MT, h, bx) &&
             gemm_make_map(m->xmaps[TC_X_O].b, m->o, (long long)MT, h, bx) &&
             gemm_make_map(m->xmaps[TC_X_U].b, m->u, (long long)MT, F, bx);
        if (!ok)
            st2 = fail(BLOOM_E_CUDA, "TMA descriptors for the prefill GEMM could not be encoded");
        else if (gemm_prepare() != cudaSuccess)
            st2 = fail(BLOOM_E_CUDA, "prefill GEMM setup: %s", cudaGetErrorString(cudaGetLastError()));
        else
            m->tc = true;
    }
    if (st2) {
        bloom_destroy(m);
        return st2;
    }
    *out = m;
    return BLOOM_OK;
}

static bloom_status check_kv(const bloom_model *m, const bloom_kv *kv) {
    if (!m) return fail(BLOOM_E_INVALID, "null model");
    if (!kv || !kv->buf) return fail(BLOOM_E_INVALID, "null kv");
    if (kv->batch < 1 || kv->batch > m->cfg.max_batch)
        return fail(BLOOM_E_CAPACITY, "kv batch %d above max_batch %d", kv->batch, m->cfg.max_batch);
    if (kv->max_seq < 1) return fail(BLOOM_E_INVALID, "kv max_seq %d", kv->max_seq);
    if (kv->offload_from < 0 || kv->offload_from > m->cfg.n_layer ||
        (kv->offload_from < m->cfg.n_layer && !kv->host_buf))
        return fail(BLOOM_E_INVALID, "kv offload_from %d / host buffer", kv->offload_from);
    if (kv->bytes < kv_layout(m->cfg, kv->batch, kv->max_seq, kv->offload_from).total)
        return fail(BLOOM_E_INVALID, "kv buffer too small");
    if (kv->offload_from < m->cfg.n_layer &&
        kv->host_bytes < kv_host_layout(m->cfg, kv->batch, kv->max_seq, kv->offload_from).total)
        return fail(BLOOM_E_INVALID, "kv host buffer too small");
    return BLOOM_OK;
}

static bool ranges_overlap(const void *a, size_t an, const void *b, size_t bn) {
    if (!a || !b) return false;
    const char *a0 = (const char *)a, *b0 = (const char *)b;
    return a0 < b0 + bn && b0 < a0 + an;
}

static bloom_status kv_init_impl(bloom_model *m, bloom_kv *kv, void *buf, size_t bytes,
                                 void *host_buf, size_t host_bytes, int32_t batch,
                                 int32_t max_seq, int32_t offload_from, void *stream) {
    if (!m || !kv || !buf) return fail(BLOOM_E_INVALID, "null argument");
    if (((uintptr_t)buf & 255u) != 0) return fail(BLOOM_E_INVALID, "kv buffer not 256-byte aligned");
    if (batch < 1 || batch > m->cfg.max_batch)
        return fail(BLOOM_E_CAPACITY, "batch %d outside 1..max_batch %d", batch, m->cfg.max_batch);
    if (max_seq < 1 || max_seq > m->cfg.max_seq)
        return fail(BLOOM_E_CAPACITY, "max_seq %d outside 1..%d", max_seq, m->cfg.max_seq);
    if (offload_from < 0 || offload_from > m->cfg.n_layer)
        return fail(BLOOM_E_INVALID, "offload_from %d outside 0..%d", offload_from, m->cfg.n_layer);
    const KvLayout L = kv_layout(m->cfg, batch, max_seq, offload_from);
    if (bytes < L.total) return fail(BLOOM_E_INVALID, "kv buffer %zu < %zu bytes", bytes, L.total);
    if (offload_from < m->cfg.n_layer) {
        if (!host_buf) return fail(BLOOM_E_INVALID, "null host buffer");
        if (((uintptr_t)host_buf & 255u) != 0)
            return fail(BLOOM_E_INVALID, "kv host buffer not 256-byte aligned");
        const KvHostLayout H = kv_host_layout(m->cfg, batch, max_seq, offload_from);
        if (host_bytes < H.total)
            return fail(BLOOM_E_INVALID, "kv host buffer %zu < %zu bytes", host_bytes, H.total);
        // the kernels dereference it directly: page-locked host memory that the
        // device addresses with the same pointer
        cudaPointerAttributes pa;
        if (cudaPointerGetAttributes(&pa, host_buf) != cudaSuccess || pa.type != cudaMemoryTypeHost ||
            pa.devicePointer != host_buf) {
            cudaGetLastError();
            return fail(BLOOM_E_INVALID, "kv host buffer is not page-locked host memory the "
                        "device maps at the same address");
        }
    } else {
        host_buf = nullptr;
        host_bytes = 0;
    }
    cudaStream_t s = (cudaStream_t)stream;
    // graphs captured on a cache that overlaps these buffers describe a layout
    // that no longer exists (the caller re-bound or re-allocated the memory)
    for (size_t i = 0; i < m->graphs.size();) {
        const GraphEntry &g = m->graphs[i];
        if (ranges_overlap(g.kvbuf, g.kvbytes, buf, bytes) ||
            ranges_overlap(g.hostbuf, g.hostbytes, host_buf, host_bytes) ||
            ranges_overlap(g.hostbuf, g.hostbytes, buf, bytes) ||
            ranges_overlap(g.kvbuf, g.kvbytes, host_buf, host_bytes)) {
            cudaGraphExecDestroy(g.exec);
            m->graphs.erase(m->graphs.begin() + (long)i);
        } else {
            ++i;
        }
    }
    CK(cudaMemsetAsync(buf, 0, L.pos, s));
    CK(cudaMemsetAsync((char *)buf + L.pos, 0xff, L.k - L.pos, s));
    kv->buf = buf;
    kv->bytes = bytes;
    kv->batch = batch;
    kv->max_seq = max_seq;
    kv->len = 0;
    for (int b = 0; b < BLOOM_MAX_BATCH; ++b) {
        kv->row_len[b] = 0;
        kv->row_active[b] = 0;
    }
    kv->host_buf = host_buf;
    kv->host_bytes = host_bytes;
    kv->offload_from = offload_from;
    return BLOOM_OK;
}

extern "C" bloom_status bloom_kv_init(bloom_model *m, bloom_kv *kv, void *buf, size_t bytes,
                                      int32_t batch, int32_t max_seq, void *stream) {
    return kv_init_impl(m, kv, buf, bytes, nullptr, 0, batch, max_seq, m ? m->cfg.n_layer : 0,
                        stream);
}

extern "C" bloom_status bloom_kv_init_offload(bloom_model *m, bloom_kv *kv, void *buf, size_t bytes,
                                              void *host_buf, size_t host_bytes, int32_t batch,
                                              int32_t max_seq, int32_t offload_from, void *stream) {
    return kv_init_impl(m, kv, buf, bytes, host_buf, host_bytes, batch, max_seq, offload_from,
                        stream);
}

// Host mirror of the cache's per-row state: kv->len = the longest active row.
static void kv_mirror_len(bloom_kv *kv) {
    int mx = 0;
    for (int b = 0; b < kv->batch; ++b)
        if (kv->row_active[b] && kv->row_len[b] > mx) mx = kv->row_len[b];
    kv->len = mx;
}
static void kv_mirror_prompt(bloom_kv *kv, const int32_t *rows, int n, int T) {
    for (int i = 0; i < n; ++i) {
        const int r = rows ? rows[i] : i;
        kv->row_len[r] = T;
        kv->row_active[r] = 1;
    }
    kv_mirror_len(kv);
}
// A decode step needs an active row, and room for one more slot in every active row.
static bloom_status kv_check_step(const bloom_kv *kv) {
    int active = 0;
    for (int b = 0; b < kv->batch; ++b) {
        if (!kv->row_active[b]) continue;
        ++active;
        if (kv->row_len[b] >= kv->max_seq)
            return fail(BLOOM_E_CAPACITY, "cache row %d full (%d slots)", b, kv->max_seq);
    }
    if (!active) return fail(BLOOM_E_INVALID, "decode with no active sequence (prefill or admit first)");
    return BLOOM_OK;
}
static void kv_mirror_step(bloom_kv *kv) {
    for (int b = 0; b < kv->batch; ++b)
        if (kv->row_active[b]) ++kv->row_len[b];
    kv_mirror_len(kv);
}

// pointers into a kv buffer
struct KvPtrs {
    int *len, *active, *next_pos, *pos;
    uint16_t *k, *v;              // layers [0, offload_from)
    uint16_t *k_host, *v_host;    // layers [offload_from, n_layer), in host memory
    int offload_from;
    size_t layer_elems;
    uint16_t *k_layer(int l) const {
        return l < offload_from ? k + layer_elems * l : k_host + layer_elems * (l - offload_from);
    }
    uint16_t *v_layer(int l) const {
        return l < offload_from ? v + layer_elems * l : v_host + layer_elems * (l - offload_from);
    }
};
static KvPtrs kv_ptrs(const bloom_model *m, const bloom_kv *kv) {
    const KvLayout L = kv_layout(m->cfg, kv->batch, kv->max_seq, kv->offload_from);
    char *b = (char *)kv->buf;
    KvPtrs p;
    p.len = (int *)(b + L.len);
    p.active = (int *)(b + L.active);
    p.next_pos = (int *)(b + L.next_pos);
    p.pos = (int *)(b + L.pos);
    p.k = (uint16_t *)(b + L.k);
    p.v = (uint16_t *)(b + L.v);
    p.offload_from = kv->offload_from;
    p.k_host = p.v_host = nullptr;
    if (kv->offload_from < m->cfg.n_layer) {
        const KvHostLayout H = kv_host_layout(m->cfg, kv->batch, kv->max_seq, kv->offload_from);
        char *h = (char *)kv->host_buf;
        p.k_host = (uint16_t *)(h + H.k);
        p.v_host = (uint16_t *)(h + H.v);
    }
    p.layer_elems = L.layer / 2;
    return p;
}

static LinearArgs lin_args(const bloom_linear &l, int int8, const uint16_t *x, int M, int N,
                           int K, int epi) {
    LinearArgs a;
    a.w = l.w;
    a.scale = (const uint16_t *)l.scale;
    a.bias = (const uint16_t *)l.bias;
    a.x = x;
    a.M = M;
    a.N = N;
    a.K = K;
    a.int8 = int8;
    a.epi = epi;
    return a;
}

// Whether the LayerNorm feeding `a` would be fused into the weight-streaming
// kernel (decode, 1-2 rows), which then beats a tensor-core kernel plus a
// LayerNorm launch: the LM head (one pass over 2 GB, where the streaming
// kernel reaches the copy peak), the int8 QKV and up projections, and the bf16
// ones of stacks too wide for tc_small.  Other bf16 block linears run on the
// tensor-core kernel at every batch size (see use_tc_linear).
static bool prefers_ln_fusion(const bloom_model *m, const LinearArgs &a) {
    return !(m->cfg.flags & BLOOM_FLAG_NO_LN_FUSION) && linear_can_fuse_ln(a) &&
           (a.epi == EPI_ARGMAX ||
            ((a.int8 || !m->tc_small) && (a.epi == EPI_QKV || a.epi == EPI_GELU)));
}

// The LM head + argmax on the tensor cores (one pass over the embedding; no K split).
static bool use_tc_head(const bloom_model *m, const LinearArgs &a) {
    return m->tcd && a.epi == EPI_ARGMAX && a.M >= 3 && a.M <= m->cfg.max_batch && !a.ln_x &&
           !prefers_ln_fusion(m, a);
}

// Index of the activation map whose box covers nt token columns (16 << index).
static int nt_class(int nt) {
    int ci = 0;
    while ((16 << ci) < nt) ++ci;
    return ci;
}

// ----------------------------------------------------------------- launch profile
// bloom_decode_profile records a CUDA event after every launch of one decode
// step; each launch site calls prof_mark with its operation and kernel.
struct LaunchProfile {
    std::vector<cudaEvent_t> ev;
    std::vector<int32_t> code;
    cudaError_t err = cudaSuccess;
};
static thread_local LaunchProfile *g_prof = nullptr;

static void prof_mark(cudaStream_t s, int op, int kernel) {
    if (!g_prof) return;
    cudaEvent_t e = nullptr;
    cudaError_t r = cudaEventCreate(&e);
    if (r == cudaSuccess) r = cudaEventRecord(e, s);
    if (r != cudaSuccess) {
        if (e) cudaEventDestroy(e);
        g_prof->err = r;
        return;
    }
    g_prof->ev.push_back(e);
    g_prof->code.push_back(op | (kernel << 8));
}

static GemvTcArgs tc_args(const bloom_model *m, const LinearArgs &a) {
    GemvTcArgs g;
    g.a = a;
    g.a.wait_ns = (unsigned long long)m->cfg.wait_us * 1000ull;
    if (!g.a.err) g.a.err = m->err;   // an expired wait is reported by bloom_check_device
    g.splits = gemv_tc_splits(a.N, a.K, a.M, a.epi, m->num_sms, a.int8);
    return g;
}

static cudaError_t run_tc_head(bloom_model *m, const LinearArgs &a, cudaStream_t s) {
    const int nt = gemv_tc_nt(a.M);
    const int ci = nt_class(nt);
    return launch_gemv_tc(m->head_wmap.b, m->head_xmaps[ci].b, tc_args(m, a), nt, s);
}

// A decode block linear on the tensor-core decode kernel.  Measured on GB300
// (7b1, 30 layers, whole decode step): bf16 at one / two sequences 3.11 / 3.11
// ms with every block linear there (LayerNorm as its own launch) vs 3.18 / 3.64
// ms on the weight-streaming kernel with the LayerNorm fused into QKV and up,
// and 4.13 / 4.39 ms with only dense and down moved: the streaming kernel's
// CTAs start early beside a predecessor that takes no shared memory, which a
// tensor-core kernel (two 108 KB CTAs per SM) in between prevents, so the two
// kernels do not mix within a layer at one or two sequences.  That holds where
// the widest block matrix is one wave of unsplit tensor-core CTAs (tc_small);
// the 176B-layer stack (448 tiles for up) at one sequence took 12.99 ms on the
// tensor-core kernel vs 12.14 streaming, and stays there below
// kTcSmallBatchMinM sequences, as int8 does (it widens the codes in registers
// at the copy rate there; the tensor-core form converts through TMEM).
constexpr int kTcSmallBatchMinM = 3;
static bool use_tc_linear(const bloom_model *m, const LinearArgs &a) {
    const int min_m = (a.int8 || !m->tc_small) ? kTcSmallBatchMinM : 1;
    return m->tcb && a.T == 0 && !a.ln_x && a.M >= min_m && a.M <= m->cfg.max_batch &&
           (!a.int8 || a.M <= kGvInt8MaxNt) && !prefers_ln_fusion(m, a);
}

// A linear layer of decoder layer l: the tensor-core GEMM for prefill batches of
// kTcMinM tokens or more, the tensor-core decode kernel where use_tc_linear
// says so, else the weight-streaming kernel.
static int wmap_op(int wmap) {
    return wmap == TC_QKV ? BLOOM_OP_QKV : wmap == TC_O ? BLOOM_OP_DENSE
                                         : wmap == TC_UP ? BLOOM_OP_UP : BLOOM_OP_DOWN;
}

static cudaError_t run_linear(bloom_model *m, const LinearArgs &a, int l, int wmap, int xmap,
                              cudaStream_t s) {
    cudaError_t e;
    int kernel;
    if (m->tc && a.T > 0 && a.M >= kTcMinM && !a.ln_x) {
        LinearArgs b = a;
        b.wait_ns = (unsigned long long)m->cfg.wait_us * 1000ull;
        if (!b.err) b.err = m->err;
        e = launch_gemm_tc(m->xmaps[xmap].b, m->wmaps[(size_t)l * TC_PER_LAYER + wmap].b, b, s);
        kernel = BLOOM_KERNEL_GEMM_TC;
    } else if (use_tc_linear(m, a)) {
        const int nt = gemv_tc_nt(a.M);
        const int ci = nt_class(nt);
        e = launch_gemv_tc(m->dwmaps[(size_t)l * TC_PER_LAYER + wmap].b, m->dxmaps[xmap][ci].b,
                           tc_args(m, a), nt, s);
        kernel = BLOOM_KERNEL_GEMV_TC;
    } else {
        e = launch_linear(a, m->num_sms, s);
        kernel = BLOOM_KERNEL_STREAM;
    }
    if (e == cudaSuccess) prof_mark(s, wmap_op(wmap), kernel);
    return e;
}

// Whether the LayerNorm feeding linear `a` runs inside it: allowed by the flags
// and the linear kernel, and `a` does not run on a tensor-core kernel (those
// read their activations from global memory through a TMA map).
static bool ln_fuses(const bloom_model *m, const LinearArgs &a) {
    return !(m->cfg.flags & BLOOM_FLAG_NO_LN_FUSION) && linear_can_fuse_ln(a) &&
           !use_tc_head(m, a) && !use_tc_linear(m, a);
}

// The LayerNorm feeding a linear layer: fused into the linear kernel's prologue
// when ln_fuses says so, else one LayerNorm launch writing the bf16 activations
// the linear layer reads.
static cudaError_t fused_ln(bloom_model *m, LinearArgs &a, const float *x, const void *g,
                            const void *b, cudaStream_t s) {
    if (ln_fuses(m, a)) {
        a.ln_x = x;
        a.ln_g = (const uint16_t *)g;
        a.ln_b = (const uint16_t *)b;
        a.ln_eps = m->cfg.ln_eps;
        return cudaSuccess;
    }
    const cudaError_t e = launch_layernorm_f32(x, (const uint16_t *)g, (const uint16_t *)b, a.M,
                                               a.K, m->cfg.ln_eps, const_cast<uint16_t *>(a.x), 1,
                                               nullptr, s);
    if (e == cudaSuccess) prof_mark(s, BLOOM_OP_LAYERNORM, BLOOM_KERNEL_LAYERNORM);
    return e;
}

// One decoder layer over M tokens.  Decode: M = B sequences, slot *len.
// Prefill: M = B*T tokens, slots [0, T).
static cudaError_t enqueue_layer(bloom_model *m, const KvPtrs &kp, int B, int max_seq, int l,
                                 int M, int T, int splits, float *x, cudaStream_t s,
                                 const int *row_map = nullptr) {
    char rname[32];
    snprintf(rname, sizeof rname, "bloom layer %d", l);
    NvtxRange range(rname);
    const bloom_config &c = m->cfg;
    const bloom_layer_weights &L = m->layers[l];
    const int h = c.hidden, F = c.ffn, n = c.n_head, d = m->d;
    const int i8 = c.weight_dtype == BLOOM_WEIGHT_INT8;
    const float eps = c.ln_eps;
    cudaError_t e;
    LinearArgs q = lin_args(L.qkv, i8, m->a, M, 3 * h, h, EPI_QKV);
    q.q_out = m->q;
    q.k_cache = kp.k_layer(l);
    q.v_cache = kp.v_layer(l);
    q.len_ptr = kp.len;
    q.active = kp.active;
    q.T = T;
    q.row_map = row_map;
    q.n_head = n;
    q.head_dim = d;
    q.max_seq = max_seq;
    q.err = m->err;
    if ((e = fused_ln(m, q, x, L.ln1_g, L.ln1_b, s))) return e;
    if ((e = run_linear(m, q, l, TC_QKV, TC_X_A, s))) return e;
    if (T == 0) {
        AttnDecodeArgs at;
        at.q = m->q;
        at.k = q.k_cache;
        at.v = q.v_cache;
        at.pos = kp.pos;
        at.slopes = m->slopes;
        at.len_ptr = kp.len;
        at.active = kp.active;
        at.B = B;
        at.n = n;
        at.d = d;
        at.max_seq = max_seq;
        at.splits = splits;
        at.early = (g_capture && g_pdl) ? 1 : 0;
        at.resident_ctas = m->attn_resident;
        at.resident_wide = m->attn_resident_wide;
        at.bulk = l < kp.offload_from ? 1 : 0;   // the layer's K / V in device memory
        at.err = m->err;
        at.wait_ns = (unsigned long long)m->cfg.wait_us * 1000ull;
        at.scale = (float)(1.0 / sqrt((double)d));
        at.part = m->attn_part;
        at.ticket = m->attn_ticket;
        at.o = m->o;
        if ((e = launch_attn_decode(at, s))) return e;
        prof_mark(s, BLOOM_OP_ATTN, BLOOM_KERNEL_ATTN);
    } else {
        AttnPrefillArgs at;
        at.q = m->q;
        at.k = q.k_cache;
        at.v = q.v_cache;
        at.pos = kp.pos;
        at.row_map = row_map;
        at.slopes = m->slopes;
        at.B = B;
        at.T = T;
        at.n = n;
        at.d = d;
        at.max_seq = max_seq;
        at.scale = (float)(1.0 / sqrt((double)d));
        at.o = m->o;
        if ((e = launch_attn_prefill_tc(at, s))) return e;
        prof_mark(s, BLOOM_OP_ATTN, BLOOM_KERNEL_ATTN_PREFILL);
    }
    LinearArgs od = lin_args(L.o, i8, m->o, M, h, h, EPI_RESID32);
    od.out32 = x;
    od.T = T;
    if ((e = run_linear(m, od, l, TC_O, TC_X_O, s))) return e;
    LinearArgs up = lin_args(L.up, i8, m->a, M, F, h, EPI_GELU);
    up.out = m->u;
    up.T = T;
    if ((e = fused_ln(m, up, x, L.ln2_g, L.ln2_b, s))) return e;
    if ((e = run_linear(m, up, l, TC_UP, TC_X_A, s))) return e;
    LinearArgs dn = lin_args(L.down, i8, m->u, M, h, F, EPI_RESID32);
    dn.out32 = x;
    dn.T = T;
    (void)eps;
    return run_linear(m, dn, l, TC_DOWN, TC_X_U, s);
}

// ln_f + tied head + argmax on rows of `x` (row r at x[(r*stride + last[r]) * h]).
static cudaError_t enqueue_head(bloom_model *m, const float *x, int B, int stride,
                                const int *last, int32_t *out_tokens, float *logits,
                                int *len_inc, int *next_pos, cudaStream_t s,
                                const int *active = nullptr) {
    const bloom_config &c = m->cfg;
    LinearArgs a;
    a.w = m->word_emb;
    a.x = m->xl;
    a.M = B;
    a.N = c.vocab;
    a.K = c.hidden;
    a.epi = EPI_ARGMAX;
    a.logits = logits;
    a.best = m->best;
    a.ticket = m->head_ticket;
    a.out_tokens = out_tokens;
    a.len_inc = len_inc;
    a.next_pos = next_pos;
    a.active = active;
    cudaError_t e;
    if (stride == 1 && !last) {
        if ((e = fused_ln(m, a, x, m->lnf_g, m->lnf_b, s))) return e;
    } else if ((e = launch_layernorm_f32(x, (const uint16_t *)m->lnf_g, (const uint16_t *)m->lnf_b,
                                         B, c.hidden, c.ln_eps, m->xl, stride, last, s))) {
        return e;
    } else {
        prof_mark(s, BLOOM_OP_LAYERNORM, BLOOM_KERNEL_LAYERNORM);
    }
    const bool tc = use_tc_head(m, a);
    e = tc ? run_tc_head(m, a, s) : launch_linear(a, m->num_sms, s);
    if (e == cudaSuccess) prof_mark(s, BLOOM_OP_HEAD, tc ? BLOOM_KERNEL_GEMV_TC : BLOOM_KERNEL_STREAM);
    return e;
}

static cudaError_t enqueue_decode(bloom_model *m, const bloom_kv *kv, const int32_t *next,
                                  int32_t *out, float *logits, cudaStream_t s) {
    const bloom_config &c = m->cfg;
    const KvPtrs kp = kv_ptrs(m, kv);
    const int B = kv->batch;
    const int splits = attn_splits(m, B, kv->max_seq);
    cudaError_t e = launch_embed(next, B, (const uint16_t *)m->word_emb, c.vocab,
                                 (const uint16_t *)m->emb_ln_g, (const uint16_t *)m->emb_ln_b,
                                 c.hidden, c.ln_eps, m->x, kp.len, kp.active, kp.next_pos, kp.pos,
                                 kv->max_seq, m->err, s);
    if (e) return e;
    prof_mark(s, BLOOM_OP_EMBED, BLOOM_KERNEL_EMBED);
    for (int l = 0; l < c.n_layer; ++l)
        if ((e = enqueue_layer(m, kp, B, kv->max_seq, l, B, 0, splits, m->x, s))) return e;
    return enqueue_head(m, m->x, B, 1, nullptr, out, logits, kp.len, kp.next_pos, s, kp.active);
}

extern "C" int32_t bloom_decode_launches(const bloom_model *m, int32_t batch) {
    if (!m) return 0;
    // embedding; per layer LN1, QKV, attention, dense, LN2, up, down; ln_f, head --
    // less the LayerNorm launches that the linear kernels absorb (ln_fuses)
    const bloom_config &c = m->cfg;
    const int i8 = c.weight_dtype == BLOOM_WEIGHT_INT8;
    LinearArgs qkv = lin_args(bloom_linear{}, i8, m->a, batch, 3 * c.hidden, c.hidden, EPI_QKV);
    LinearArgs up = lin_args(bloom_linear{}, i8, m->a, batch, c.ffn, c.hidden, EPI_GELU);
    LinearArgs head = lin_args(bloom_linear{}, 0, m->xl, batch, c.vocab, c.hidden, EPI_ARGMAX);
    const int block_ln = (ln_fuses(m, qkv) ? 0 : 1) + (ln_fuses(m, up) ? 0 : 1);
    const int head_ln = ln_fuses(m, head) ? 0 : 1;
    return 1 + (5 + block_ln) * c.n_layer + 1 + head_ln;
}

extern "C" bloom_status bloom_kv_set_prompt(bloom_model *m, bloom_kv *kv, const uint8_t *mask,
                                            int32_t B, int32_t T, void *stream) {
    if (m) g_pdl = !(m->cfg.flags & BLOOM_FLAG_NO_PDL);
    bloom_status st = check_kv(m, kv);
    if (st) return st;
    if (!mask) return fail(BLOOM_E_INVALID, "null mask");
    if (B != kv->batch) return fail(BLOOM_E_CAPACITY, "B=%d but kv batch is %d", B, kv->batch);
    if (T < 1 || T > kv->max_seq) return fail(BLOOM_E_CAPACITY, "T=%d outside 1..%d", T, kv->max_seq);
    const KvPtrs kp = kv_ptrs(m, kv);
    CK(launch_prompt_setup(mask, B, T, nullptr, kp.pos, kv->max_seq, kp.next_pos, kp.len, kp.active,
                           m->last, m->err, (cudaStream_t)stream));
    kv_mirror_prompt(kv, nullptr, B, T);
    return BLOOM_OK;
}

// Prefill of n prompts (tokens / mask [n][T]) into cache rows rows_dev[i]
// (null: rows 0..n-1); the greedy token of each to out_tokens [n].
static bloom_status prefill_rows(bloom_model *m, bloom_kv *kv, const int32_t *tokens,
                                 const uint8_t *mask, int32_t n, int32_t T, const int *rows_dev,
                                 int32_t *out_tokens, float *out_logits, cudaStream_t s) {
    const bloom_config &c = m->cfg;
    const KvPtrs kp = kv_ptrs(m, kv);
    const int M = n * T;
    CK(launch_prompt_setup(mask, n, T, rows_dev, kp.pos, kv->max_seq, kp.next_pos, kp.len,
                           kp.active, m->last, m->err, s));
    CK(launch_embed(tokens, M, (const uint16_t *)m->word_emb, c.vocab, (const uint16_t *)m->emb_ln_g,
                    (const uint16_t *)m->emb_ln_b, c.hidden, c.ln_eps, m->x, nullptr, nullptr,
                    nullptr, nullptr, 0, m->err, s));
    for (int l = 0; l < c.n_layer; ++l)
        CK(enqueue_layer(m, kp, n, kv->max_seq, l, M, T, 1, m->x, s, rows_dev));
    CK(enqueue_head(m, m->x, n, T, m->last, out_tokens, out_logits, nullptr, nullptr, s));
    return BLOOM_OK;
}

extern "C" bloom_status bloom_prefill(bloom_model *m, bloom_kv *kv, const int32_t *tokens,
                                      const uint8_t *mask, int32_t B, int32_t T,
                                      int32_t *out_tokens, float *out_logits, void *stream) {
    NvtxRange range("bloom_prefill");
    if (m) g_pdl = !(m->cfg.flags & BLOOM_FLAG_NO_PDL);
    bloom_status st = check_kv(m, kv);
    if (st) return st;
    if (!tokens || !mask || !out_tokens) return fail(BLOOM_E_INVALID, "null tokens/mask/out_tokens");
    if (B != kv->batch) return fail(BLOOM_E_CAPACITY, "B=%d but kv batch is %d", B, kv->batch);
    if (T < 1 || T > kv->max_seq) return fail(BLOOM_E_CAPACITY, "T=%d outside 1..%d", T, kv->max_seq);
    if ((long long)B * T > m->cfg.max_tokens)
        return fail(BLOOM_E_CAPACITY, "B*T=%lld above max_tokens %d", (long long)B * T, m->cfg.max_tokens);
    if ((st = prefill_rows(m, kv, tokens, mask, B, T, nullptr, out_tokens, out_logits,
                           (cudaStream_t)stream)))
        return st;
    kv_mirror_prompt(kv, nullptr, B, T);
    return BLOOM_OK;
}

extern "C" bloom_status bloom_kv_admit(bloom_model *m, bloom_kv *kv, const int32_t *rows,
                                       int32_t n, const int32_t *tokens, const uint8_t *mask,
                                       int32_t T, int32_t *out_tokens, float *out_logits,
                                       void *stream) {
    NvtxRange range("bloom_kv_admit");
    if (m) g_pdl = !(m->cfg.flags & BLOOM_FLAG_NO_PDL);
    bloom_status st = check_kv(m, kv);
    if (st) return st;
    if (!rows || !tokens || !mask || !out_tokens) return fail(BLOOM_E_INVALID, "null argument");
    if (n < 1 || n > kv->batch) return fail(BLOOM_E_INVALID, "n=%d outside 1..%d", n, kv->batch);
    if (T < 1 || T > kv->max_seq) return fail(BLOOM_E_CAPACITY, "T=%d outside 1..%d", T, kv->max_seq);
    if ((long long)n * T > m->cfg.max_tokens)
        return fail(BLOOM_E_CAPACITY, "n*T=%lld above max_tokens %d", (long long)n * T, m->cfg.max_tokens);
    RowList rl;
    rl.n = n;
    for (int i = 0; i < n; ++i) {
        if (rows[i] < 0 || rows[i] >= kv->batch) return fail(BLOOM_E_INVALID, "row %d", rows[i]);
        for (int j = 0; j < i; ++j)
            if (rows[j] == rows[i]) return fail(BLOOM_E_INVALID, "row %d given twice", rows[i]);
        rl.rows[i] = rows[i];
    }
    cudaStream_t s = (cudaStream_t)stream;
    CK(launch_set_rows(rl, m->rowmap, s));
    if ((st = prefill_rows(m, kv, tokens, mask, n, T, m->rowmap, out_tokens, out_logits, s))) return st;
    kv_mirror_prompt(kv, rows, n, T);
    return BLOOM_OK;
}

extern "C" bloom_status bloom_kv_retire(bloom_model *m, bloom_kv *kv, const int32_t *rows,
                                        int32_t n, void *stream) {
    if (m) g_pdl = !(m->cfg.flags & BLOOM_FLAG_NO_PDL);
    bloom_status st = check_kv(m, kv);
    if (st) return st;
    if (!rows || n < 0 || n > kv->batch) return fail(BLOOM_E_INVALID, "rows / n=%d", n);
    RowList rl;
    rl.n = n;
    for (int i = 0; i < n; ++i) {
        if (rows[i] < 0 || rows[i] >= kv->batch) return fail(BLOOM_E_INVALID, "row %d", rows[i]);
        rl.rows[i] = rows[i];
    }
    CK(launch_set_active(rl, 0, kv_ptrs(m, kv).active, (cudaStream_t)stream));
    for (int i = 0; i < n; ++i) kv->row_active[rows[i]] = 0;
    kv_mirror_len(kv);
    return BLOOM_OK;
}

extern "C" bloom_status bloom_decode_step(bloom_model *m, bloom_kv *kv, const int32_t *next_tokens,
                                          int32_t *out_tokens, float *out_logits, void *stream) {
    NvtxRange range("bloom_decode_step");
    if (m) g_pdl = !(m->cfg.flags & BLOOM_FLAG_NO_PDL);
    bloom_status st = check_kv(m, kv);
    if (st) return st;
    if (!next_tokens || !out_tokens) return fail(BLOOM_E_INVALID, "null next_tokens/out_tokens");
    if ((st = kv_check_step(kv))) return st;
    cudaStream_t s = (cudaStream_t)stream;
    if (m->cfg.flags & BLOOM_FLAG_NO_GRAPH) {
        CK(enqueue_decode(m, kv, next_tokens, out_tokens, out_logits, s));
    } else {
        cudaGraphExec_t exec = nullptr;
        for (auto &g : m->graphs)
            if (g.kvbuf == kv->buf && g.kvbytes == kv->bytes && g.hostbuf == kv->host_buf &&
                g.hostbytes == kv->host_bytes && g.offload_from == kv->offload_from &&
                g.B == kv->batch && g.max_seq == kv->max_seq && g.next == next_tokens &&
                g.out == out_tokens && g.logits == out_logits) {
                exec = g.exec;
                break;
            }
        if (!exec) {
            cudaGraph_t graph = nullptr;
            CK(cudaStreamBeginCapture(m->cap, cudaStreamCaptureModeThreadLocal));
            g_capture = true;
            cudaError_t e = enqueue_decode(m, kv, next_tokens, out_tokens, out_logits, m->cap);
            g_capture = false;
            cudaError_t e2 = cudaStreamEndCapture(m->cap, &graph);
            if (e != cudaSuccess || e2 != cudaSuccess) {
                if (graph) cudaGraphDestroy(graph);
                return fail(BLOOM_E_CUDA, "decode capture: %s / %s", cudaGetErrorString(e),
                            cudaGetErrorString(e2));
            }
            e = cudaGraphInstantiate(&exec, graph, 0);
            cudaGraphDestroy(graph);
            if (e != cudaSuccess) return fail(BLOOM_E_CUDA, "graph instantiate: %s", cudaGetErrorString(e));
            if (m->graphs.size() >= 16) {
                cudaGraphExecDestroy(m->graphs.front().exec);
                m->graphs.erase(m->graphs.begin());
            }
            m->graphs.push_back({kv->buf, kv->bytes, kv->host_buf, kv->host_bytes,
                                 kv->offload_from, kv->batch, kv->max_seq, next_tokens,
                                 out_tokens, out_logits, exec});
        }
        CK(cudaGraphLaunch(exec, s));
    }
    kv_mirror_step(kv);
    return BLOOM_OK;
}

extern "C" bloom_status bloom_decode_profile(bloom_model *m, bloom_kv *kv,
                                             const int32_t *next_tokens, int32_t *out_tokens,
                                             int32_t *codes, float *ms, int32_t cap, int32_t *n,
                                             void *stream) {
    bloom_status st = check_kv(m, kv);
    if (st) return st;
    if (!next_tokens || !out_tokens || !codes || !ms || !n || cap < 1)
        return fail(BLOOM_E_INVALID, "null or empty argument");
    if ((st = kv_check_step(kv))) return st;
    *n = 0;
    cudaStream_t s = (cudaStream_t)stream;
    g_pdl = false;   // each launch starts after the previous one has finished
    LaunchProfile prof;
    cudaEvent_t start = nullptr;
    CK(cudaEventCreate(&start));
    cudaError_t e = cudaEventRecord(start, s);
    if (e == cudaSuccess) {
        g_prof = &prof;
        e = enqueue_decode(m, kv, next_tokens, out_tokens, nullptr, s);
        g_prof = nullptr;
    }
    if (e == cudaSuccess) e = prof.err;
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    cudaEvent_t prev = start;
    for (size_t i = 0; i < prof.ev.size(); ++i) {
        float t = 0.f;
        if (e == cudaSuccess) e = cudaEventElapsedTime(&t, prev, prof.ev[i]);
        if ((int32_t)i < cap) {
            codes[i] = prof.code[i];
            ms[i] = t;
        }
        prev = prof.ev[i];
    }
    for (cudaEvent_t ev : prof.ev) cudaEventDestroy(ev);
    cudaEventDestroy(start);
    g_pdl = !(m->cfg.flags & BLOOM_FLAG_NO_PDL);
    CK(e);
    *n = (int32_t)std::min<size_t>(prof.ev.size(), (size_t)cap);
    kv_mirror_step(kv);
    return BLOOM_OK;
}

extern "C" bloom_status bloom_check_device(bloom_model *m, void *stream) {
    if (!m) return fail(BLOOM_E_INVALID, "null model");
    cudaStream_t s = (cudaStream_t)stream;
    int flag = 0;
    CK(cudaMemcpyAsync(&flag, m->err, 4, cudaMemcpyDeviceToHost, s));
    CK(cudaMemsetAsync(m->err, 0, 4, s));
    CK(cudaStreamSynchronize(s));
    if (flag)
        return fail(BLOOM_E_DEVICE_FLAG, "device flag 0x%x (1: token id out of range, 2: cache "
                    "slot out of range, 4: prompt row without a token, 8: a bounded device wait "
                    "expired)", flag);
    return BLOOM_OK;
}

extern "C" bloom_status bloom_generate(bloom_model *m, bloom_kv *kv, const int32_t *tokens_host,
                                       const uint8_t *mask_host, int32_t B, int32_t T,
                                       int32_t n_new, int32_t *out_host, void *stream) {
    NvtxRange range("bloom_generate");
    bloom_status st = check_kv(m, kv);
    if (st) return st;
    if (!tokens_host || !mask_host || !out_host) return fail(BLOOM_E_INVALID, "null host buffer");
    if (n_new < 1) return fail(BLOOM_E_INVALID, "n_new %d", n_new);
    if ((long long)T + n_new - 1 > kv->max_seq)
        return fail(BLOOM_E_CAPACITY, "T + n_new - 1 = %d above kv max_seq %d", T + n_new - 1, kv->max_seq);
    if ((long long)B * T > m->cfg.max_tokens)
        return fail(BLOOM_E_CAPACITY, "B*T above max_tokens");
    if (n_new > m->cfg.max_seq) return fail(BLOOM_E_CAPACITY, "n_new above max_seq");
    cudaStream_t s = (cudaStream_t)stream;
    CK(cudaMemcpyAsync(m->ptok, tokens_host, (size_t)B * T * 4, cudaMemcpyHostToDevice, s));
    CK(cudaMemcpyAsync(m->pmask, mask_host, (size_t)B * T, cudaMemcpyHostToDevice, s));
    if ((st = bloom_prefill(m, kv, m->ptok, m->pmask, B, T, m->tok, nullptr, stream))) return st;
    CK(cudaMemcpyAsync(m->gen, m->tok, (size_t)B * 4, cudaMemcpyDeviceToDevice, s));
    for (int i = 1; i < n_new; ++i) {
        if ((st = bloom_decode_step(m, kv, m->tok, m->tok, nullptr, stream))) return st;
        CK(cudaMemcpyAsync(m->gen + (size_t)i * B, m->tok, (size_t)B * 4, cudaMemcpyDeviceToDevice, s));
    }
    CK(cudaMemcpyAsync(out_host, m->gen, (size_t)n_new * B * 4, cudaMemcpyDeviceToHost, s));
    return bloom_check_device(m, stream);
}

// ----------------------------------------------------------------- layer-level
extern "C" bloom_status bloom_layer_decode(bloom_model *m, bloom_kv *kv, int32_t layer, void *x,
                                           void *stream) {
    if (m) g_pdl = !(m->cfg.flags & BLOOM_FLAG_NO_PDL);
    bloom_status st = check_kv(m, kv);
    if (st) return st;
    if (!x) return fail(BLOOM_E_INVALID, "null x");
    if (layer < 0 || layer >= m->cfg.n_layer) return fail(BLOOM_E_INVALID, "layer %d", layer);
    if ((st = kv_check_step(kv))) return st;
    cudaStream_t s = (cudaStream_t)stream;
    const KvPtrs kp = kv_ptrs(m, kv);
    CK(launch_slot_pos(kv->batch, kp.len, kp.active, kp.next_pos, kp.pos, kv->max_seq, m->err, s));
    CK(enqueue_layer(m, kp, kv->batch, kv->max_seq, layer, kv->batch, 0,
                     attn_splits(m, kv->batch, kv->max_seq), (float *)x, s));
    return BLOOM_OK;
}

extern "C" bloom_status bloom_layer_prefill(bloom_model *m, bloom_kv *kv, int32_t layer, void *x,
                                            int32_t B, int32_t T, void *stream) {
    if (m) g_pdl = !(m->cfg.flags & BLOOM_FLAG_NO_PDL);
    bloom_status st = check_kv(m, kv);
    if (st) return st;
    if (!x) return fail(BLOOM_E_INVALID, "null x");
    if (layer < 0 || layer >= m->cfg.n_layer) return fail(BLOOM_E_INVALID, "layer %d", layer);
    if (B != kv->batch || T < 1 || T > kv->max_seq || (long long)B * T > m->cfg.max_tokens)
        return fail(BLOOM_E_CAPACITY, "B=%d T=%d", B, T);
    const KvPtrs kp = kv_ptrs(m, kv);
    CK(enqueue_layer(m, kp, B, kv->max_seq, layer, B * T, T, 1, (float *)x, (cudaStream_t)stream));
    return BLOOM_OK;
}

extern "C" bloom_status bloom_head(bloom_model *m, const void *x, int32_t B, int32_t *out_tokens,
                                   float *out_logits, void *stream) {
    if (m) g_pdl = !(m->cfg.flags & BLOOM_FLAG_NO_PDL);
    if (!m || !x || !out_tokens) return fail(BLOOM_E_INVALID, "null argument");
    if (B < 1 || B > m->cfg.max_batch) return fail(BLOOM_E_CAPACITY, "B=%d", B);
    CK(enqueue_head(m, (const float *)x, B, 1, nullptr, out_tokens, out_logits, nullptr, nullptr,
                    (cudaStream_t)stream));
    return BLOOM_OK;
}

extern "C" bloom_status bloom_lm_head(bloom_model *m, const void *xn, int32_t B,
                                      int32_t *out_tokens, float *out_logits, void *stream) {
    if (m) g_pdl = !(m->cfg.flags & BLOOM_FLAG_NO_PDL);
    if (!m || !xn || !out_tokens) return fail(BLOOM_E_INVALID, "null argument");
    if (B < 1 || B > m->cfg.max_batch) return fail(BLOOM_E_CAPACITY, "B=%d", B);
    if (!aligned16(xn)) return fail(BLOOM_E_INVALID, "xn not 16-byte aligned");
    LinearArgs a;
    a.w = m->word_emb;
    a.x = (const uint16_t *)xn;
    a.M = B;
    a.N = m->cfg.vocab;
    a.K = m->cfg.hidden;
    a.epi = EPI_ARGMAX;
    a.logits = out_logits;
    a.best = m->best;
    a.ticket = m->head_ticket;
    a.out_tokens = out_tokens;
    if (use_tc_head(m, a)) {
        // the decode step's kernel for this batch: a TMA descriptor of the caller's rows
        const int nt = gemv_tc_nt(B);
        TcMap mx;
        if (!gemm_make_map(mx.b, xn, B, m->cfg.hidden, nt))
            return fail(BLOOM_E_UNSUPPORTED, "TMA descriptor of xn could not be encoded");
        CK(launch_gemv_tc(m->head_wmap.b, mx.b, tc_args(m, a), nt, (cudaStream_t)stream));
        return BLOOM_OK;
    }
    CK(launch_linear(a, m->num_sms, (cudaStream_t)stream));
    return BLOOM_OK;
}

extern "C" bloom_status bloom_embed(bloom_model *m, const int32_t *tokens, int32_t n, void *x,
                                    void *stream) {
    if (m) g_pdl = !(m->cfg.flags & BLOOM_FLAG_NO_PDL);
    if (!m || !tokens || !x) return fail(BLOOM_E_INVALID, "null argument");
    if (n < 1) return fail(BLOOM_E_INVALID, "n=%d", n);
    const bloom_config &c = m->cfg;
    CK(launch_embed(tokens, n, (const uint16_t *)m->word_emb, c.vocab, (const uint16_t *)m->emb_ln_g,
                    (const uint16_t *)m->emb_ln_b, c.hidden, c.ln_eps, (float *)x, nullptr,
                    nullptr, nullptr, nullptr, 0, m->err, (cudaStream_t)stream));
    return BLOOM_OK;
}

// ----------------------------------------------------------------- operators
static int device_sms() {
    static int sms = 0;
    if (!sms) {
        linear_prepare();
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (sms <= 0) sms = 1;
    }
    return sms;
}

int bloom::bloom_device_sms() { return device_sms(); }

extern "C" bloom_status bloom_op_layernorm(const void *x, const void *g, const void *b,
                                           int32_t rows, int32_t h, float eps, void *y,
                                           void *stream) {
    g_pdl = true;
    if (!x || !y) return fail(BLOOM_E_INVALID, "null x/y");
    if (rows < 0 || h < 8 || h % 8 || h > kMaxHidden) return fail(BLOOM_E_UNSUPPORTED, "h=%d", h);
    if (!aligned16(x) || !aligned16(y) || (g && !aligned16(g)) || (b && !aligned16(b)))
        return fail(BLOOM_E_INVALID, "pointers must be 16-byte aligned");
    CK(launch_layernorm((const uint16_t *)x, (const uint16_t *)g, (const uint16_t *)b, rows, h, eps,
                        (uint16_t *)y, 1, nullptr, (cudaStream_t)stream));
    return BLOOM_OK;
}

extern "C" bloom_status bloom_op_linear(const bloom_linear *lin, int32_t int8, const void *x,
                                        int32_t M, int32_t N, int32_t K, int32_t epilogue, void *y,
                                        void *stream) {
    g_pdl = true;
    if (!lin) return fail(BLOOM_E_INVALID, "null argument");
    bloom_status st = check_linear(*lin, int8, N, K, "op", -1);
    if (st) return st;
    if (M < 0 || N < 1) return fail(BLOOM_E_INVALID, "M=%d N=%d", M, N);
    if (epilogue < BLOOM_EPI_STORE || epilogue > BLOOM_EPI_RESID)
        return fail(BLOOM_E_INVALID, "epilogue %d", epilogue);
    if (M == 0) return BLOOM_OK;
    if (!x || !y) return fail(BLOOM_E_INVALID, "null argument");
    if (!aligned16(x)) return fail(BLOOM_E_INVALID, "x not 16-byte aligned");
    cudaStream_t s = (cudaStream_t)stream;
    LinearArgs a = lin_args(*lin, int8, (const uint16_t *)x, M, N, K, epilogue);
    a.out = (uint16_t *)y;
    CK(launch_linear(a, device_sms(), s));
    return BLOOM_OK;
}

extern "C" bloom_status bloom_op_gemm(const bloom_linear *lin, const void *x, int32_t M,
                                      int32_t N, int32_t K, int32_t epilogue, void *y,
                                      void *stream) {
    g_pdl = true;
    if (!lin) return fail(BLOOM_E_INVALID, "null argument");
    bloom_status st = check_linear(*lin, 0, N, K, "op", -1);
    if (st) return st;
    if (M < 0 || N < 1) return fail(BLOOM_E_INVALID, "M=%d N=%d", M, N);
    if (epilogue < BLOOM_EPI_STORE || epilogue > BLOOM_EPI_RESID)
        return fail(BLOOM_E_INVALID, "epilogue %d", epilogue);
    if (M == 0) return BLOOM_OK;
    if (!x || !y) return fail(BLOOM_E_INVALID, "null argument");
    if (!aligned16(x)) return fail(BLOOM_E_INVALID, "x not 16-byte aligned");
    device_sms();
    TcMap mx, mw;
    if (gemm_map_bytes() != sizeof(TcMap) ||
        !gemm_make_map(mx.b, x, M, K, gemm_box_rows_x()) ||
        !gemm_make_map(mw.b, lin->w, N, K, gemm_box_rows_w()))
        return fail(BLOOM_E_UNSUPPORTED, "TMA descriptors could not be encoded");
    LinearArgs a = lin_args(*lin, 0, (const uint16_t *)x, M, N, K, epilogue);
    a.out = (uint16_t *)y;
    CK(launch_gemm_tc(mx.b, mw.b, a, (cudaStream_t)stream));
    return BLOOM_OK;
}

extern "C" bloom_status bloom_op_linear_tc(const bloom_linear *lin, int32_t int8, const void *x,
                                           int32_t M, int32_t N, int32_t K, int32_t epilogue,
                                           void *y, void *stream) {
    g_pdl = true;
    if (!lin) return fail(BLOOM_E_INVALID, "null argument");
    bloom_status st = check_linear(*lin, int8, N, K, "op", -1);
    if (st) return st;
    if (M < 0 || N < 1) return fail(BLOOM_E_INVALID, "M=%d N=%d", M, N);
    if (M > (int8 ? kGvInt8MaxNt : kMaxBatch))
        return fail(BLOOM_E_CAPACITY, "M=%d above %d", M, int8 ? kGvInt8MaxNt : kMaxBatch);
    if (epilogue < BLOOM_EPI_STORE || epilogue > BLOOM_EPI_RESID)
        return fail(BLOOM_E_INVALID, "epilogue %d", epilogue);
    if (M == 0) return BLOOM_OK;
    if (!x || !y) return fail(BLOOM_E_INVALID, "null argument");
    if (!aligned16(x)) return fail(BLOOM_E_INVALID, "x not 16-byte aligned");
    const int sms = device_sms();
    const int nt = gemv_tc_nt(M);
    TcMap mx, mw;
    if (gemm_map_bytes() != sizeof(TcMap) || !gemm_make_map(mx.b, x, M, K, nt) ||
        !(int8 ? gemm_make_map_u8 : gemm_make_map)(mw.b, lin->w, N, K, gemv_tc_box_rows_w()))
        return fail(BLOOM_E_UNSUPPORTED, "TMA descriptors could not be encoded");
    CK(gemv_tc_prepare());
    cudaStream_t s = (cudaStream_t)stream;
    GemvTcArgs g;
    g.a = lin_args(*lin, int8, (const uint16_t *)x, M, N, K, epilogue);
    g.a.out = (uint16_t *)y;
    g.splits = gemv_tc_splits(N, K, M, epilogue, sms, int8);
    CK(launch_gemv_tc(mw.b, mx.b, g, nt, s));
    return BLOOM_OK;
}

extern "C" bloom_status bloom_op_attn_decode(const void *q, const void *k_cache,
                                             const void *v_cache, const int32_t *pos,
                                             const float *slopes, int32_t B, int32_t n_head,
                                             int32_t d, int32_t max_seq, int32_t len,
                                             int32_t splits, void *o, void *stream) {
    g_pdl = true;
    if (!q || !k_cache || !v_cache || !pos || !slopes || !o) return fail(BLOOM_E_INVALID, "null argument");
    if (d != 64 && d != 128) return fail(BLOOM_E_UNSUPPORTED, "d=%d", d);
    if (B < 1 || n_head < 1 || max_seq < 1 || len < 0 || len >= max_seq)
        return fail(BLOOM_E_INVALID, "B=%d n=%d max_seq=%d len=%d", B, n_head, max_seq, len);
    // q, K, V and o are read and written 16 bytes at a time (K / V also by bulk copies)
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o))
        return fail(BLOOM_E_INVALID, "q, k_cache, v_cache and o must be 16-byte aligned");
    if (splits <= 0) {
        int want = (2 * device_sms() + B * n_head - 1) / (B * n_head);
        int cap = (len + 1 + 31) / 32;
        splits = want < cap ? want : cap;
        if (splits < 1) splits = 1;
    }
    if (splits > kMaxSplits) splits = kMaxSplits;
    cudaStream_t s = (cudaStream_t)stream;
    AttnDecodeArgs a;
    a.q = (const uint16_t *)q;
    a.k = (const uint16_t *)k_cache;
    a.v = (const uint16_t *)v_cache;
    a.pos = pos;
    a.slopes = slopes;
    a.len_host = len;
    a.B = B;
    a.n = n_head;
    a.d = d;
    a.max_seq = max_seq;
    a.splits = splits;
    a.scale = (float)(1.0 / sqrt((double)d));
    a.resident_ctas = attn_decode_resident_ctas(d, device_sms());
    a.resident_wide = attn_decode_resident_ctas(d, device_sms(), 1);
    {   // bulk copies only from device memory
        cudaPointerAttributes pk{}, pv{};
        a.bulk = cudaPointerGetAttributes(&pk, k_cache) == cudaSuccess &&
                 cudaPointerGetAttributes(&pv, v_cache) == cudaSuccess &&
                 pk.type == cudaMemoryTypeDevice && pv.type == cudaMemoryTypeDevice;
        cudaGetLastError();
    }
    void *scratch = nullptr;
    const size_t part_bytes = align256((size_t)B * n_head * splits * (d + 2) * 4);
    const size_t bytes = part_bytes + (size_t)B * n_head * 4;
    CK(cudaMallocAsync(&scratch, bytes, s));
    cudaError_t e = cudaMemsetAsync(scratch, 0, bytes, s);
    a.part = (float *)scratch;
    a.ticket = (int *)((char *)scratch + part_bytes);
    a.o = (uint16_t *)o;
    if (e == cudaSuccess) e = launch_attn_decode(a, s);
    cudaError_t e2 = cudaFreeAsync(scratch, s);
    CK(e);
    CK(e2);
    return BLOOM_OK;
}

extern "C" bloom_status bloom_op_sample(const float *logits, int32_t B, int32_t V, int64_t ld,
                                        const float *temperature, const float *top_p,
                                        const float *u, int32_t *out_tokens, void *stream) {
    g_pdl = true;
    if (!logits || !temperature || !top_p || !u || !out_tokens)
        return fail(BLOOM_E_INVALID, "null argument");
    if (B < 1 || B > 65535 || V < 1 || ld < V)
        return fail(BLOOM_E_INVALID, "B=%d V=%d ld=%lld", B, V, (long long)ld);
    SampleArgs a;
    a.logits = logits;
    a.ld = ld;
    a.B = B;
    a.V = V;
    a.temperature = temperature;
    a.top_p = top_p;
    a.u = u;
    a.out = out_tokens;
    CK(launch_sample(a, (cudaStream_t)stream));
    return BLOOM_OK;
}

extern "C" bloom_status bloom_decode_step_sampled(bloom_model *m, bloom_kv *kv,
                                                  const int32_t *next_tokens, int32_t *out_tokens,
                                                  float *logits, const float *temperature,
                                                  const float *top_p, const float *u,
                                                  void *stream) {
    NvtxRange range("bloom_decode_step_sampled");
    if (!logits || !temperature || !top_p || !u) return fail(BLOOM_E_INVALID, "null argument");
    bloom_status st = bloom_decode_step(m, kv, next_tokens, out_tokens, logits, stream);
    if (st) return st;
    SampleArgs a;
    a.logits = logits;
    a.ld = m->cfg.vocab;
    a.B = kv->batch;
    a.V = m->cfg.vocab;
    a.temperature = temperature;
    a.top_p = top_p;
    a.u = u;
    a.active = kv_ptrs(m, kv).active;
    a.out = out_tokens;
    CK(launch_sample(a, (cudaStream_t)stream));
    return BLOOM_OK;
}

extern "C" bloom_status bloom_op_lmhead_argmax(const void *x, const void *emb, int32_t M,
                                               int32_t V, int32_t K, int32_t *out_tokens,
                                               float *out_logits, void *stream) {
    g_pdl = true;
    if (!x || !emb || !out_tokens) return fail(BLOOM_E_INVALID, "null argument");
    if (M < 1 || M > kMaxBatch || V < 1 || K < 8 || K % 8)
        return fail(BLOOM_E_UNSUPPORTED, "M=%d V=%d K=%d", M, V, K);
    if (!aligned16(x) || !aligned16(emb)) return fail(BLOOM_E_INVALID, "pointers must be 16-byte aligned");
    cudaStream_t s = (cudaStream_t)stream;
    void *scratch = nullptr;
    const size_t bytes = 256 + align256((size_t)M * 8);
    CK(cudaMallocAsync(&scratch, bytes, s));
    cudaError_t e = cudaMemsetAsync(scratch, 0, bytes, s);
    LinearArgs a;
    a.w = emb;
    a.x = (const uint16_t *)x;
    a.M = M;
    a.N = V;
    a.K = K;
    a.epi = EPI_ARGMAX;
    a.logits = out_logits;
    a.ticket = (int *)scratch;
    a.best = (unsigned long long *)((char *)scratch + 256);
    a.out_tokens = out_tokens;
    if (e == cudaSuccess) e = launch_linear(a, device_sms(), s);
    cudaError_t e2 = cudaFreeAsync(scratch, s);
    CK(e);
    CK(e2);
    return BLOOM_OK;
}
