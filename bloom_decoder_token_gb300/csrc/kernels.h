// Host-side launch interface of the kernels (internal to the library).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace bloom {

// Programmatic dependent launch for every kernel of the path (set per call from
// the model's flags; BLOOM_FLAG_NO_PDL turns it off).
extern thread_local bool g_pdl;

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_smem(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = g_pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, cudaStream_t s,
                       Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = g_pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

constexpr int kMaxBatch = 256;      // largest batch the argmax / decode kernels take
constexpr int kMaxSplits = 16;      // largest split-KV count
constexpr int kMaxHidden = 16384;   // LayerNorm register tile bound
constexpr int kLnFuseMaxM = 2;      // fused input LayerNorm: at most this many token rows
constexpr int kLnFuseSmemMax = kLnFuseMaxM * (2 * kMaxHidden + 64);

enum Epi : int {
    EPI_STORE = 0,   // out = acc + bias
    EPI_GELU = 1,    // out = gelu(acc + bias)
    EPI_RESID = 2,   // out += acc + bias
    EPI_QKV = 3,     // head-interleaved q | k | v scatter: q -> q_out, k/v -> cache slot
    EPI_ARGMAX = 4,  // tied LM head: float logits (optional) + fused argmax
    EPI_RESID32 = 5, // out32 += acc + bias (float32 residual stream)
};

struct LinearArgs {
    const void *w = nullptr;          // bf16 or int8 [N][K]
    const uint16_t *scale = nullptr;  // bf16 [N] (int8)
    const uint16_t *bias = nullptr;   // bf16 [N] or null
    const uint16_t *x = nullptr;      // bf16 [M][K]
    int M = 0, N = 0, K = 0;
    int int8 = 0;
    int epi = EPI_STORE;
    uint16_t *out = nullptr;          // bf16 [M][N] (STORE / GELU / RESID)
    float *out32 = nullptr;           // float [M][N] (RESID32)
    // EPI_QKV
    uint16_t *q_out = nullptr;        // bf16 [M][n_head * d]
    uint16_t *k_cache = nullptr;      // bf16 [Bkv][n_head][max_seq][d] (this layer)
    uint16_t *v_cache = nullptr;
    // decode: token m is sequence m, appended at slot len_ptr[m] if active[m]
    const int *len_ptr = nullptr;
    const int *active = nullptr;
    // prefill: token m is slot m % T of prompt m / T, which goes to cache row
    // row_map[m / T] (row_map null: row m / T)
    int T = 0;
    const int *row_map = nullptr;
    int n_head = 0, head_dim = 0, max_seq = 0;
    // EPI_ARGMAX
    float *logits = nullptr;          // float [M][N] or null
    unsigned long long *best = nullptr;  // [M], zero at rest
    int *ticket = nullptr;            // zero at rest
    int *out_tokens = nullptr;        // [M]
    // decode step: rows with active[m] == 0 get token -1; if len_inc is set, the
    // last CTA advances len_inc[m] and next_pos[m] of every active row
    int *len_inc = nullptr;
    int *next_pos = nullptr;
    int *err = nullptr;
    unsigned long long wait_ns = 0;   // bound of the tensor-core kernels' waits (0: ~2 s)
    // fused input LayerNorm (decode, see linear_can_fuse_ln): x = LN(ln_x) with ln_g, ln_b
    const float *ln_x = nullptr;      // float [M][K] residual rows
    const uint16_t *ln_g = nullptr, *ln_b = nullptr;
    float ln_eps = 1e-5f;
};

// Whether the input LayerNorm can be fused into this linear layer (decode, at
// most kLnFuseMaxM rows that fit in shared memory).
bool linear_can_fuse_ln(const LinearArgs &a);

cudaError_t launch_linear(const LinearArgs &a, int num_sms, cudaStream_t s);

// Tensor-core GEMM (tcgen05 / TMEM / TMA) for prefill-sized M, bf16 weights.
// A map describes a row-major bf16 [rows][K] matrix for the kernel's TMA loads:
// gemm_make_map fills gemm_map_bytes() bytes (64-byte aligned storage) and
// returns false if the driver refuses (base not 16-byte aligned, K % 8 != 0).
// X maps use box rows gemm_box_rows_x(), W maps gemm_box_rows_w().
bool gemm_make_map(void *map, const void *base, long long rows, long long K, int box_rows);
// The same for int8 weights [rows][K] (K % 16 == 0): boxes of box_rows x 128 bytes.
bool gemm_make_map_u8(void *map, const void *base, long long rows, long long K, int box_rows);
size_t gemm_map_bytes();
int gemm_box_rows_x();
int gemm_box_rows_w();
cudaError_t gemm_prepare();
// Epilogues STORE / GELU / RESID / RESID32 / QKV (prefill: a.T > 0, d % 32 == 0).
cudaError_t launch_gemm_tc(const void *map_x, const void *map_w, const LinearArgs &a,
                           cudaStream_t s);
constexpr int kTcMinM = 128;        // prefill linears with at least this many tokens use it

// Decode linear on the tensor cores (tcgen05 / TMEM / TMA): W is the 128-row
// A operand, the M <= 256 tokens the N operand (NT = gemv_tc_nt(M) columns).
// map_w: W [N][K] with box rows gemv_tc_box_rows_w() (gemm_make_map, or
// gemm_make_map_u8 for int8 weights: a.int8, a.scale, M <= 128, not ARGMAX);
// map_x: x [>= M][K] with box rows NT.  splits > 1 splits K over a thread-block cluster of that many
// CTAs per row tile (gemv_tc_splits; not for ARGMAX or NT = 256).
struct GemvTcArgs {
    LinearArgs a;
    int splits = 1;
};
int gemv_tc_nt(int M);
int gemv_tc_splits(int N, int K, int M, int epi, int num_sms, int int8 = 0);
constexpr int kGvInt8MaxNt = 128;   // int8 weights: token columns up to this
int gemv_tc_box_rows_w();
cudaError_t gemv_tc_prepare();
cudaError_t launch_gemv_tc(const void *map_w, const void *map_x, const GemvTcArgs &g, int nt,
                           cudaStream_t s);

// Library-internal host helpers (defined with the C ABI): set the message of
// bloom_last_error(), and the SM count of the current device.
void bloom_set_error(const char *fmt, ...);
int bloom_device_sms();
cudaError_t linear_prepare();

// LayerNorm of `rows` rows.  Source row r is x[(r * src_stride + (last ? last[r] : 0)) * h].
cudaError_t launch_layernorm(const uint16_t *x, const uint16_t *g, const uint16_t *b, int rows,
                             int h, float eps, uint16_t *y, int src_stride, const int *last,
                             cudaStream_t s);

cudaError_t launch_layernorm_f32(const float *x, const uint16_t *g, const uint16_t *b, int rows,
                                 int h, float eps, uint16_t *y, int src_stride, const int *last,
                                 cudaStream_t s);

// Embedding gather + LN for n tokens into the float32 residual stream x.  With
// step state (len != null) it also records, for each active sequence r, the
// position of its next slot: pos[r][len[r]] = next_pos[r].
cudaError_t launch_embed(const int *tokens, int n, const uint16_t *emb, int vocab,
                         const uint16_t *g, const uint16_t *b, int h, float eps, float *x,
                         const int *len, const int *active, const int *next_pos, int *pos,
                         int max_seq, int *err, cudaStream_t s);

// pos[b][len[b]] = next_pos[b] for the active ones of B sequences (layer-level
// decode entry).
cudaError_t launch_slot_pos(int B, const int *len, const int *active, const int *next_pos,
                            int *pos, int max_seq, int *err, cudaStream_t s);

// Prompt setup of n prompts going to cache rows row_map[i] (null: row i): pos of
// their T slots from the mask cumsum, next_pos, len = T, active = 1 for those
// rows, and last[i] (the prompt's last token slot).
cudaError_t launch_prompt_setup(const uint8_t *mask, int n, int T, const int *row_map, int *pos,
                                int max_seq, int *next_pos, int *len, int *active, int *last,
                                int *err, cudaStream_t s);

// active[rows[i]] = value for n rows given by value (n <= kMaxBatch).
struct RowList {
    int rows[256];
    int n = 0;
};
cudaError_t launch_set_active(const RowList &r, int value, int *active, cudaStream_t s);
// dst[i] = rows[i] for the n rows.
cudaError_t launch_set_rows(const RowList &r, int *dst, cudaStream_t s);

struct AttnDecodeArgs {
    const uint16_t *q = nullptr;     // [B][n][d]
    const uint16_t *k = nullptr;     // [B][n][max_seq][d]
    const uint16_t *v = nullptr;
    const int *pos = nullptr;        // [B][max_seq]
    const float *slopes = nullptr;   // [n]
    // keys [0, len_ptr[b]] of an active sequence, [0, len_ptr[b]) of an idle one
    // (active null: all active); len_ptr null: keys [0, len_host] of every sequence
    const int *len_ptr = nullptr;
    const int *active = nullptr;
    int len_host = 0;
    int B = 0, n = 0, d = 0, max_seq = 0;
    int splits = 1;
    // the lengths, the activity and every key below the length were written before
    // the previous kernel started (a decode step replayed as a graph): the kernel
    // loads them before it waits for the previous kernel
    int early = 0;
    // 128-thread CTAs of the d = 128 kernel resident at once (larger grids take
    // 64-thread CTAs); attn_decode_resident_ctas
    long long resident_ctas = 0;
    long long resident_wide = 0;       // the same for the 64-thread form
    // K and V in device memory: grids beyond resident_wide stage them by bulk
    // copies (attn_decode_block_bulk); host-resident (offloaded) caches are read directly
    int bulk = 0;
    int *err = nullptr;                // device flag word (8: a bounded wait expired)
    unsigned long long wait_ns = 0;    // bound of its waits (0: about 2 s)
    float scale = 0.f;               // 1/sqrt(d)
    float *part = nullptr;           // [B][n][splits][d + 2]
    int *ticket = nullptr;           // [B][n], zero at rest
    uint16_t *o = nullptr;           // [B][n*d]
};
cudaError_t launch_attn_decode(const AttnDecodeArgs &a, cudaStream_t s);
int attn_decode_resident_ctas(int d, int num_sms, int wide = 0);

// Per-member temperature + top-p sampling of B rows of float32 logits
// (k_sample.cu): row b's logits at logits + b * ld, its temperature, top-p and
// uniform number u in [0, 1) at index b of the three arrays; out[b] = token.
struct SampleArgs {
    const float *logits = nullptr;
    long long ld = 0;
    int B = 0, V = 0;
    const float *temperature = nullptr;
    const float *top_p = nullptr;
    const float *u = nullptr;
    const int32_t *active = nullptr;   // optional: rows with active[b] == 0 get -1
    int32_t *out = nullptr;
};
cudaError_t launch_sample(const SampleArgs &a, cudaStream_t s);

struct AttnPrefillArgs {
    const uint16_t *q = nullptr;     // [B*T][n][d], prompt i's tokens at rows i*T ..
    const uint16_t *k = nullptr;     // [rows][n][max_seq][d] (the cache)
    const uint16_t *v = nullptr;
    const int *pos = nullptr;        // [rows][max_seq]
    const int *row_map = nullptr;    // prompt i's cache row (null: row i)
    const float *slopes = nullptr;
    int B = 0, T = 0, n = 0, d = 0, max_seq = 0;
    float scale = 0.f;
    uint16_t *o = nullptr;           // [B*T][n*d]
};
// Causal, pad-masked ALiBi attention of every prompt slot on the tensor cores
// (mma.sync, 64-query x 64-key tiles); d in {64, 128}; rows of q, k and v
// 16-byte aligned.
cudaError_t launch_attn_prefill_tc(const AttnPrefillArgs &a, cudaStream_t s);

}  // namespace bloom
