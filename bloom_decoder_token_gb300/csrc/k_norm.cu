// LayerNorm, embedding gather + LayerNorm, and the small step-state kernels.
//
// The residual stream x is a running sum over layers and is kept in float32
// (upcasting only the sums and accumulations, as the fused softmax of "Hugging
// Face BLOOM Inference Optimization" does); LayerNorm reads it and writes the
// bf16 activations the weight-streaming kernels consume.
//
// One CTA normalises one row, all its values held in registers: float32 mean,
// then float32 biased variance of the deviations (two passes over registers,
// no E[x^2] - mean^2 cancellation), eps inside the square root, affine gamma /
// beta, bf16 out.  "DeepSpeed Inference", III.B: all micro-operations of the
// layer norm, its reductions included, run in one kernel because the reduced
// dimension stays inside one thread block.
#include "common.cuh"
#include "kernels.h"
#include "norm_ops.cuh"

namespace bloom {

template <int CH, typename TIn>
__global__ void __launch_bounds__(kLnThreads)
layernorm_kernel(const TIn *x, const uint16_t *g, const uint16_t *b, int h, float eps,
                 uint16_t *y, int src_stride, const int *last) {
    __shared__ float red[kLnWarps];
    griddep_launch();
    LnAffine<CH> p;
    ln_affine_load(g, b, h, p);
    griddep_wait();
    const int r = blockIdx.x;
    const size_t src_row = (size_t)r * src_stride + (last ? last[r] : 0);
    ln_row(x + src_row * h, p, h, eps, y + (size_t)r * h, red);
}

template <int CH>
__global__ void __launch_bounds__(kLnThreads)
embed_kernel(const int *tokens, const uint16_t *emb, int vocab, const uint16_t *g,
             const uint16_t *b, int h, float eps, float *x, const int *len, const int *active,
             const int *next_pos, int *pos, int max_seq, int *err) {
    __shared__ float red[kLnWarps];
    griddep_launch();
    LnAffine<CH> p;
    ln_affine_load(g, b, h, p);
    griddep_wait();
    const int r = blockIdx.x;
    int tok = tokens[r];
    if (tok < 0 || tok >= vocab) {
        if (threadIdx.x == 0) atomicOr(err, kErrToken);
        tok = 0;
    }
    if (len && threadIdx.x == 0 && active[r]) {
        const int slot = len[r];
        if (slot >= 0 && slot < max_seq) pos[(size_t)r * max_seq + slot] = next_pos[r];
        else atomicOr(err, kErrSlot);
    }
    ln_row(emb + (size_t)tok * h, p, h, eps, x + (size_t)r * h, red);
}

__global__ void slot_pos_kernel(int B, const int *len, const int *active, const int *next_pos,
                                int *pos, int max_seq, int *err) {
    griddep_launch();
    griddep_wait();
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= B || !active[r]) return;
    const int slot = len[r];
    if (slot >= 0 && slot < max_seq) pos[(size_t)r * max_seq + slot] = next_pos[r];
    else atomicOr(err, kErrSlot);
}

// One warp per prompt: running count of tokens with a ballot scan.
__global__ void prompt_setup_kernel(const uint8_t *mask, int T, const int *row_map, int *pos,
                                    int max_seq, int *next_pos, int *len, int *active, int *last,
                                    int *err) {
    griddep_launch();
    griddep_wait();
    const int i = blockIdx.x;                       // prompt
    const int r = row_map ? row_map[i] : i;         // its cache row
    const int lane = threadIdx.x;
    int count = 0, last_t = -1;
    for (int t0 = 0; t0 < T; t0 += kWarp) {
        const int t = t0 + lane;
        const bool tok = (t < T) && mask[(size_t)i * T + t] != 0;
        const unsigned bal = __ballot_sync(0xffffffffu, tok);
        const int before = __popc(bal & ((1u << lane) - 1u));
        if (t < T) pos[(size_t)r * max_seq + t] = tok ? count + before : -1;
        count += __popc(bal);
        if (bal) last_t = t0 + 31 - __clz((int)bal);
    }
    if (lane == 0) {
        next_pos[r] = count;
        len[r] = T;
        active[r] = 1;
        last[i] = last_t < 0 ? T - 1 : last_t;
        if (count == 0) atomicOr(err, kErrEmptyRow);
    }
}

__global__ void set_active_kernel(const RowList rl, int value, int *active) {
    griddep_launch();
    griddep_wait();
    const int i = threadIdx.x;
    if (i < rl.n) active[rl.rows[i]] = value;
}

__global__ void set_rows_kernel(const RowList rl, int *dst) {
    griddep_launch();
    griddep_wait();
    const int i = threadIdx.x;
    if (i < rl.n) dst[i] = rl.rows[i];
}

template <typename TIn>
static cudaError_t launch_ln(const TIn *x, const uint16_t *g, const uint16_t *b, int rows, int h,
                             float eps, uint16_t *y, int src_stride, const int *last,
                             cudaStream_t s) {
    if (rows <= 0) return cudaSuccess;
    switch (ln_chunks(h)) {
    case 2:
        return launch_pdl(layernorm_kernel<2, TIn>, dim3(rows), dim3(kLnThreads), s, x, g, b, h,
                          eps, y, src_stride, last);
    case 4:
        return launch_pdl(layernorm_kernel<4, TIn>, dim3(rows), dim3(kLnThreads), s, x, g, b, h,
                          eps, y, src_stride, last);
    default:
        return launch_pdl(layernorm_kernel<kLnChunks, TIn>, dim3(rows), dim3(kLnThreads), s, x, g,
                          b, h, eps, y, src_stride, last);
    }
}

cudaError_t launch_layernorm(const uint16_t *x, const uint16_t *g, const uint16_t *b, int rows,
                             int h, float eps, uint16_t *y, int src_stride, const int *last,
                             cudaStream_t s) {
    return launch_ln(x, g, b, rows, h, eps, y, src_stride, last, s);
}

cudaError_t launch_layernorm_f32(const float *x, const uint16_t *g, const uint16_t *b, int rows,
                                 int h, float eps, uint16_t *y, int src_stride, const int *last,
                                 cudaStream_t s) {
    return launch_ln(x, g, b, rows, h, eps, y, src_stride, last, s);
}

cudaError_t launch_embed(const int *tokens, int n, const uint16_t *emb, int vocab,
                         const uint16_t *g, const uint16_t *b, int h, float eps, float *x,
                         const int *len, const int *active, const int *next_pos, int *pos,
                         int max_seq, int *err, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    switch (ln_chunks(h)) {
    case 2:
        return launch_pdl(embed_kernel<2>, dim3(n), dim3(kLnThreads), s, tokens, emb, vocab, g, b,
                          h, eps, x, len, active, next_pos, pos, max_seq, err);
    case 4:
        return launch_pdl(embed_kernel<4>, dim3(n), dim3(kLnThreads), s, tokens, emb, vocab, g, b,
                          h, eps, x, len, active, next_pos, pos, max_seq, err);
    default:
        return launch_pdl(embed_kernel<kLnChunks>, dim3(n), dim3(kLnThreads), s, tokens, emb,
                          vocab, g, b, h, eps, x, len, active, next_pos, pos, max_seq, err);
    }
}

cudaError_t launch_slot_pos(int B, const int *len, const int *active, const int *next_pos,
                            int *pos, int max_seq, int *err, cudaStream_t s) {
    return launch_pdl(slot_pos_kernel, dim3((B + 127) / 128), dim3(128), s, B, len, active,
                      next_pos, pos, max_seq, err);
}

cudaError_t launch_prompt_setup(const uint8_t *mask, int n, int T, const int *row_map, int *pos,
                                int max_seq, int *next_pos, int *len, int *active, int *last,
                                int *err, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    return launch_pdl(prompt_setup_kernel, dim3(n), dim3(kWarp), s, mask, T, row_map, pos, max_seq,
                      next_pos, len, active, last, err);
}

cudaError_t launch_set_active(const RowList &r, int value, int *active, cudaStream_t s) {
    if (r.n <= 0) return cudaSuccess;
    if (r.n > 256) return cudaErrorInvalidValue;
    return launch_pdl(set_active_kernel, dim3(1), dim3(256), s, r, value, active);
}

cudaError_t launch_set_rows(const RowList &r, int *dst, cudaStream_t s) {
    if (r.n <= 0) return cudaSuccess;
    if (r.n > 256) return cudaErrorInvalidValue;
    return launch_pdl(set_rows_kernel, dim3(1), dim3(256), s, r, dst);
}

}  // namespace bloom
