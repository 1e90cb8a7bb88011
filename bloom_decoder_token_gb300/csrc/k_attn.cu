// ALiBi attention over the KV cache: split-KV decode kernel and prefill kernel.
//
// Score of key k for a query of head j:  s_k = (q . k_k) / sqrt(d) + slope_j * pos_k,
// where pos_k is the key's position counted from the sequence's first token;
// a masked key (pad slot, pos_k = -1) takes no part in the softmax (its
// probability is exactly 0), which is what the masked_fill + float32 softmax
// of "Hugging Face BLOOM Inference Optimization" (Custom CUDA Kernels) computes.
// Scores, maxima, sums and the output accumulators are float32; only K, V, q
// and the output are bf16.
#include <math.h>

#include "attn_ops.cuh"
#include "common.cuh"
#include "kernels.h"

namespace bloom {

constexpr int kAttnThreads = 128;

// ---------------------------------------------------------------------------
// Decode: one query per (sequence, head).  Grid (splits, n_head, B): each CTA
// takes one contiguous key range (attn_decode_block).
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kAttnThreads) attn_decode_kernel(const AttnDecodeArgs a) {
    __shared__ AttnSmem<D, kAttnThreads> sm;
    griddep_launch();
    griddep_wait();
    attn_decode_block<D, kAttnThreads>(a, blockIdx.x, blockIdx.y, blockIdx.z, sm);
}

// ---------------------------------------------------------------------------
// Prefill: causal + pad-masked ALiBi attention of every prompt slot.  One warp
// per query; blocks of 32 keys with an online softmax: lane i scores key i of
// the block (q broadcast from shared memory), then every lane accumulates its
// d/32 output elements over the block's keys.
// ---------------------------------------------------------------------------
constexpr int kPrefillWarps = 4;

template <int D>
__global__ void __launch_bounds__(kPrefillWarps * 32) attn_prefill_kernel(const AttnPrefillArgs a) {
    constexpr int EPL = D / 32;
    __shared__ __align__(16) float s_q[kPrefillWarps][D];
    griddep_launch();
    griddep_wait();
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * kPrefillWarps + w;
    const int j = blockIdx.y, b = blockIdx.z;
    if (t >= a.T) return;
    const size_t m = (size_t)b * a.T + t;
    uint16_t *out = a.o + m * a.n * D + (size_t)j * D + lane * EPL;
    const int pt = a.pos[(size_t)b * a.max_seq + t];
    if (pt < 0) {
#pragma unroll
        for (int e = 0; e < EPL; ++e) out[e] = 0;
        return;
    }
    const uint16_t *qp = a.q + m * a.n * D + (size_t)j * D;
    for (int e = lane; e < D; e += 32) s_q[w][e] = bf2f(qp[e]);
    __syncwarp();
    const size_t bh = (size_t)b * a.n + j;
    const uint16_t *kbase = a.k + bh * a.max_seq * D;
    const uint16_t *vbase = a.v + bh * a.max_seq * D;
    const int *posb = a.pos + (size_t)b * a.max_seq;
    const float slope = a.slopes[j];

    float m_run = -INFINITY, l_run = 0.f, acc[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
    for (int kb = 0; kb <= t; kb += 32) {
        const int k = kb + lane;
        float s = -INFINITY;
        if (k <= t) {
            const int pk = posb[k];
            if (pk >= 0) {
                const uint16_t *kp = kbase + (size_t)k * D;
                float dot = 0.f;
#pragma unroll 4
                for (int i = 0; i < D; i += 8) {
                    float kf[8];
                    unpack8(*reinterpret_cast<const uint4 *>(kp + i), kf);
                    const float4 q0 = *reinterpret_cast<const float4 *>(&s_q[w][i]);
                    const float4 q1 = *reinterpret_cast<const float4 *>(&s_q[w][i + 4]);
                    dot = fmaf(q0.x, kf[0], dot); dot = fmaf(q0.y, kf[1], dot);
                    dot = fmaf(q0.z, kf[2], dot); dot = fmaf(q0.w, kf[3], dot);
                    dot = fmaf(q1.x, kf[4], dot); dot = fmaf(q1.y, kf[5], dot);
                    dot = fmaf(q1.z, kf[6], dot); dot = fmaf(q1.w, kf[7], dot);
                }
                s = dot * a.scale + slope * (float)pk;
            }
        }
        const float bmax = warp_max(s);
        const float m_new = fmaxf(m_run, bmax);
        if (m_new == -INFINITY) continue;   // whole block masked, nothing seen yet
        const float corr = expf(m_run - m_new);
        const float p = (s == -INFINITY) ? 0.f : expf(s - m_new);
        l_run = l_run * corr + warp_sum(p);
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[e] *= corr;
        const int kn = min(32, t + 1 - kb);
        for (int i = 0; i < kn; ++i) {
            const float pi = __shfl_sync(0xffffffffu, p, i);
            if (pi == 0.f) continue;
            const uint16_t *vp = vbase + (size_t)(kb + i) * D + lane * EPL;
            if constexpr (EPL == 4) {
                const uint2 vv = *reinterpret_cast<const uint2 *>(vp);
                acc[0] = fmaf(pi, bf_lo(vv.x), acc[0]);
                acc[1] = fmaf(pi, bf_hi(vv.x), acc[1]);
                acc[2] = fmaf(pi, bf_lo(vv.y), acc[2]);
                acc[3] = fmaf(pi, bf_hi(vv.y), acc[3]);
            } else {
                const uint32_t vv = *reinterpret_cast<const uint32_t *>(vp);
                acc[0] = fmaf(pi, bf_lo(vv), acc[0]);
                acc[1] = fmaf(pi, bf_hi(vv), acc[1]);
            }
        }
        m_run = m_new;
    }
    const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) out[e] = f2bf(acc[e] * inv);
}

cudaError_t launch_attn_decode(const AttnDecodeArgs &a, cudaStream_t s) {
    dim3 grid(a.splits, a.n, a.B);
    if (a.d == 64) return launch_pdl(attn_decode_kernel<64>, grid, dim3(kAttnThreads), s, a);
    if (a.d == 128) return launch_pdl(attn_decode_kernel<128>, grid, dim3(kAttnThreads), s, a);
    return cudaErrorInvalidValue;
}

cudaError_t launch_attn_prefill(const AttnPrefillArgs &a, cudaStream_t s) {
    dim3 grid((a.T + kPrefillWarps - 1) / kPrefillWarps, a.n, a.B);
    if (a.d == 64) return launch_pdl(attn_prefill_kernel<64>, grid, dim3(kPrefillWarps * 32), s, a);
    if (a.d == 128) return launch_pdl(attn_prefill_kernel<128>, grid, dim3(kPrefillWarps * 32), s, a);
    return cudaErrorInvalidValue;
}

}  // namespace bloom
