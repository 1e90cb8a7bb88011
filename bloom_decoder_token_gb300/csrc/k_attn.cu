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

#include "common.cuh"
#include "kernels.h"

namespace bloom {

constexpr int kAttnThreads = 128;
constexpr int kKeyTile = 64;

// ---------------------------------------------------------------------------
// Decode: one query per (sequence, head).  Grid (splits, n_head, B): each CTA
// takes one contiguous key range and runs an online softmax over tiles of 64
// keys; the last CTA of a (sequence, head) to finish merges the split partials
// (m, l, acc) by rescaling with exp(m_split - m_max).
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kAttnThreads) attn_decode_kernel(const AttnDecodeArgs a) {
    constexpr int EPT = D / 8;             // q / k elements per lane of an 8-lane group
    constexpr int GV = kAttnThreads / (D / 2);   // value groups (each thread: 2 elements)
    __shared__ float s_tile[kKeyTile];
    __shared__ float s_acc[GV][D];
    __shared__ int s_last;

    const int split = blockIdx.x, j = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31;
    const int nk = min((a.len_ptr ? *a.len_ptr : a.len_host) + 1, a.max_seq);
    const int chunk = (nk + a.splits - 1) / a.splits;
    const int k0 = split * chunk;
    const int k1 = min(nk, k0 + chunk);

    const size_t bh = (size_t)b * a.n + j;
    const uint16_t *kbase = a.k + bh * a.max_seq * D;
    const uint16_t *vbase = a.v + bh * a.max_seq * D;
    const int *posb = a.pos + (size_t)b * a.max_seq;
    const float slope = a.slopes[j];

    // q slice of this lane within its 8-lane group
    const int grp = tid >> 3, sub = tid & 7;
    float qf[EPT];
    {
        const uint16_t *qp = a.q + bh * D + sub * EPT;
#pragma unroll
        for (int i = 0; i < EPT; i += 8) unpack8(*reinterpret_cast<const uint4 *>(qp + i), qf + i);
    }
    // value slice: two elements
    const int vg = tid / (D / 2), e2 = tid - vg * (D / 2);

    float m_run = -INFINITY, l_run = 0.f, acc0 = 0.f, acc1 = 0.f;
    for (int kt = k0; kt < k1; kt += kKeyTile) {
        const int kn = min(kKeyTile, k1 - kt);
        // scores: 16 groups x 4 rounds
        for (int kk = grp; kk < kKeyTile; kk += kAttnThreads / 8) {
            float dot = 0.f;
            const bool live = kk < kn;
            if (live) {
                const uint16_t *kp = kbase + (size_t)(kt + kk) * D + sub * EPT;
#pragma unroll
                for (int i = 0; i < EPT; i += 8) {
                    float kf[8];
                    unpack8(*reinterpret_cast<const uint4 *>(kp + i), kf);
#pragma unroll
                    for (int e = 0; e < 8; ++e) dot = fmaf(qf[i + e], kf[e], dot);
                }
            }
            dot += __shfl_xor_sync(0xffffffffu, dot, 4);
            dot += __shfl_xor_sync(0xffffffffu, dot, 2);
            dot += __shfl_xor_sync(0xffffffffu, dot, 1);
            if (sub == 0) {
                float s = -INFINITY;
                if (live) {
                    const int p = posb[kt + kk];
                    if (p >= 0) s = dot * a.scale + slope * (float)p;
                }
                s_tile[kk] = s;
            }
        }
        __syncthreads();
        // tile max and sum (every warp computes the same values)
        const float s0 = s_tile[lane], s1 = s_tile[lane + 32];
        const float tmax = warp_max(fmaxf(s0, s1));
        const float m_new = fmaxf(m_run, tmax);
        float corr, p0, p1;
        if (m_new == -INFINITY) {
            corr = 1.f; p0 = 0.f; p1 = 0.f;
        } else {
            corr = expf(m_run - m_new);
            p0 = (s0 == -INFINITY) ? 0.f : expf(s0 - m_new);
            p1 = (s1 == -INFINITY) ? 0.f : expf(s1 - m_new);
        }
        l_run = l_run * corr + warp_sum(p0 + p1);
        acc0 *= corr;
        acc1 *= corr;
        if (m_new != -INFINITY) {
            for (int kk = vg; kk < kn; kk += GV) {
                const float s = s_tile[kk];
                if (s == -INFINITY) continue;
                const float p = expf(s - m_new);
                const uint32_t vv =
                    *reinterpret_cast<const uint32_t *>(vbase + (size_t)(kt + kk) * D + 2 * e2);
                acc0 = fmaf(p, bf_lo(vv), acc0);
                acc1 = fmaf(p, bf_hi(vv), acc1);
            }
        }
        m_run = m_new;
        __syncthreads();
    }
    s_acc[vg][2 * e2] = acc0;
    s_acc[vg][2 * e2 + 1] = acc1;
    __syncthreads();

    if (a.splits == 1) {
        if (tid < D) {
            float t = 0.f;
#pragma unroll
            for (int g = 0; g < GV; ++g) t += s_acc[g][tid];
            a.o[(size_t)b * a.n * D + (size_t)j * D + tid] = f2bf(l_run > 0.f ? t / l_run : 0.f);
        }
        return;
    }
    float *part = a.part + (bh * a.splits + split) * (D + 2);
    if (tid < D) {
        float t = 0.f;
#pragma unroll
        for (int g = 0; g < GV; ++g) t += s_acc[g][tid];
        part[2 + tid] = t;
    }
    if (tid == 0) {
        part[0] = m_run;
        part[1] = l_run;
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = (atomicAdd(a.ticket + bh, 1) == a.splits - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (tid < D) {
        const float *pb = a.part + bh * a.splits * (D + 2);
        float M = -INFINITY;
        for (int sp = 0; sp < a.splits; ++sp) M = fmaxf(M, __ldcg(pb + sp * (D + 2)));
        float L = 0.f, A = 0.f;
        if (M != -INFINITY) {
            for (int sp = 0; sp < a.splits; ++sp) {
                const float ms = __ldcg(pb + sp * (D + 2));
                if (ms == -INFINITY) continue;
                const float w = expf(ms - M);
                L = fmaf(__ldcg(pb + sp * (D + 2) + 1), w, L);
                A = fmaf(__ldcg(pb + sp * (D + 2) + 2 + tid), w, A);
            }
        }
        a.o[(size_t)b * a.n * D + (size_t)j * D + tid] = f2bf(L > 0.f ? A / L : 0.f);
    }
    if (tid == 0) a.ticket[bh] = 0;
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
    if (a.d == 64) attn_decode_kernel<64><<<grid, kAttnThreads, 0, s>>>(a);
    else if (a.d == 128) attn_decode_kernel<128><<<grid, kAttnThreads, 0, s>>>(a);
    else return cudaErrorInvalidValue;
    return cudaGetLastError();
}

cudaError_t launch_attn_prefill(const AttnPrefillArgs &a, cudaStream_t s) {
    dim3 grid((a.T + kPrefillWarps - 1) / kPrefillWarps, a.n, a.B);
    if (a.d == 64) attn_prefill_kernel<64><<<grid, kPrefillWarps * 32, 0, s>>>(a);
    else if (a.d == 128) attn_prefill_kernel<128><<<grid, kPrefillWarps * 32, 0, s>>>(a);
    else return cudaErrorInvalidValue;
    return cudaGetLastError();
}

}  // namespace bloom
