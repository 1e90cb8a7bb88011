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

// ---------------------------------------------------------------------------
// Decode: one query per (sequence, head).  Grid (splits, n_head, B): each CTA
// takes one contiguous key range.  Inside a CTA, 16 groups of 8 lanes each run
// an online softmax (running max m, sum l, accumulator) over their own keys,
// two keys in flight per group; lane `sub` of a group owns d/8 elements of q
// and of the accumulator, so a key costs one 3-step shuffle for the dot
// product and no other communication.  Groups merge by shuffles, warps through
// shared memory, and the last CTA of a (sequence, head) to finish merges the
// split partials by rescaling with exp(m_split - m_max) -- no second kernel and
// no waiting.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void softmax_merge(float &m, float &l, float *acc, int n, float mo,
                                              float lo, const float *acco) {
    const float M = fmaxf(m, mo);
    if (M == -INFINITY) return;
    const float a = (m == -INFINITY) ? 0.f : expf(m - M);
    const float b = (mo == -INFINITY) ? 0.f : expf(mo - M);
    l = l * a + lo * b;
    for (int e = 0; e < n; ++e) acc[e] = acc[e] * a + acco[e] * b;
    m = M;
}

template <int D>
__global__ void __launch_bounds__(kAttnThreads) attn_decode_kernel(const AttnDecodeArgs a) {
    constexpr int EPT = D / 8;             // elements per lane of an 8-lane group
    constexpr int NW = kAttnThreads / 32;
    __shared__ float s_m[NW], s_l[NW];
    __shared__ float s_acc[NW][D];
    __shared__ int s_last;

    griddep_launch();
    griddep_wait();
    const int split = blockIdx.x, j = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int grp = tid >> 3, sub = tid & 7;   // 16 groups
    const int nk = min((a.len_ptr ? *a.len_ptr : a.len_host) + 1, a.max_seq);
    const int chunk = (nk + a.splits - 1) / a.splits;
    const int k0 = split * chunk;
    const int k1 = min(nk, k0 + chunk);

    const size_t bh = (size_t)b * a.n + j;
    const uint16_t *kbase = a.k + bh * a.max_seq * D + sub * EPT;
    const uint16_t *vbase = a.v + bh * a.max_seq * D + sub * EPT;
    const int *posb = a.pos + (size_t)b * a.max_seq;
    const float slope = a.slopes[j];

    float qf[EPT], acc[EPT];
    {
        const uint16_t *qp = a.q + bh * D + sub * EPT;
#pragma unroll
        for (int i = 0; i < EPT; i += 8) unpack8(*reinterpret_cast<const uint4 *>(qp + i), qf + i);
#pragma unroll
        for (int e = 0; e < EPT; ++e) {
            qf[e] *= a.scale;
            acc[e] = 0.f;
        }
    }
    float m_run = -INFINITY, l_run = 0.f;
    const int rounds = (k1 - k0 + 31) / 32;
    for (int r = 0; r < rounds; ++r) {
        const int ka = k0 + r * 32 + grp, kb = ka + 16;
        const bool la = ka < k1, lb = kb < k1;
        uint4 kva[EPT / 8], kvb[EPT / 8], vva[EPT / 8], vvb[EPT / 8];
        int pa = -1, pb = -1;
        if (la) {
            pa = posb[ka];
#pragma unroll
            for (int i = 0; i < EPT / 8; ++i) {
                kva[i] = *reinterpret_cast<const uint4 *>(kbase + (size_t)ka * D + 8 * i);
                vva[i] = *reinterpret_cast<const uint4 *>(vbase + (size_t)ka * D + 8 * i);
            }
        }
        if (lb) {
            pb = posb[kb];
#pragma unroll
            for (int i = 0; i < EPT / 8; ++i) {
                kvb[i] = *reinterpret_cast<const uint4 *>(kbase + (size_t)kb * D + 8 * i);
                vvb[i] = *reinterpret_cast<const uint4 *>(vbase + (size_t)kb * D + 8 * i);
            }
        }
        float da = 0.f, db = 0.f;
#pragma unroll
        for (int i = 0; i < EPT / 8; ++i) {
            float f[8];
            if (la) {
                unpack8(kva[i], f);
#pragma unroll
                for (int e = 0; e < 8; ++e) da = fmaf(qf[8 * i + e], f[e], da);
            }
            if (lb) {
                unpack8(kvb[i], f);
#pragma unroll
                for (int e = 0; e < 8; ++e) db = fmaf(qf[8 * i + e], f[e], db);
            }
        }
#pragma unroll
        for (int o = 4; o > 0; o >>= 1) {
            da += __shfl_xor_sync(0xffffffffu, da, o);
            db += __shfl_xor_sync(0xffffffffu, db, o);
        }
        const float sa = (la && pa >= 0) ? da + slope * (float)pa : -INFINITY;
        const float sb = (lb && pb >= 0) ? db + slope * (float)pb : -INFINITY;
        const float m_new = fmaxf(m_run, fmaxf(sa, sb));
        if (m_new == -INFINITY) continue;   // uniform within the group
        const float corr = (m_run == -INFINITY) ? 0.f : expf(m_run - m_new);
        const float wa = (sa == -INFINITY) ? 0.f : expf(sa - m_new);
        const float wb = (sb == -INFINITY) ? 0.f : expf(sb - m_new);
        l_run = l_run * corr + wa + wb;
#pragma unroll
        for (int i = 0; i < EPT / 8; ++i) {
            float fa[8], fb[8];
            if (wa != 0.f) unpack8(vva[i], fa);
            else for (int e = 0; e < 8; ++e) fa[e] = 0.f;
            if (wb != 0.f) unpack8(vvb[i], fb);
            else for (int e = 0; e < 8; ++e) fb[e] = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e)
                acc[8 * i + e] = fmaf(wb, fb[e], fmaf(wa, fa[e], acc[8 * i + e] * corr));
        }
        m_run = m_new;
    }
    // merge the 4 groups of this warp (lanes with equal `sub` hold the same slice)
#pragma unroll
    for (int o = 8; o < 32; o <<= 1) {
        const float mo = __shfl_xor_sync(0xffffffffu, m_run, o);
        const float lo = __shfl_xor_sync(0xffffffffu, l_run, o);
        float ao[EPT];
#pragma unroll
        for (int e = 0; e < EPT; ++e) ao[e] = __shfl_xor_sync(0xffffffffu, acc[e], o);
        softmax_merge(m_run, l_run, acc, EPT, mo, lo, ao);
    }
    // merge the warps through shared memory
    if (lane < 8) {
#pragma unroll
        for (int e = 0; e < EPT; ++e) s_acc[warp][sub * EPT + e] = acc[e];
        if (lane == 0) {
            s_m[warp] = m_run;
            s_l[warp] = l_run;
        }
    }
    __syncthreads();
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, s_m[w]);
    float L = 0.f, A = 0.f;
    if (tid < D && M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            if (s_m[w] == -INFINITY) continue;
            const float wgt = expf(s_m[w] - M);
            L = fmaf(s_l[w], wgt, L);
            A = fmaf(s_acc[w][tid], wgt, A);
        }
    }
    if (a.splits == 1) {
        if (tid < D) a.o[(size_t)b * a.n * D + (size_t)j * D + tid] = f2bf(L > 0.f ? A / L : 0.f);
        return;
    }
    float *part = a.part + (bh * a.splits + split) * (D + 2);
    if (tid < D) part[2 + tid] = A;
    if (tid == 0) {
        part[0] = M;
        part[1] = L;
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = (atomicAdd(a.ticket + bh, 1) == a.splits - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (tid < D) {
        const float *pb = a.part + bh * a.splits * (D + 2);
        float Mx = -INFINITY;
        for (int sp = 0; sp < a.splits; ++sp) Mx = fmaxf(Mx, __ldcg(pb + sp * (D + 2)));
        float Ls = 0.f, As = 0.f;
        if (Mx != -INFINITY) {
            for (int sp = 0; sp < a.splits; ++sp) {
                const float ms = __ldcg(pb + sp * (D + 2));
                if (ms == -INFINITY) continue;
                const float wgt = expf(ms - Mx);
                Ls = fmaf(__ldcg(pb + sp * (D + 2) + 1), wgt, Ls);
                As = fmaf(__ldcg(pb + sp * (D + 2) + 2 + tid), wgt, As);
            }
        }
        a.o[(size_t)b * a.n * D + (size_t)j * D + tid] = f2bf(Ls > 0.f ? As / Ls : 0.f);
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
