// Split-KV decode attention for one (sequence, head, key range), as a device
// function of a whole thread block (the body of the decode attention kernel).
//
// Score of key k for a query of head j:  s_k = (q . k_k) / sqrt(d) + slope_j * pos_k,
// where pos_k is the key's position counted from the sequence's first token;
// a masked key (pad slot, pos_k = -1) takes no part in the softmax (its
// probability is exactly 0), which is what the masked_fill + float32 softmax
// of "Hugging Face BLOOM Inference Optimization" (Custom CUDA Kernels) computes.
// Scores, maxima, sums and the output accumulators are float32; only K, V, q
// and the output are bf16.
//
// The block takes one contiguous key range.  Inside it, groups of 8 lanes run
// an online softmax (running max m, sum l, accumulator) over their own keys,
// two keys in flight per group; lane `sub` of a group owns d/8 elements of q
// and of the accumulator, so a key costs one 3-step shuffle for the dot
// product and no other communication.  Groups merge by shuffles, warps through
// shared memory, and the last block of a (sequence, head) to finish merges the
// split partials by rescaling with exp(m_split - m_max) -- no second pass and
// no waiting.
#pragma once

#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace bloom {

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

template <int D, int NT>
struct AttnSmem {
    float m[NT / 32], l[NT / 32];
    float acc[NT / 32][D];
    int last;
};

// All NT threads of the block call it with the same (split, j, b).  Contains
// barriers; the first one also protects `sm` from a previous call's readers.
template <int D, int NT>
__device__ __forceinline__ void attn_decode_block(const AttnDecodeArgs &a, int split, int j, int b,
                                                  AttnSmem<D, NT> &sm) {
    constexpr int EPT = D / 8;             // elements per lane of an 8-lane group
    constexpr int NW = NT / 32;
    constexpr int NG = NT / 8;             // groups; a round covers 2 * NG keys
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int grp = tid >> 3, sub = tid & 7;
    // keys [0, len] with the step's new one; an idle row appended none
    const int nk = a.len_ptr ? min(a.len_ptr[b] + ((!a.active || a.active[b]) ? 1 : 0), a.max_seq)
                             : min(a.len_host + 1, a.max_seq);
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
    const int rounds = (k1 - k0 + 2 * NG - 1) / (2 * NG);
    for (int r = 0; r < rounds; ++r) {
        const int ka = k0 + r * 2 * NG + grp, kb = ka + NG;
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
    __syncthreads();   // sm may still be read by a previous call
    // merge the warps through shared memory
    if (lane < 8) {
#pragma unroll
        for (int e = 0; e < EPT; ++e) sm.acc[warp][sub * EPT + e] = acc[e];
        if (lane == 0) {
            sm.m[warp] = m_run;
            sm.l[warp] = l_run;
        }
    }
    __syncthreads();
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, sm.m[w]);
    float L = 0.f, A = 0.f;
    if (tid < D && M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            if (sm.m[w] == -INFINITY) continue;
            const float wgt = expf(sm.m[w] - M);
            L = fmaf(sm.l[w], wgt, L);
            A = fmaf(sm.acc[w][tid], wgt, A);
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
    if (tid == 0) sm.last = (atomicAdd(a.ticket + bh, 1) == a.splits - 1);
    __syncthreads();
    if (!sm.last) return;
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

}  // namespace bloom
