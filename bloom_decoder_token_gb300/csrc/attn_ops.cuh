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
// kAttnKeysPerGroup keys in flight per group; lane `sub` of a group owns d/8
// elements of q and of the accumulator, so a key costs one 3-step shuffle for
// the dot product and no other communication.  Groups merge by shuffles, warps
// through shared memory, and the last block of a (sequence, head) to finish
// merges the split partials by rescaling with exp(m_split - m_max) -- no second
// pass and no waiting.
//
// The launch fixes an upper bound on the split count (the graph of a decode
// step is captured once for every length); a block derives the split count it
// uses from the live key count, at least kAttnMinKeysPerSplit keys a split, and
// blocks beyond it return at once.
//
// Two bodies share the per-round arithmetic (attn_round) and the merge
// (attn_finish), so they give the same bits: attn_decode_block loads each
// round's K / V rows into registers; attn_decode_block_bulk (64-thread blocks
// over a cache in device memory) stages them in shared memory by bulk copies
// three rounds ahead.
#pragma once

#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_ops.cuh"

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

constexpr int kAttnKeysPerGroup = 2;       // keys in flight per 8-lane group
constexpr int kAttnMinKeysPerSplit = 32;   // a split takes at least this many keys

template <int D, int NT>
struct AttnSmem {
    float m[NT / 32], l[NT / 32];
    float acc[NT / 32][D];
    int last;
};

// One round of a group's online softmax over its KPG keys (live, positions pk,
// K rows kv, V rows vv; lane `sub` holds elements [sub * EPT, (sub + 1) * EPT)):
// the scores, then the running max, sum and accumulator rescaled and updated.
template <int EPT, int KPG>
__device__ __forceinline__ void attn_round(const uint4 (&qv)[EPT / 8], const bool (&live)[KPG],
                                           const int (&pk)[KPG], const uint4 (&kv)[KPG][EPT / 8],
                                           const uint4 (&vv)[KPG][EPT / 8], float scale, float slope,
                                           float &m_run, float &l_run, float (&acc)[EPT]) {
    float sc[KPG];
#pragma unroll
    for (int u = 0; u < KPG; ++u) {
        float d = 0.f;
        if (live[u]) {
#pragma unroll
            for (int i = 0; i < EPT / 8; ++i) {
                float f[8], qq[8];
                unpack8(kv[u][i], f);
                unpack8(qv[i], qq);
#pragma unroll
                for (int e = 0; e < 8; ++e) d = fmaf(qq[e], f[e], d);
            }
        }
#pragma unroll
        for (int o = 4; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
        sc[u] = (live[u] && pk[u] >= 0) ? fmaf(d, scale, slope * (float)pk[u]) : -INFINITY;
    }
    float m_new = m_run;
#pragma unroll
    for (int u = 0; u < KPG; ++u) m_new = fmaxf(m_new, sc[u]);
    if (m_new == -INFINITY) return;   // uniform within the group
    const float corr = (m_run == -INFINITY) ? 0.f : expf(m_run - m_new);
    float wt[KPG];
    l_run *= corr;
#pragma unroll
    for (int u = 0; u < KPG; ++u) {
        wt[u] = (sc[u] == -INFINITY) ? 0.f : expf(sc[u] - m_new);
        l_run += wt[u];
    }
#pragma unroll
    for (int e = 0; e < EPT; ++e) acc[e] *= corr;
#pragma unroll
    for (int u = 0; u < KPG; ++u) {
        if (wt[u] == 0.f) continue;   // masked or absent key: adds exactly nothing
#pragma unroll
        for (int i = 0; i < EPT / 8; ++i) {
            float f[8];
            unpack8(vv[u][i], f);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[8 * i + e] = fmaf(wt[u], f[e], acc[8 * i + e]);
        }
    }
    m_run = m_new;
}

// The block's result from every thread's (m, l, accumulator): the groups of a
// warp merged by shuffles, the warps through shared memory (sm.m, sm.l, sm.acc),
// then o written (one split) or the split partial stored and the last block of
// the (sequence, head) merging the partials (a ticket, no waiting).
template <int D, int NT, class SM>
__device__ __forceinline__ void attn_finish(const AttnDecodeArgs &a, int split, int splits, int j,
                                            int b, size_t bh, float m_run, float l_run,
                                            float (&acc)[D / 8], SM &sm) {
    constexpr int EPT = D / 8;
    constexpr int NW = NT / 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, sub = tid & 7;
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
    // column c of the block's output: the warps' accumulators rescaled to the block maximum
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, sm.m[w]);
    float L = 0.f, wg[NW];
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        wg[w] = 0.f;
        if (M == -INFINITY || sm.m[w] == -INFINITY) continue;
        wg[w] = expf(sm.m[w] - M);
        L = fmaf(sm.l[w], wg[w], L);
    }
    auto col = [&](int c) {
        float A = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w)
            if (wg[w] != 0.f) A = fmaf(sm.acc[w][c], wg[w], A);
        return A;
    };
    if (splits == 1) {
        for (int c = tid; c < D; c += NT)
            a.o[(size_t)b * a.n * D + (size_t)j * D + c] = f2bf(L > 0.f ? col(c) / L : 0.f);
        return;
    }
    float *part = a.part + (bh * a.splits + split) * (D + 2);
    for (int c = tid; c < D; c += NT) part[2 + c] = col(c);
    if (tid == 0) {
        part[0] = M;
        part[1] = L;
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) sm.last = (atomicAdd(a.ticket + bh, 1) == splits - 1);
    __syncthreads();
    if (!sm.last) return;
    __threadfence();
    const float *pb = a.part + bh * a.splits * (D + 2);
    float Mx = -INFINITY;
    for (int sp = 0; sp < splits; ++sp) Mx = fmaxf(Mx, __ldcg(pb + sp * (D + 2)));
    for (int c = tid; c < D; c += NT) {
        float Ls = 0.f, As = 0.f;
        if (Mx != -INFINITY) {
            for (int sp = 0; sp < splits; ++sp) {
                const float ms = __ldcg(pb + sp * (D + 2));
                if (ms == -INFINITY) continue;
                const float wgt = expf(ms - Mx);
                Ls = fmaf(__ldcg(pb + sp * (D + 2) + 1), wgt, Ls);
                As = fmaf(__ldcg(pb + sp * (D + 2) + 2 + c), wgt, As);
            }
        }
        a.o[(size_t)b * a.n * D + (size_t)j * D + c] = f2bf(Ls > 0.f ? As / Ls : 0.f);
    }
    if (tid == 0) a.ticket[bh] = 0;
}

// All NT threads of the block call it with the same (split, j, b).  Contains
// barriers; the first one also protects `sm` from a previous call's readers.
// It waits for the previous kernel itself (griddepcontrol.wait): with a.early
// the length, the activity and the K / V / positions of the keys that earlier
// steps cached (slots below the length) are read first, so that the first
// round's loads overlap the QKV kernel that is still appending this step's key.
template <int D, int NT>
__device__ __forceinline__ void attn_decode_block(const AttnDecodeArgs &a, int split, int j, int b,
                                                  AttnSmem<D, NT> &sm) {
    constexpr int EPT = D / 8;             // elements per lane of an 8-lane group
    constexpr int NW = NT / 32;
    constexpr int NG = NT / 8;             // groups; a round covers kAttnKeysPerGroup * NG keys
    constexpr int KPG = kAttnKeysPerGroup;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int grp = tid >> 3, sub = tid & 7;
    if (!a.early) griddep_wait();
    // keys [0, len] with the step's new one; an idle row appended none
    const int len = a.len_ptr ? a.len_ptr[b] : a.len_host;
    const int nk = min(len + ((!a.len_ptr || !a.active || a.active[b]) ? 1 : 0), a.max_seq);
    int chunk = (nk + a.splits - 1) / a.splits;
    if (chunk < kAttnMinKeysPerSplit) chunk = kAttnMinKeysPerSplit;
    const int splits = nk > 0 ? (nk + chunk - 1) / chunk : 1;   // uniform over the blocks of (b, j)
    if (split >= splits) return;
    const int k0 = split * chunk;
    const int k1 = min(nk, k0 + chunk);

    const size_t bh = (size_t)b * a.n + j;
    const uint16_t *kbase = a.k + bh * a.max_seq * D + sub * EPT;
    const uint16_t *vbase = a.v + bh * a.max_seq * D + sub * EPT;
    const int *posb = a.pos + (size_t)b * a.max_seq;
    const float slope = a.slopes[j];

    bool live[KPG], have[KPG];
    int pk[KPG];
    uint4 kv[KPG][EPT / 8], vv[KPG][EPT / 8];
    auto load_key = [&](int u, int key) {
        pk[u] = posb[key];
#pragma unroll
        for (int i = 0; i < EPT / 8; ++i) {
            kv[u][i] = *reinterpret_cast<const uint4 *>(kbase + (size_t)key * D + 8 * i);
            vv[u][i] = *reinterpret_cast<const uint4 *>(vbase + (size_t)key * D + 8 * i);
        }
    };
#pragma unroll
    for (int u = 0; u < KPG; ++u) {
        const int key = k0 + u * NG + grp;   // round 0
        have[u] = a.early && key < k1 && key < len;
        if (have[u]) load_key(u, key);
    }
    if (a.early) griddep_wait();   // q, and the new key's K / V / position, come from this step

    // q stays packed bf16 (widened per use, exact); the scale multiplies the dot product
    uint4 qv[EPT / 8];
    float acc[EPT];
    {
        const uint16_t *qp = a.q + bh * D + sub * EPT;
#pragma unroll
        for (int i = 0; i < EPT / 8; ++i) qv[i] = *reinterpret_cast<const uint4 *>(qp + 8 * i);
#pragma unroll
        for (int e = 0; e < EPT; ++e) acc[e] = 0.f;
    }
    float m_run = -INFINITY, l_run = 0.f;
    const int rounds = (k1 - k0 + KPG * NG - 1) / (KPG * NG);
    for (int r = 0; r < rounds; ++r) {
#pragma unroll
        for (int u = 0; u < KPG; ++u) {
            const int key = k0 + (r * KPG + u) * NG + grp;
            live[u] = key < k1;
            if (live[u] && !(r == 0 && have[u])) load_key(u, key);
            if (!live[u]) pk[u] = -1;
        }
        attn_round<EPT, KPG>(qv, live, pk, kv, vv, a.scale, slope, m_run, l_run, acc);
    }
    attn_finish<D, NT>(a, split, splits, j, b, bh, m_run, l_run, acc, sm);
}

// The same block for 64-thread CTAs over a cache in device memory, with the K / V
// rows of each round (16 consecutive keys) staged in shared memory by bulk
// copies (cp.async.bulk, one for the round's K rows and one for its V rows,
// completing on an mbarrier) three rounds ahead, and each lane's key positions
// by cp.async; the keys, rounds, groups and arithmetic are those of
// attn_decode_block, so the two give the same bits.  With a.early the copies of
// the first three rounds' cached keys (below the length) go out before the
// wait for the QKV kernel; the step's new key is read from global memory after
// it.  Every wait is bounded (a.wait_ns; flag 8 on expiry, its keys skipped).
template <int D>
struct AttnSmemBulk {
    static constexpr int kStages = 3, kRoundKeys = 2 * 8;   // KPG keys x 8 groups
    alignas(128) uint16_t k[kStages][kRoundKeys][D];
    alignas(128) uint16_t v[kStages][kRoundKeys][D];
    int pos[kStages][64][2];
    uint64_t bar[kStages];
    float m[2], l[2];
    float acc[2][D];
    int last;
};

template <int D>
__device__ __forceinline__ void attn_decode_block_bulk(const AttnDecodeArgs &a, int split, int j,
                                                       int b, AttnSmemBulk<D> &sm) {
    constexpr int NT = 64, EPT = D / 8, NG = NT / 8, KPG = kAttnKeysPerGroup;
    constexpr int ST = AttnSmemBulk<D>::kStages, RK = AttnSmemBulk<D>::kRoundKeys;
    static_assert(KPG * NG == RK && KPG == 2, "a round is the stage's 16 keys");
    const int tid = threadIdx.x, grp = tid >> 3, sub = tid & 7;
    if (tid == 0) {
        for (int st = 0; st < ST; ++st) tc_mbar_init(&sm.bar[st], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (!a.early) griddep_wait();
    const int len = a.len_ptr ? a.len_ptr[b] : a.len_host;
    const int nk = min(len + ((!a.len_ptr || !a.active || a.active[b]) ? 1 : 0), a.max_seq);
    int chunk = (nk + a.splits - 1) / a.splits;
    if (chunk < kAttnMinKeysPerSplit) chunk = kAttnMinKeysPerSplit;
    const int splits = nk > 0 ? (nk + chunk - 1) / chunk : 1;
    if (split >= splits) return;   // uniform over the block; nothing issued yet
    const int k0 = split * chunk;
    const int k1 = min(nk, k0 + chunk);
    const size_t bh = (size_t)b * a.n + j;
    const uint16_t *krow = a.k + bh * a.max_seq * D;
    const uint16_t *vrow = a.v + bh * a.max_seq * D;
    const int *posb = a.pos + (size_t)b * a.max_seq;
    const float slope = a.slopes[j];
    const int rounds = (k1 - k0 + RK - 1) / RK;
    const unsigned long long lim = a.wait_ns ? a.wait_ns : kTcWaitNs;

    // round r into stage r % ST: its cached keys [lo, hi) (below len) by two bulk
    // copies, and this lane's positions of them; one cp.async group per round
    auto issue = [&](int r) {
        if (r < rounds) {
            const int st = r % ST, lo = k0 + r * RK, hi = min(min(k1, lo + RK), len);
            const uint32_t bar = tc_smem(&sm.bar[st]);
            if (tid == 0) {
                if (hi > lo) {
                    const uint32_t bytes = (uint32_t)(hi - lo) * D * 2;
                    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                                 "r"(2 * bytes)
                                 : "memory");
                    asm volatile(
                        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                            tc_smem(&sm.k[st][0][0])),
                        "l"(krow + (size_t)lo * D), "r"(bytes), "r"(bar)
                        : "memory");
                    asm volatile(
                        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                            tc_smem(&sm.v[st][0][0])),
                        "l"(vrow + (size_t)lo * D), "r"(bytes), "r"(bar)
                        : "memory");
                } else {
                    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
                }
            }
#pragma unroll
            for (int u = 0; u < KPG; ++u) {
                const int key = lo + u * NG + grp;
                if (key < hi)
                    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                                     tc_smem(&sm.pos[st][tid][u])),
                                 "l"(posb + key)
                                 : "memory");
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    for (int r = 0; r < ST; ++r) issue(r);
    if (a.early) griddep_wait();   // q, and the new key's K / V / position, come from this step

    uint4 qv[EPT / 8];
    float acc[EPT];
    {
        const uint16_t *qp = a.q + bh * D + sub * EPT;
#pragma unroll
        for (int i = 0; i < EPT / 8; ++i) qv[i] = *reinterpret_cast<const uint4 *>(qp + 8 * i);
#pragma unroll
        for (int e = 0; e < EPT; ++e) acc[e] = 0.f;
    }
    float m_run = -INFINITY, l_run = 0.f;
    for (int r = 0; r < rounds; ++r) {
        const int st = r % ST, lo = k0 + r * RK;
        asm volatile("cp.async.wait_group 2;" ::: "memory");   // this round's positions
        // the stage's bulk copies; on expiry its staged keys are skipped (flag 8), after
        // a second bounded wait so that no copy still lands once the block moves on
        const uint32_t parity = (uint32_t)((r / ST) & 1);
        const bool okb = tc_mbar_wait(&sm.bar[st], parity, lim);
        if (!okb) {
            if (a.err) atomicOr(a.err, kErrTimeout);
            tc_mbar_wait(&sm.bar[st], parity, kTcWaitNs);
        }
        bool live[KPG];
        int pk[KPG];
        uint4 kv[KPG][EPT / 8], vv[KPG][EPT / 8];
#pragma unroll
        for (int u = 0; u < KPG; ++u) {
            const int key = lo + u * NG + grp;
            live[u] = key < k1 && (okb || key >= len);
            pk[u] = -1;
            if (!live[u]) {
#pragma unroll
                for (int i = 0; i < EPT / 8; ++i) kv[u][i] = vv[u][i] = make_uint4(0u, 0u, 0u, 0u);
            } else if (key < len) {   // staged
                pk[u] = sm.pos[st][tid][u];
#pragma unroll
                for (int i = 0; i < EPT / 8; ++i) {
                    kv[u][i] = *reinterpret_cast<const uint4 *>(&sm.k[st][key - lo][sub * EPT + 8 * i]);
                    vv[u][i] = *reinterpret_cast<const uint4 *>(&sm.v[st][key - lo][sub * EPT + 8 * i]);
                }
            } else {   // the step's new key
                pk[u] = posb[key];
#pragma unroll
                for (int i = 0; i < EPT / 8; ++i) {
                    kv[u][i] = *reinterpret_cast<const uint4 *>(krow + (size_t)key * D + sub * EPT + 8 * i);
                    vv[u][i] = *reinterpret_cast<const uint4 *>(vrow + (size_t)key * D + sub * EPT + 8 * i);
                }
            }
        }
        attn_round<EPT, KPG>(qv, live, pk, kv, vv, a.scale, slope, m_run, l_run, acc);
        __syncthreads();   // every thread is done with stage st
        issue(r + ST);
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    attn_finish<D, NT>(a, split, splits, j, b, bh, m_run, l_run, acc, sm);
}

}  // namespace bloom
