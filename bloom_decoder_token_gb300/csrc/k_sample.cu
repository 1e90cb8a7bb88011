// Per-member temperature + top-p sampling after the LM head; one cluster of
// kSmpCluster CTAs per row, each CTA a contiguous slice of the vocabulary.
//
// "Hugging Face BLOOM Inference Optimization", Webserver Architecture and
// Request Handling: the generation loop applies each batch member's own
// sampling parameters (temperature, top-p).  For a row with logits z,
// temperature t and top-p p (the caller's uniform number u in [0, 1) is the
// draw, so the same inputs give the same token):
//   prob_i proportional to exp((z_i - max z) / t);
//   the nucleus is the shortest prefix of the tokens ordered by probability,
//   highest first (equal logits: lower index first), whose mass reaches p;
//   the token is where the nucleus's cumulative mass, taken in vocabulary
//   order, first exceeds u times the nucleus mass.
// t <= 0 (or not a number) is greedy: the argmax, lowest index on ties.
//
// The masses are fixed point: m_i = floor(exp(-(max z - z_i) / t) * 2^40)
// (float32; 0 once the exponent passes 27, where it is below 2^-38), summed
// in 64-bit integers, so every sum, cut and comparison is exact and
// independent of the summation order: the same logits give the same token on
// every run.  The nucleus cut (the logit t* of its last token) is found by
// narrowing:
//  1. a 2048-bin histogram of mass over d_i = (max z - z_i) / t,
//     spread over the row's own range of d, and the bin where the cumulative
//     mass (bins in order of d) reaches ceil(p * total);
//  2. if that bin holds more than kSmpCand tokens: a second 2048-bin histogram
//     over the order-preserving keys of its logits, and the sub-bin where the
//     mass is reached (a bin of one logit value is the cut at once);
//  3. the region's tokens sorted by (logit desc, index asc) in the first CTA's
//     shared memory and scanned to the cut -- or, for a region of more than
//     kSmpCand tokens (only heavy repetition of a few logit values), a
//     bisection over its key range;
//  4. the tokens with logit t* enter in index order, as many as the mass still
//     missing needs.
// A last pass over contiguous index chunks scans the nucleus masses in
// vocabulary order (block scans in thread order, then over the cluster in
// rank order) and the thread holding the sampled position walks its chunk to
// the token.  Every histogram, total and scan is combined across the cluster
// through distributed shared memory, in rank order.
#include <math.h>
#include <stdint.h>

#include "common.cuh"
#include "kernels.h"

namespace bloom {

constexpr int kSmpCluster = 8;                 // CTAs per row
constexpr int kSmpThreads = 512;
constexpr int kSmpWarps = kSmpThreads / 32;
constexpr int kSmpBins = 2048;
constexpr int kSmpCand = 4096;                 // region tokens sorted in shared memory
constexpr float kSmpScale = 1099511627776.f;   // 2^40: fixed-point unit of mass
constexpr float kSmpDmax = 27.f;               // d beyond this: mass 0 (exp(-27) * 2^40 > 2)
constexpr int kSmpXch = 16;                    // exchange slots (u64) per CTA

struct SmpSmem {
    unsigned long long hmass[kSmpBins];        // this CTA's histogram
    unsigned long long hsum[kSmpBins];         // the cluster's
    unsigned long long cand[kSmpCand];         // (~key << 32) | index: ascending = key desc, index asc
    unsigned long long wsum[kSmpWarps];
    unsigned long long xch[kSmpXch];           // values the peers read
    float wmax[kSmpWarps], wmin[kSmpWarps];
    int widx[kSmpWarps];
    unsigned long long bcast[4];
    int ibcast[4];
    unsigned int ncand;
};

// ---- cluster helpers
__device__ __forceinline__ void smp_cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t smp_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t smp_map(const void *p, uint32_t rank) {
    const uint32_t local = (uint32_t)__cvta_generic_to_shared(p);
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}
__device__ __forceinline__ unsigned long long smp_ld64(uint32_t a) {
    unsigned long long v;
    asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(a) : "memory");
    return v;
}
__device__ __forceinline__ unsigned int smp_ld32(uint32_t a) {
    unsigned int v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
    return v;
}
__device__ __forceinline__ void smp_st64(uint32_t a, unsigned long long v) {
    asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(a), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned int smp_atom_add(uint32_t a, unsigned int v) {
    unsigned int old;
    asm volatile("atom.shared::cluster.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(a), "r"(v) : "memory");
    return old;
}

// order-preserving key of a float (NaN never reaches it)
__device__ __forceinline__ uint32_t smp_key(float f) {
    const uint32_t b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float smp_unkey(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// d = (max z - z) / t of one logit (as a product with 1 / t), its first-level
// bin (inv = bins per unit of d) and its fixed-point mass; NaN and -inf logits,
// and d >= kSmpDmax, take mass 0 (every other mass is at least 2).
__device__ __forceinline__ float smp_d(float z, float zmax, float rt) { return (zmax - z) * rt; }
__device__ __forceinline__ unsigned long long smp_mass(float z, float zmax, float rt, float inv,
                                                       int &bin) {
    const float d = smp_d(z, zmax, rt);
    if (!(d < kSmpDmax)) {
        bin = kSmpBins - 1;
        return 0ull;
    }
    bin = min(kSmpBins - 1, (int)(d * inv));
    return (unsigned long long)(exp2f(-d * 1.4426950408889634f) * kSmpScale);
}
// whether a logit carries mass, and its bin (no exponential)
__device__ __forceinline__ bool smp_live(float z, float zmax, float rt, float inv, int &bin) {
    const float d = smp_d(z, zmax, rt);
    const bool live = d < kSmpDmax;
    bin = live ? min(kSmpBins - 1, (int)(d * inv)) : kSmpBins - 1;
    return live;
}

// Calls f(i, z[i]) for this thread's indices of [s0, s1) (i = s0 + tid, then
// steps of kSmpThreads, ascending), eight loads in flight at a time.
template <typename F>
__device__ __forceinline__ void smp_each(const float *z, int s0, int s1, F &&f) {
    for (int i0 = s0 + (int)threadIdx.x; i0 < s1; i0 += 8 * kSmpThreads) {
        float v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int i = i0 + k * kSmpThreads;
            v[k] = i < s1 ? z[i] : 0.f;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int i = i0 + k * kSmpThreads;
            if (i < s1) f(i, v[k]);
        }
    }
}
// The same over this thread's contiguous chunk [c0, c1), in index order.
template <typename F>
__device__ __forceinline__ void smp_chunk(const float *z, int c0, int c1, F &&f) {
    for (int i0 = c0; i0 < c1; i0 += 8) {
        float v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = i0 + k < c1 ? z[i0 + k] : 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k)
            if (i0 + k < c1) f(i0 + k, v[k]);
    }
}

// Exclusive scan of one 64-bit value per thread in thread order; every thread
// gets its prefix, `total` the sum.  Contains barriers.
__device__ __forceinline__ unsigned long long smp_scan(unsigned long long v, SmpSmem &sm,
                                                       unsigned long long &total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned long long x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    __syncthreads();   // wsum may still be read by a previous call
    if (lane == 31) sm.wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
        unsigned long long w = lane < kSmpWarps ? sm.wsum[lane] : 0ull;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < kSmpWarps) sm.wsum[lane] = w;   // inclusive
    }
    __syncthreads();
    total = sm.wsum[kSmpWarps - 1];
    return (warp ? sm.wsum[warp - 1] : 0ull) + x - v;
}

// Cluster-wide exclusive prefix (in rank order) and total of one value per CTA
// (the value of thread 0), through exchange slot `slot`: every slot is written
// once per launch.  Contains a cluster barrier.
__device__ __forceinline__ unsigned long long smp_cluster_scan(unsigned long long v, int slot,
                                                               SmpSmem &sm, uint32_t rank,
                                                               unsigned long long &total) {
    if (threadIdx.x == 0) sm.xch[slot] = v;
    smp_cluster_sync();
    unsigned long long pre = 0ull, tot = 0ull;
#pragma unroll
    for (int r = 0; r < kSmpCluster; ++r) {
        const unsigned long long x = smp_ld64(smp_map(&sm.xch[slot], (uint32_t)r));
        if ((uint32_t)r < rank) pre += x;
        tot += x;
    }
    total = tot;
    return pre;
}

// Combines one value per CTA (thread 0's) over the cluster through exchange
// slot `slot` (written once per launch): max (op 0) or min (op 1) of u64.
// Contains a cluster barrier.
__device__ __forceinline__ unsigned long long smp_cluster_combine(unsigned long long v, int slot,
                                                                  int op, SmpSmem &sm) {
    if (threadIdx.x == 0) sm.xch[slot] = v;
    smp_cluster_sync();
    unsigned long long r = op == 0 ? 0ull : ~0ull;
#pragma unroll
    for (int k = 0; k < kSmpCluster; ++k) {
        const unsigned long long x = smp_ld64(smp_map(&sm.xch[slot], (uint32_t)k));
        r = op == 0 ? (x > r ? x : r) : (x < r ? x : r);
    }
    return r;
}

// The cluster's histogram: every rank's hmass summed in rank order into hsum.
// The caller has synchronised the cluster after the histograms were built.
__device__ __forceinline__ void smp_merge(SmpSmem &sm) {
    for (int bin = threadIdx.x; bin < kSmpBins; bin += kSmpThreads) {
        unsigned long long m = 0ull;
#pragma unroll
        for (int r = 0; r < kSmpCluster; ++r) m += smp_ld64(smp_map(&sm.hmass[bin], (uint32_t)r));
        sm.hsum[bin] = m;
    }
    __syncthreads();
}

// In the merged histogram: the bin where the cumulative mass (bins in index
// order) reaches `target` (1 .. the total), and the mass before it; each
// thread takes kSmpBins / kSmpThreads consecutive bins.  Contains barriers.
__device__ __forceinline__ void smp_select(unsigned long long target, SmpSmem &sm, int &bin,
                                           unsigned long long &before) {
    constexpr int BPT = kSmpBins / kSmpThreads;
    const int b0 = threadIdx.x * BPT;
    unsigned long long mine = 0ull;
#pragma unroll
    for (int k = 0; k < BPT; ++k) mine += sm.hsum[b0 + k];
    unsigned long long tot;
    unsigned long long run = smp_scan(mine, sm, tot);
    if (run < target && run + mine >= target) {
#pragma unroll
        for (int k = 0; k < BPT; ++k) {
            const unsigned long long m = sm.hsum[b0 + k];
            if (run < target && run + m >= target) {
                sm.ibcast[0] = b0 + k;
                sm.bcast[0] = run;
            }
            run += m;
        }
    }
    __syncthreads();
    bin = sm.ibcast[0];
    before = sm.bcast[0];
}

// Zeroes this CTA's histogram.  Contains a barrier.
__device__ __forceinline__ void smp_clear(SmpSmem &sm) {
    for (int i = threadIdx.x; i < kSmpBins; i += kSmpThreads) sm.hmass[i] = 0ull;
    __syncthreads();
}

__global__ void __launch_bounds__(kSmpThreads) sample_kernel(const SampleArgs a) {
    extern __shared__ __align__(16) unsigned char smp_raw[];
    SmpSmem &sm = *reinterpret_cast<SmpSmem *>(smp_raw);
    griddep_launch();
    griddep_wait();   // the logits come from the previous kernel
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t rank = smp_rank();
    const int b = blockIdx.y;
    if (a.active && !a.active[b]) {   // an idle row of a dynamic batch (the whole cluster)
        if (rank == 0 && tid == 0) a.out[b] = -1;
        return;
    }
    const int V = a.V;
    const int per = (V + kSmpCluster - 1) / kSmpCluster;
    const int s0 = min(V, (int)rank * per), s1 = min(V, s0 + per);   // this CTA's slice
    const float *z = a.logits + (size_t)b * a.ld;
    if (tid == 0) sm.ncand = 0u;   // the first CTA's candidate counter (ordered by the next cluster barrier)

    // ---- maximum (lowest index on ties) and minimum over the row
    float mx = -INFINITY, mn = INFINITY;
    int mi = 0x7fffffff;
    smp_each(z, s0, s1, [&](int i, float v) {
        if (v > mx) {   // NaN never wins; i ascends, so a thread keeps its lowest index
            mx = v;
            mi = i;
        }
        if (v < mn) mn = v;
    });
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, mx, o);
        const int oi = __shfl_xor_sync(0xffffffffu, mi, o);
        if (ov > mx || (ov == mx && oi < mi)) {
            mx = ov;
            mi = oi;
        }
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    }
    if (lane == 0) {
        sm.wmax[warp] = mx;
        sm.widx[warp] = mi;
        sm.wmin[warp] = mn;
    }
    __syncthreads();
    mx = sm.wmax[0];
    mi = sm.widx[0];
    mn = sm.wmin[0];
    for (int w = 1; w < kSmpWarps; ++w) {
        if (sm.wmax[w] > mx || (sm.wmax[w] == mx && sm.widx[w] < mi)) {
            mx = sm.wmax[w];
            mi = sm.widx[w];
        }
        mn = fminf(mn, sm.wmin[w]);
    }
    {
        // larger logit first, then the lower index: (key << 32) | ~index, maximised
        const unsigned long long pk =
            ((unsigned long long)smp_key(mx) << 32) | (unsigned int)(0xffffffffu - (unsigned int)mi);
        const unsigned long long best = smp_cluster_combine(pk, 0, 0, sm);
        const unsigned long long low = smp_cluster_combine(smp_key(mn), 1, 1, sm);
        mx = smp_unkey((uint32_t)(best >> 32));
        mi = (int)(0xffffffffu - (uint32_t)best);
        mn = smp_unkey((uint32_t)low);
    }
    const float t = a.temperature[b];
    const bool greedy = !(t > 0.f) || !(mx > -INFINITY) || mx == INFINITY;
    if (greedy) {   // greedy (or nothing to sample)
        if (rank == 0 && tid == 0) a.out[b] = mi == 0x7fffffff ? 0 : mi;
        smp_cluster_sync();   // no CTA leaves while a peer may still read its exchange slots
        return;
    }
    const float tp = a.top_p[b];
    float u = a.u[b];
    if (!(u >= 0.f)) u = 0.f;
    const float rt = 1.f / t;
    // first-level bins spread over the row's range of d (at most kSmpDmax)
    const float span = fminf(kSmpDmax, (mx - mn) * rt);
    const float inv = span > 0.f ? (float)kSmpBins / span : 0.f;

    // ---- first-level histogram of the slice, merged over the cluster
    smp_clear(sm);
    smp_each(z, s0, s1, [&](int i, float v) {
        int bin;
        const unsigned long long q = smp_mass(v, mx, rt, inv, bin);
        if (q) atomicAdd(&sm.hmass[bin], q);
    });
    __syncthreads();
    smp_cluster_sync();
    smp_merge(sm);
    // total mass Q (> 0: the maximum has mass 2^40) and the target ceil(p * Q)
    unsigned long long Q;
    {
        unsigned long long mine = 0ull;
        for (int k = tid; k < kSmpBins; k += kSmpThreads) mine += sm.hsum[k];
        smp_scan(mine, sm, Q);
    }
    unsigned long long target = Q;
    if (tp < 1.f) {
        const double want = ceil((double)(tp > 0.f ? tp : 0.f) * (double)Q);
        target = want < 1.0 ? 1ull : (unsigned long long)want;
        if (target > Q) target = Q;
    }
    int b1;
    unsigned long long above1;
    smp_select(target, sm, b1, above1);
    // tokens in bin b1 (a pass without atomics, summed over the block and the cluster)
    unsigned long long n1;
    {
        unsigned long long c = 0ull;
        smp_each(z, s0, s1, [&](int i, float v) {
            int bin;
            if (smp_live(v, mx, rt, inv, bin) && bin == b1) ++c;
        });
        unsigned long long cta;
        smp_scan(c, sm, cta);
        smp_cluster_scan(cta, 4, sm, rank, n1);
    }

    // ---- the region of the cut: bin b1, or one of its second-level sub-bins
    bool level2 = false;
    unsigned long long base = above1;      // mass of the tokens above the region
    unsigned long long nreg = n1;
    uint32_t rlo = 0u, rhi = 0xffffffffu;  // key bounds of a second-level region
    uint32_t tkey = 0u;
    unsigned long long mass_gt = 0ull;
    bool cut_found = false;
    if (n1 > (unsigned long long)kSmpCand) {
        uint32_t lo = 0xffffffffu, hi = 0u;
        smp_each(z, s0, s1, [&](int i, float v) {
            int bin;
            if (smp_live(v, mx, rt, inv, bin) && bin == b1) {
                const uint32_t k = smp_key(v);
                lo = min(lo, k);
                hi = max(hi, k);
            }
        });
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
            hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
        }
        if (lane == 0) sm.wsum[warp] = ((unsigned long long)hi << 32) | lo;
        __syncthreads();
        lo = 0xffffffffu;
        hi = 0u;
        for (int w = 0; w < kSmpWarps; ++w) {
            lo = min(lo, (uint32_t)sm.wsum[w]);
            hi = max(hi, (uint32_t)(sm.wsum[w] >> 32));
        }
        const uint32_t kmin = (uint32_t)smp_cluster_combine(lo, 2, 1, sm);
        const uint32_t kmax = (uint32_t)smp_cluster_combine(hi, 3, 0, sm);
        if (kmin == kmax) {   // one logit value: the cut is there
            tkey = kmin;
            mass_gt = above1;
            cut_found = true;
        } else {
            level2 = true;
            const unsigned long long range = (unsigned long long)(kmax - kmin) + 1ull;
            smp_clear(sm);   // every peer finished merging the first level (cluster barriers since)
            smp_each(z, s0, s1, [&](int i, float v) {
                    int bin;
                const unsigned long long q = smp_mass(v, mx, rt, inv, bin);
                if (q && bin == b1) {
                    // sub-bins in descending key order, so that the walk runs from the top
                    const int sb = kSmpBins - 1 -
                                   (int)((unsigned long long)(smp_key(v) - kmin) * kSmpBins / range);
                    atomicAdd(&sm.hmass[sb], q);
                }
            });
            __syncthreads();
            smp_cluster_sync();
            smp_merge(sm);
            int b2;
            unsigned long long above2;
            smp_select(target - above1, sm, b2, above2);
            const int s2 = kSmpBins - 1 - b2;
            base = above1 + above2;
            // the keys k of sub-bin s2: floor((k - kmin) * 2048 / range) == s2
            rlo = kmin + (uint32_t)(((unsigned long long)s2 * range + kSmpBins - 1) / kSmpBins);
            rhi = kmin + (uint32_t)(((unsigned long long)(s2 + 1) * range + kSmpBins - 1) / kSmpBins) - 1u;
            unsigned long long c = 0ull;
            smp_each(z, s0, s1, [&](int i, float v) {
                    int bin;
                if (smp_live(v, mx, rt, inv, bin) && bin == b1) {
                    const uint32_t k = smp_key(v);
                    c += (k >= rlo && k <= rhi) ? 1ull : 0ull;
                }
            });
            unsigned long long cta;
            smp_scan(c, sm, cta);
            smp_cluster_scan(cta, 5, sm, rank, nreg);
        }
    }
    auto in_region = [&](float v, int bin) {
        if (bin != b1) return false;
        if (!level2) return true;
        const uint32_t k = smp_key(v);
        return k >= rlo && k <= rhi;
    };
    if (!cut_found) {
        const unsigned long long need = target - base;   // 1 .. the region's mass
        if (nreg <= (unsigned long long)kSmpCand) {
            // ---- the region gathered in the first CTA, sorted by (logit desc,
            // index asc) and scanned to the cut
            const uint32_t cnt0 = smp_map(&sm.ncand, 0u);
            smp_each(z, s0, s1, [&](int i, float v) {
                    int bin;
                if (smp_live(v, mx, rt, inv, bin) && in_region(v, bin)) {
                    const unsigned int slot = smp_atom_add(cnt0, 1u);
                    if (slot < (unsigned int)kSmpCand)
                        smp_st64(smp_map(&sm.cand[slot], 0u),
                                 ((unsigned long long)(~smp_key(v)) << 32) | (unsigned int)i);
                }
            });
            smp_cluster_sync();
            if (rank == 0) {
                const int n = (int)min(sm.ncand, (unsigned int)kSmpCand);
                int np = 1;
                while (np < n) np <<= 1;
                for (int j = n + tid; j < np; j += kSmpThreads) sm.cand[j] = ~0ull;
                __syncthreads();
                for (int k = 2; k <= np; k <<= 1)   // bitonic sort, ascending
                    for (int jj = k >> 1; jj > 0; jj >>= 1) {
                        for (int x = tid; x < np; x += kSmpThreads) {
                            const int y = x ^ jj;
                            if (y > x) {
                                const unsigned long long p0 = sm.cand[x], p1 = sm.cand[y];
                                if ((p0 > p1) == ((x & k) == 0)) {
                                    sm.cand[x] = p1;
                                    sm.cand[y] = p0;
                                }
                            }
                        }
                        __syncthreads();
                    }
                constexpr int E = kSmpCand / kSmpThreads;
                unsigned long long qs[E], loc = 0ull;
                uint32_t ks[E];
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const int j = tid * E + e;
                    qs[e] = 0ull;
                    ks[e] = 0u;
                    if (j < n) {
                        ks[e] = ~(uint32_t)(sm.cand[j] >> 32);
                        int bin;
                        qs[e] = smp_mass(smp_unkey(ks[e]), mx, rt, inv, bin);
                    }
                    loc += qs[e];
                }
                unsigned long long tot;
                const unsigned long long pre = smp_scan(loc, sm, tot);
                // the first entry whose inclusive cumulative mass reaches `need`
                unsigned long long run = pre;
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const int j = tid * E + e;
                    if (j < n && run < need && run + qs[e] >= need) sm.ibcast[1] = j;
                    run += qs[e];
                }
                __syncthreads();
                const uint32_t tk = ~(uint32_t)(sm.cand[sm.ibcast[1]] >> 32);
                // the first entry with that logit, and the region's mass before it
                run = pre;
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const int j = tid * E + e;
                    if (j < n && ks[e] == tk && (j == 0 || ~(uint32_t)(sm.cand[j - 1] >> 32) != tk))
                        sm.bcast[1] = run;
                    run += qs[e];
                }
                __syncthreads();
                if (tid == 0) {
                    sm.xch[8] = tk;
                    sm.xch[9] = sm.bcast[1];
                }
            }
            smp_cluster_sync();
            tkey = (uint32_t)smp_ld64(smp_map(&sm.xch[8], 0u));
            mass_gt = base + smp_ld64(smp_map(&sm.xch[9], 0u));
        } else {
            // ---- a region of few repeated logit values: bisection over its keys for
            // the largest K with mass(region, key >= K) >= need
            unsigned long long lo = rlo, hi = (unsigned long long)rhi + 1ull, m_hi = 0ull;
            int it = 0;
            while (hi - lo > 1ull) {
                const unsigned long long mid = (lo + hi) >> 1;
                unsigned long long part = 0ull;
                smp_each(z, s0, s1, [&](int i, float v) {
                            int bin;
                    const unsigned long long q = smp_mass(v, mx, rt, inv, bin);
                    if (q && in_region(v, bin) && (unsigned long long)smp_key(v) >= mid) part += q;
                });
                unsigned long long cta;
                smp_scan(part, sm, cta);
                unsigned long long mm;
                smp_cluster_scan(cta, 10 + (it & 1), sm, rank, mm);
                if (mm >= need) {
                    lo = mid;
                } else {
                    hi = mid;
                    m_hi = mm;
                }
                ++it;
            }
            tkey = (uint32_t)lo;
            mass_gt = base + m_hi;
        }
    }
    int bin_t;
    const unsigned long long qt = smp_mass(smp_unkey(tkey), mx, rt, inv, bin_t);   // > 0
    // tokens with logit t* taken in index order: the fewest that reach the target
    const unsigned long long kties = (target - mass_gt + qt - 1ull) / qt;

    // ---- inverse cumulative mass over the nucleus in vocabulary order: this
    // thread's contiguous chunk of the slice, offsets by block and cluster scans
    const int chunk = (s1 - s0 + kSmpThreads - 1) / kSmpThreads;
    const int c0 = min(s1, s0 + tid * chunk), c1 = min(s1, c0 + chunk);
    unsigned long long gt = 0ull, nt = 0ull;
    smp_chunk(z, c0, c1, [&](int i, float v) {
        if (!(v == v)) return;
        const uint32_t k = smp_key(v);
        if (k > tkey) {
            int bin;
            gt += smp_mass(v, mx, rt, inv, bin);
        } else if (k == tkey) {
            ++nt;
        }
    });
    unsigned long long tie_cta, tie_all, mass_cta, Mn;
    const unsigned long long tie_in = smp_scan(nt, sm, tie_cta);
    const unsigned long long tie0 = smp_cluster_scan(tie_cta, 12, sm, rank, tie_all) + tie_in;
    const unsigned long long inc = tie0 >= kties ? 0ull : (kties - tie0 < nt ? kties - tie0 : nt);
    const unsigned long long mym = gt + inc * qt;
    const unsigned long long m_in = smp_scan(mym, sm, mass_cta);
    const unsigned long long start = smp_cluster_scan(mass_cta, 13, sm, rank, Mn) + m_in;
    unsigned long long s = (unsigned long long)floor((double)u * (double)Mn);
    if (s >= Mn) s = Mn - 1ull;
    if (start <= s && s < start + mym) {
        unsigned long long cum = start, tr = tie0;
        int tok = c1 - 1;
        for (int i = c0; i < c1; ++i) {
            const float v = z[i];
            if (!(v == v)) continue;
            const uint32_t k = smp_key(v);
            unsigned long long q = 0ull;
            if (k > tkey) {
                int bin;
                q = smp_mass(v, mx, rt, inv, bin);
            } else if (k == tkey) {
                q = tr < kties ? qt : 0ull;
                ++tr;
            }
            cum += q;
            if (q && cum > s) {
                tok = i;
                break;
            }
        }
        a.out[b] = tok;
    }
    smp_cluster_sync();   // no CTA leaves while a peer may still read its shared memory
}

cudaError_t launch_sample(const SampleArgs &a, cudaStream_t s) {
    if (a.B <= 0) return cudaSuccess;
    if (a.V <= 0 || a.ld < a.V || a.B > 65535) return cudaErrorInvalidValue;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(sample_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)sizeof(SmpSmem));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kSmpCluster, (unsigned)a.B);
    cfg.blockDim = dim3(kSmpThreads);
    cfg.dynamicSmemBytes = sizeof(SmpSmem);
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = g_pdl ? 1 : 0;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = kSmpCluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, sample_kernel, a);
}

}  // namespace bloom
