// Per-member temperature + top-p sampling after the LM head, one row per CTA.
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
// every run.  The nucleus cut
// (the logit t* of its last token) is found by narrowing:
//  1. a 2048-bin histogram of mass and count over d_i = (max z - z_i) / t,
//     spread over the row's own range of d, and the bin where the cumulative
//     mass (bins in order of d) reaches ceil(p * total);
//  2. if that bin holds more than kSmpCand tokens: a second 2048-bin histogram
//     over the order-preserving keys of its logits, and the sub-bin where the
//     mass is reached (a bin of one logit value is the cut at once);
//  3. the region's tokens sorted by (logit desc, index asc) in shared memory
//     and scanned to the cut -- or, for a region of more than kSmpCand tokens
//     (only heavy repetition of a few logit values), a bisection over its key
//     range;
//  4. the tokens with logit t* enter in index order, as many as the mass still
//     missing needs.
// A last pass over contiguous index chunks scans the nucleus masses in
// vocabulary order (block scans in thread order) and the thread holding the
// sampled position walks its chunk to the token.
#include <math.h>
#include <stdint.h>

#include "common.cuh"
#include "kernels.h"

namespace bloom {

constexpr int kSmpThreads = 1024;
constexpr int kSmpWarps = kSmpThreads / 32;
constexpr int kSmpBins = 2048;
constexpr int kSmpCand = 4096;                 // bin elements sorted in shared memory
constexpr float kSmpScale = 1099511627776.f;   // 2^40: fixed-point unit of mass
constexpr float kSmpDmax = 27.f;               // d beyond this: mass 0 (exp(-27) * 2^40 > 2)

struct SmpSmem {
    unsigned long long hmass[kSmpBins];
    unsigned int hcount[kSmpBins];
    unsigned long long cand[kSmpCand];         // (~key << 32) | index, ascending = key desc, index asc
    unsigned long long wsum[kSmpWarps];
    float wmax[kSmpWarps], wmin[kSmpWarps];
    int widx[kSmpWarps];
    unsigned long long bcast[4];
    int ibcast[4];
    unsigned int ncand;
};

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
        unsigned long long w = sm.wsum[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        sm.wsum[lane] = w;   // inclusive
    }
    __syncthreads();
    total = sm.wsum[kSmpWarps - 1];
    return (warp ? sm.wsum[warp - 1] : 0ull) + x - v;
}

// Sum of one 64-bit value per thread.  Contains barriers.
__device__ __forceinline__ unsigned long long smp_sum(unsigned long long v, SmpSmem &sm) {
    unsigned long long total;
    smp_scan(v, sm, total);
    return total;
}

// The bin of sm.hmass where the cumulative mass (bins in index order) reaches
// `target` (1 .. the total), and the mass of the bins before it; two bins per
// thread.  Contains barriers.
__device__ __forceinline__ void smp_select(unsigned long long target, SmpSmem &sm, int &bin,
                                           unsigned long long &before) {
    const int tid = threadIdx.x;
    const unsigned long long m0 = sm.hmass[2 * tid], m1 = sm.hmass[2 * tid + 1];
    unsigned long long tot;
    const unsigned long long pre = smp_scan(m0 + m1, sm, tot);
    if (pre < target && pre + m0 + m1 >= target) {
        const bool first = pre + m0 >= target;
        sm.ibcast[0] = first ? 2 * tid : 2 * tid + 1;
        sm.bcast[0] = first ? pre : pre + m0;
    }
    __syncthreads();
    bin = sm.ibcast[0];
    before = sm.bcast[0];
}

// Block-wide minimum and maximum of one 32-bit key per thread.  Contains barriers.
__device__ __forceinline__ void smp_minmax(uint32_t lo, uint32_t hi, SmpSmem &sm, uint32_t &mn,
                                           uint32_t &mxk) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
        hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    __syncthreads();   // the scratch may still be read by a previous call
    if (lane == 0) sm.wsum[warp] = ((unsigned long long)hi << 32) | lo;
    __syncthreads();
    mn = 0xffffffffu;
    mxk = 0u;
    for (int w = 0; w < kSmpWarps; ++w) {
        mn = min(mn, (uint32_t)sm.wsum[w]);
        mxk = max(mxk, (uint32_t)(sm.wsum[w] >> 32));
    }
}

__global__ void __launch_bounds__(kSmpThreads, 1) sample_kernel(const SampleArgs a) {
    extern __shared__ __align__(16) unsigned char smp_raw[];
    SmpSmem &sm = *reinterpret_cast<SmpSmem *>(smp_raw);
    griddep_launch();
    griddep_wait();   // the logits come from the previous kernel
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = blockIdx.x;
    const int V = a.V;
    const float *z = a.logits + (size_t)b * a.ld;
    if (a.active && !a.active[b]) {   // an idle row of a dynamic batch
        if (tid == 0) a.out[b] = -1;
        return;
    }

    // ---- maximum (and its lowest index), minimum
    float mx = -INFINITY, mn = INFINITY;
    int mi = 0x7fffffff;
    for (int i = tid; i < V; i += kSmpThreads) {
        const float v = z[i];
        if (v > mx) {   // NaN never wins; i ascends, so a thread keeps its lowest index
            mx = v;
            mi = i;
        }
        if (v < mn) mn = v;
    }
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
    const float t = a.temperature[b];
    if (!(t > 0.f) || !(mx > -INFINITY) || mx == INFINITY) {   // greedy (or nothing to sample)
        if (tid == 0) a.out[b] = mi == 0x7fffffff ? 0 : mi;
        return;
    }
    const float tp = a.top_p[b];
    float u = a.u[b];
    if (!(u >= 0.f)) u = 0.f;
    // first-level bins spread over the row's range of d (at most kSmpDmax)
    const float rt = 1.f / t;
    const float span = fminf(kSmpDmax, (mx - mn) * rt);
    const float inv = span > 0.f ? (float)kSmpBins / span : 0.f;

    // ---- total mass and the first-level histogram
    for (int i = tid; i < kSmpBins; i += kSmpThreads) {
        sm.hmass[i] = 0ull;
        sm.hcount[i] = 0u;
    }
    __syncthreads();
    unsigned long long mine = 0ull;
    for (int i = tid; i < V; i += kSmpThreads) {
        int bin;
        const unsigned long long q = smp_mass(z[i], mx, rt, inv, bin);
        if (q) {
            mine += q;
            atomicAdd(&sm.hmass[bin], q);
            atomicAdd(&sm.hcount[bin], 1u);
        }
    }
    const unsigned long long Q = smp_sum(mine, sm);   // > 0: the maximum has mass 2^40
    unsigned long long target = Q;
    if (tp < 1.f) {
        const double want = ceil((double)(tp > 0.f ? tp : 0.f) * (double)Q);
        target = want < 1.0 ? 1ull : (unsigned long long)want;
        if (target > Q) target = Q;
    }
    int b1;
    unsigned long long above1;
    smp_select(target, sm, b1, above1);
    const unsigned int n1 = sm.hcount[b1];

    // ---- the region of the cut: bin b1, or one of its second-level sub-bins
    bool level2 = false;
    uint32_t kmin = 0u, krange_m1 = 0u;   // second level: keys kmin .. kmin + krange_m1
    int s2 = 0;                           // the sub-bin (by key, ascending)
    unsigned long long base = above1;     // mass of the tokens above the region
    unsigned int nreg = n1;
    uint32_t rlo = 0u, rhi = 0xffffffffu; // key bounds of the region (second level)
    uint32_t tkey = 0u;
    unsigned long long mass_gt = 0ull;
    bool cut_found = false;
    if (n1 > (unsigned int)kSmpCand) {
        uint32_t lo = 0xffffffffu, hi = 0u;
        for (int i = tid; i < V; i += kSmpThreads) {
            const float v = z[i];
            int bin;
            if (smp_live(v, mx, rt, inv, bin) && bin == b1) {
                const uint32_t k = smp_key(v);
                lo = min(lo, k);
                hi = max(hi, k);
            }
        }
        uint32_t kmax;
        smp_minmax(lo, hi, sm, kmin, kmax);
        if (kmin == kmax) {   // one logit value: the cut is there
            tkey = kmin;
            mass_gt = above1;
            cut_found = true;
        } else {
            level2 = true;
            krange_m1 = kmax - kmin;
            const unsigned long long range = (unsigned long long)krange_m1 + 1ull;
            __syncthreads();
            for (int i = tid; i < kSmpBins; i += kSmpThreads) {
                sm.hmass[i] = 0ull;
                sm.hcount[i] = 0u;
            }
            __syncthreads();
            for (int i = tid; i < V; i += kSmpThreads) {
                const float v = z[i];
                int bin;
                const unsigned long long q = smp_mass(v, mx, rt, inv, bin);
                if (q && bin == b1) {
                    // sub-bins in descending key order, so that the walk runs from the top
                    const int sb = kSmpBins - 1 -
                                   (int)((unsigned long long)(smp_key(v) - kmin) * kSmpBins / range);
                    atomicAdd(&sm.hmass[sb], q);
                    atomicAdd(&sm.hcount[sb], 1u);
                }
            }
            __syncthreads();
            int b2;
            unsigned long long above2;
            smp_select(target - above1, sm, b2, above2);
            s2 = kSmpBins - 1 - b2;
            base = above1 + above2;
            nreg = sm.hcount[b2];
            // keys k of sub-bin s2: floor((k - kmin) * 2048 / range) == s2
            rlo = kmin + (uint32_t)(((unsigned long long)s2 * range + kSmpBins - 1) / kSmpBins);
            rhi = kmin + (uint32_t)(((unsigned long long)(s2 + 1) * range + kSmpBins - 1) / kSmpBins) - 1u;
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
        if (nreg <= (unsigned int)kSmpCand) {
            // ---- the region sorted by (logit desc, index asc), scanned to the cut
            __syncthreads();
            if (tid == 0) sm.ncand = 0u;
            __syncthreads();
            for (int i = tid; i < V; i += kSmpThreads) {
                const float v = z[i];
                int bin;
                if (smp_live(v, mx, rt, inv, bin) && in_region(v, bin)) {
                    const unsigned int slot = atomicAdd(&sm.ncand, 1u);
                    if (slot < (unsigned int)kSmpCand)
                        sm.cand[slot] = ((unsigned long long)(~smp_key(v)) << 32) | (unsigned int)i;
                }
            }
            __syncthreads();
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
            tkey = ~(uint32_t)(sm.cand[sm.ibcast[1]] >> 32);
            // the first entry with that logit, and the region's mass before it
            run = pre;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const int j = tid * E + e;
                if (j < n && ks[e] == tkey && (j == 0 || ~(uint32_t)(sm.cand[j - 1] >> 32) != tkey))
                    sm.bcast[1] = run;
                run += qs[e];
            }
            __syncthreads();
            mass_gt = base + sm.bcast[1];
        } else {
            // ---- a region of few repeated logit values: bisection over its keys for
            // the largest K with mass(region, key >= K) >= need
            unsigned long long lo = rlo, hi = (unsigned long long)rhi + 1ull, m_hi = 0ull;
            while (hi - lo > 1ull) {
                const unsigned long long mid = (lo + hi) >> 1;
                unsigned long long part = 0ull;
                for (int i = tid; i < V; i += kSmpThreads) {
                    const float v = z[i];
                    int bin;
                    const unsigned long long q = smp_mass(v, mx, rt, inv, bin);
                    if (q && in_region(v, bin) && (unsigned long long)smp_key(v) >= mid) part += q;
                }
                const unsigned long long mm = smp_sum(part, sm);
                if (mm >= need) {
                    lo = mid;
                } else {
                    hi = mid;
                    m_hi = mm;
                }
            }
            tkey = (uint32_t)lo;
            mass_gt = base + m_hi;
        }
    }
    int bin_t;
    const unsigned long long qt = smp_mass(smp_unkey(tkey), mx, rt, inv, bin_t);   // > 0
    // tokens with logit t* taken in index order: the fewest that reach the target
    const unsigned long long kties = (target - mass_gt + qt - 1ull) / qt;

    // ---- 4. inverse cumulative mass over the nucleus in vocabulary order
    const int chunk = (V + kSmpThreads - 1) / kSmpThreads;
    const int c0 = min(V, tid * chunk), c1 = min(V, c0 + chunk);
    unsigned long long gt = 0ull, nt = 0ull;
    for (int i = c0; i < c1; ++i) {
        const float v = z[i];
        if (!(v == v)) continue;
        const uint32_t k = smp_key(v);
        if (k > tkey) {
            int bin;
            gt += smp_mass(v, mx, rt, inv, bin);
        } else if (k == tkey) {
            ++nt;
        }
    }
    unsigned long long ntot;
    const unsigned long long tie0 = smp_scan(nt, sm, ntot);   // ties before this chunk
    const unsigned long long inc =
        tie0 >= kties ? 0ull : (kties - tie0 < nt ? kties - tie0 : nt);
    const unsigned long long mym = gt + inc * qt;
    unsigned long long Mn;
    const unsigned long long start = smp_scan(mym, sm, Mn);   // nucleus mass before this chunk
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
}

cudaError_t launch_sample(const SampleArgs &a, cudaStream_t s) {
    if (a.B <= 0) return cudaSuccess;
    if (a.V <= 0 || a.ld < a.V) return cudaErrorInvalidValue;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(sample_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)sizeof(SmpSmem));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    return launch_pdl_smem(sample_kernel, dim3(a.B), dim3(kSmpThreads), sizeof(SmpSmem), s, a);
}

}  // namespace bloom
