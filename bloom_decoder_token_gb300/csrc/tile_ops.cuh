// Tile-level device helpers of the weight-streaming linear kernels: the
// mma.sync fragment op, exact int8 -> bf16 widening, the LayerNorm prologue
// into shared memory, and the argmax publication.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace bloom {

// D[16x8] += A[16x16] * B[16x8], bf16 inputs, float32 accumulators.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two int8 codes (bytes i, i+1 of w) -> bf16x2, exactly.  With the sign bits
// flipped (w ^ 0x80808080), byte permutes place q + 128 as the low mantissa
// byte of two floats 2^23 + (q + 128); one paired float32 add removes
// 2^23 + 128 from both and one conversion packs them (|q| <= 128 is exact in
// bf16).  Four instructions per pair, the flip shared by a word's two pairs.
__device__ __forceinline__ uint32_t i8x2_to_bf16x2(uint32_t w, int i) {
    const uint32_t wx = w ^ 0x80808080u;
    uint32_t u0, u1;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(u0) : "r"(wx), "r"(0x4b000000u), "r"(0x7540u | i));
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(u1) : "r"(wx), "r"(0x4b000000u), "r"(0x7540u | (i + 1)));
    const unsigned long long p = ((unsigned long long)u1 << 32) | u0;
    const unsigned long long off = 0xcb000080cb000080ull;   // -(2^23 + 128) in both halves
    unsigned long long r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(p), "l"(off));
    uint32_t o;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;"
        : "=r"(o)
        : "f"(__uint_as_float((uint32_t)(r >> 32))), "f"(__uint_as_float((uint32_t)r)));
    return o;
}

// Two int8 codes (bytes i, i+1 of w) -> f16x2, exactly.  With the sign bits
// flipped (w ^ 0x80808080), one byte permute places q + 128 as the low
// mantissa byte of two halves 1024 + (q + 128) (high byte 0x64), and one paired
// half subtraction removes 1152 (|q| <= 128 is exact in f16).  Two
// instructions per pair, the flip shared by a word's two pairs.
__device__ __forceinline__ uint32_t i8x2_to_f16x2(uint32_t w, int i) {
    const uint32_t wx = w ^ 0x80808080u;
    uint32_t h, o;
    asm("prmt.b32 %0, %1, %2, %3;"
        : "=r"(h)
        : "r"(wx), "r"(0x64646464u), "r"(0x4040u | (uint32_t)i | ((uint32_t)(i + 1) << 8)));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(o) : "r"(h), "r"(0x64806480u));
    return o;
}

// Eight bf16 -> eight f16 (round to nearest; exact for |x| in [2^-14, 65504],
// where f16 holds every bf16 value).
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 v) {
    auto cv = [](uint32_t w) {
        uint32_t o;
        asm("cvt.rn.f16x2.f32 %0, %1, %2;"
            : "=r"(o)
            : "f"(__uint_as_float(w & 0xffff0000u)), "f"(__uint_as_float(w << 16)));
        return o;
    };
    return make_uint4(cv(v.x), cv(v.y), cv(v.z), cv(v.w));
}

// LayerNorm of the M float32 rows a.ln_x[M][K] into shared memory as bf16
// (row pitch px bytes), the register-lean form for kernels whose occupancy
// matters more than the latency of the prologue: float32 statistics, biased
// variance, eps inside the square root.  Rows are spread over the CTA's warps (a team of 256 / rows
// threads per row, at least one warp); the statistics come from one pass of
// sums shifted by the row's first element (sum (x-s), sum (x-s)^2), which keeps
// the variance free of cancellation when |mean| >> std.  All threads of the CTA
// call it (two barriers).
__device__ __forceinline__ void layernorm_rows_to_smem_shifted(const LinearArgs &a, unsigned char *xs,
                                                       int px, float *s_sum, int tid, int warp,
                                                       int lane) {
    const int nthr = blockDim.x, nw = nthr / 32;
    int team_w = nw;                        // warps per row
    while (team_w > 1 && team_w > nw / (a.M < nw ? a.M : nw)) team_w >>= 1;
    const int teams = nw / team_w;
    const int team = warp / team_w, tw = warp % team_w;
    const int tthr = team_w * 32, ttid = tw * 32 + lane;
    float *stat = s_sum;                    // [nw][2]
    for (int m0 = 0; m0 < a.M; m0 += teams) {
        const int m = m0 + team;
        float s1 = 0.f, s2 = 0.f, shift = 0.f;
        if (m < a.M) {
            const float *xr = a.ln_x + (size_t)m * a.K;
            shift = xr[0];
            for (int k = ttid * 4; k < a.K; k += 4 * tthr) {
                const float4 v = *reinterpret_cast<const float4 *>(xr + k);
                const float d0 = v.x - shift, d1 = v.y - shift, d2 = v.z - shift, d3 = v.w - shift;
                s1 += (d0 + d1) + (d2 + d3);
                s2 += (d0 * d0 + d1 * d1) + (d2 * d2 + d3 * d3);
            }
        }
        s1 = warp_sum(s1);
        s2 = warp_sum(s2);
        if (lane == 0) {
            stat[2 * warp] = s1;
            stat[2 * warp + 1] = s2;
        }
        __syncthreads();
        if (m < a.M) {
            float t1 = 0.f, t2 = 0.f;
            for (int w = team * team_w; w < (team + 1) * team_w; ++w) {
                t1 += stat[2 * w];
                t2 += stat[2 * w + 1];
            }
            const float inv_k = 1.f / (float)a.K;
            const float dm = t1 * inv_k;
            const float var = fmaxf(t2 * inv_k - dm * dm, 0.f);
            const float mean = shift + dm;
            const float rstd = rsqrtf(var + a.ln_eps);
            const float *xr = a.ln_x + (size_t)m * a.K;
            uint16_t *dst = reinterpret_cast<uint16_t *>(xs + (size_t)m * px);
            for (int k = ttid * 4; k < a.K; k += 4 * tthr) {
                const float4 v = *reinterpret_cast<const float4 *>(xr + k);
                const uint2 gg = *reinterpret_cast<const uint2 *>(a.ln_g + k);
                const uint2 bb = *reinterpret_cast<const uint2 *>(a.ln_b + k);
                uint2 o;
                o.x = pack_bf2((v.x - mean) * rstd * bf_lo(gg.x) + bf_lo(bb.x),
                               (v.y - mean) * rstd * bf_hi(gg.x) + bf_hi(bb.x));
                o.y = pack_bf2((v.z - mean) * rstd * bf_lo(gg.y) + bf_lo(bb.y),
                               (v.w - mean) * rstd * bf_hi(gg.y) + bf_hi(bb.y));
                *reinterpret_cast<uint2 *>(dst + k) = o;
            }
        }
        __syncthreads();
    }
}

// Merge of two (count, mean, sum of squared deviations) summaries of a set of
// values (the pairwise update of Chan, Golub and LeVeque).
__device__ __forceinline__ void stats_merge(float &n, float &mean, float &m2, float nb, float meanb,
                                            float m2b) {
    const float nn = n + nb;
    if (nb == 0.f) return;
    if (n == 0.f) {
        n = nb;
        mean = meanb;
        m2 = m2b;
        return;
    }
    const float delta = meanb - mean;
    const float f = nb / nn;
    mean += delta * f;
    m2 += m2b + delta * delta * n * f;
    n = nn;
}

// LayerNorm of the M float32 rows a.ln_x[M][K] into shared memory as bf16
// (row pitch px bytes); float32 statistics, biased variance, eps inside the
// square root.  Rows are spread over the CTA's warps (a team of 256 / rows
// threads per row, at least one warp).  Every load of a row is issued before
// any is used (one L2 round trip), each thread summarises its values as
// (count, mean, squared deviations) around its own first value and the
// summaries are merged pairwise (no E[x^2] - mean^2 cancellation); the gamma /
// beta lines are pulled into L1 meanwhile, so that the normalising pass, which
// re-reads the row from L1, waits on nothing.  All threads of the CTA call it.
template <int UL>   // float4 loads in flight per thread (register budget of the caller)
__device__ __forceinline__ void layernorm_rows_to_smem(const LinearArgs &a, unsigned char *xs,
                                                       int px, float *s_sum, int tid, int warp,
                                                       int lane) {
    const int nthr = blockDim.x, nw = nthr / 32;
    int team_w = nw;                        // warps per row
    while (team_w > 1 && team_w > nw / (a.M < nw ? a.M : nw)) team_w >>= 1;
    const int teams = nw / team_w;
    const int team = warp / team_w, tw = warp % team_w;
    const int tthr = team_w * 32, ttid = tw * 32 + lane;
    float *stat = s_sum;                    // [nw][3] (s_sum holds 3 * nw floats)
    for (int m0 = 0; m0 < a.M; m0 += teams) {
        const int m = m0 + team;
        float n = 0.f, mean = 0.f, m2 = 0.f;
        if (m < a.M) {
            const float *xr = a.ln_x + (size_t)m * a.K;
            for (int kb = ttid * 4; kb < a.K; kb += 4 * tthr * UL) {
                float4 v[UL];
#pragma unroll
                for (int u = 0; u < UL; ++u) {
                    const int k = kb + u * 4 * tthr;
                    if (k < a.K) {
                        v[u] = *reinterpret_cast<const float4 *>(xr + k);
                        // the normalising pass needs gamma / beta of these k from L1
                        asm volatile("prefetch.global.L1 [%0];" ::"l"(a.ln_g + k));
                        asm volatile("prefetch.global.L1 [%0];" ::"l"(a.ln_b + k));
                    }
                }
#pragma unroll
                for (int u = 0; u < UL; ++u) {
                    const int k = kb + u * 4 * tthr;
                    if (k < a.K) {
                        // summary of these four values, merged into the running one
                        const float c = 0.25f * ((v[u].x + v[u].y) + (v[u].z + v[u].w));
                        const float d0 = v[u].x - c, d1 = v[u].y - c, d2 = v[u].z - c, d3 = v[u].w - c;
                        stats_merge(n, mean, m2, 4.f, c, (d0 * d0 + d1 * d1) + (d2 * d2 + d3 * d3));
                    }
                }
            }
        }
        // merge over the warp, then over the team's warps
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float nb = __shfl_xor_sync(0xffffffffu, n, o);
            const float mb = __shfl_xor_sync(0xffffffffu, mean, o);
            const float qb = __shfl_xor_sync(0xffffffffu, m2, o);
            stats_merge(n, mean, m2, nb, mb, qb);
        }
        if (lane == 0) {
            stat[3 * warp] = n;
            stat[3 * warp + 1] = mean;
            stat[3 * warp + 2] = m2;
        }
        __syncthreads();
        if (m < a.M) {
            float tn = 0.f, tmean = 0.f, tm2 = 0.f;
            for (int w = team * team_w; w < (team + 1) * team_w; ++w)
                stats_merge(tn, tmean, tm2, stat[3 * w], stat[3 * w + 1], stat[3 * w + 2]);
            const float var = fmaxf(tm2 / (float)a.K, 0.f);
            const float rstd = rsqrtf(var + a.ln_eps);
            const float *xr = a.ln_x + (size_t)m * a.K;
            uint16_t *dst = reinterpret_cast<uint16_t *>(xs + (size_t)m * px);
            for (int kb = ttid * 4; kb < a.K; kb += 4 * tthr * UL) {
                // every load of this round first, then the arithmetic
                float4 v[UL];
                uint2 gg[UL], bb[UL];
#pragma unroll
                for (int u = 0; u < UL; ++u) {
                    const int k = kb + u * 4 * tthr;
                    if (k < a.K) {
                        v[u] = *reinterpret_cast<const float4 *>(xr + k);
                        gg[u] = __ldg(reinterpret_cast<const uint2 *>(a.ln_g + k));
                        bb[u] = __ldg(reinterpret_cast<const uint2 *>(a.ln_b + k));
                    }
                }
#pragma unroll
                for (int u = 0; u < UL; ++u) {
                    const int k = kb + u * 4 * tthr;
                    if (k < a.K) {
                        uint2 o;
                        o.x = pack_bf2((v[u].x - tmean) * rstd * bf_lo(gg[u].x) + bf_lo(bb[u].x),
                                       (v[u].y - tmean) * rstd * bf_hi(gg[u].x) + bf_hi(bb[u].x));
                        o.y = pack_bf2((v[u].z - tmean) * rstd * bf_lo(gg[u].y) + bf_lo(bb[u].y),
                                       (v[u].w - tmean) * rstd * bf_hi(gg[u].y) + bf_hi(bb[u].y));
                        *reinterpret_cast<uint2 *>(dst + k) = o;
                    }
                }
            }
        }
        __syncthreads();
    }
}

// CTA maxima -> global; the last CTA of the grid publishes the tokens and
// leaves the scratch zeroed for the next launch (no waiting: a ticket decides
// which CTA is last).  Contains barriers; all threads call it.
__device__ __forceinline__ void argmax_publish(const LinearArgs &a, unsigned long long *s_best,
                                               int *s_last, int tid, int grid) {
    __syncthreads();
    for (int i = tid; i < a.M; i += blockDim.x)
        if (s_best[i]) atomicMax(&a.best[i], s_best[i]);
    __threadfence();
    __syncthreads();
    if (tid == 0) *s_last = (atomicAdd(a.ticket, 1) == grid - 1);
    __syncthreads();
    if (*s_last) {
        __threadfence();
        for (int i = tid; i < a.M; i += blockDim.x) {
            const unsigned long long p = atomicExch(&a.best[i], 0ull);
            const bool act = !a.active || a.active[i];
            a.out_tokens[i] = act ? (int)unpack_index(p) : -1;
            if (a.len_inc && act) {   // the step appended a slot to this row
                a.len_inc[i] += 1;
                a.next_pos[i] += 1;
            }
        }
        if (tid == 0) *a.ticket = 0;
    }
}

}  // namespace bloom
