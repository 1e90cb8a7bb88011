// LayerNorm of one row by one 256-thread block, all values held in registers:
// float32 mean, then float32 biased variance of the deviations (two passes over
// registers, no E[x^2] - mean^2 cancellation), eps inside the square root,
// affine gamma / beta.  "DeepSpeed Inference", III.B: all micro-operations of
// the layer norm, its reductions included, run in one kernel because the
// reduced dimension stays inside one thread block.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace bloom {

constexpr int kLnThreads = 256;
constexpr int kLnWarps = kLnThreads / kWarp;
constexpr int kLnChunks = kMaxHidden / 8 / kLnThreads;   // 8-element chunks per thread, at most

__device__ __forceinline__ void load8(const uint16_t *p, float *f) {
    unpack8(*reinterpret_cast<const uint4 *>(p), f);
}
__device__ __forceinline__ void load8(const float *p, float *f) {
    const float4 a = reinterpret_cast<const float4 *>(p)[0];
    const float4 b = reinterpret_cast<const float4 *>(p)[1];
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}
__device__ __forceinline__ void store8(uint16_t *p, const float *y) {
    uint4 o;
    o.x = pack_bf2(y[0], y[1]);
    o.y = pack_bf2(y[2], y[3]);
    o.z = pack_bf2(y[4], y[5]);
    o.w = pack_bf2(y[6], y[7]);
    *reinterpret_cast<uint4 *>(p) = o;
}
__device__ __forceinline__ void store8(float *p, const float *y) {
    reinterpret_cast<float4 *>(p)[0] = make_float4(y[0], y[1], y[2], y[3]);
    reinterpret_cast<float4 *>(p)[1] = make_float4(y[4], y[5], y[6], y[7]);
}

// The affine parameters of a row (gamma 1 and beta 0 where absent).  They are
// weights: for rows of up to 4 chunks a thread the kernels load them, packed
// bf16, before waiting for the previous kernel, so that only the row itself is
// on the critical path; wider rows read them at the end (registers).
template <int CH>
struct LnAffine {
    static constexpr bool kPre = CH <= 4;
    uint4 g[kPre ? CH : 1], b[kPre ? CH : 1];
    const uint16_t *gp, *bp;
};

// Chunks per thread that a row of h features needs (the kernels are compiled for 2, 4
// and kLnChunks, so that narrow rows keep few registers).
inline int ln_chunks(int h) {
    const int c = (h / 8 + kLnThreads - 1) / kLnThreads;
    return c <= 2 ? 2 : c <= 4 ? 4 : kLnChunks;
}

template <int CH>
__device__ __forceinline__ void ln_affine_load(const uint16_t *g, const uint16_t *b, int h,
                                               LnAffine<CH> &p) {
    p.gp = g;
    p.bp = b;
    if constexpr (LnAffine<CH>::kPre) {
        const int nch = h / 8;
#pragma unroll
        for (int i = 0; i < CH; ++i) {
            const int c = threadIdx.x + i * kLnThreads;
            p.g[i] = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);   // bf16 1.0
            p.b[i] = make_uint4(0u, 0u, 0u, 0u);
            if (c < nch) {
                if (g) p.g[i] = *reinterpret_cast<const uint4 *>(g + (size_t)c * 8);
                if (b) p.b[i] = *reinterpret_cast<const uint4 *>(b + (size_t)c * 8);
            }
        }
    }
}

template <int CH, typename TIn, typename TOut>
__device__ __forceinline__ void ln_row(const TIn *src, const LnAffine<CH> &p, int h, float eps,
                                       TOut *dst, float *red) {
    const int nch = h / 8;
    float v[CH][8];
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < CH; ++i) {
        const int c = threadIdx.x + i * kLnThreads;
        if (c < nch) {
            load8(src + (size_t)c * 8, v[i]);
#pragma unroll
            for (int e = 0; e < 8; ++e) s += v[i][e];
        }
    }
    const float mean = block_sum<kLnWarps>(s, red) / (float)h;
    float q = 0.f;
#pragma unroll
    for (int i = 0; i < CH; ++i) {
        const int c = threadIdx.x + i * kLnThreads;
        if (c < nch) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float dlt = v[i][e] - mean;
                q += dlt * dlt;
            }
        }
    }
    const float var = block_sum<kLnWarps>(q, red) / (float)h;
    const float rstd = rsqrtf(var + eps);
#pragma unroll
    for (int i = 0; i < CH; ++i) {
        const int c = threadIdx.x + i * kLnThreads;
        if (c < nch) {
            float gg[8], bb[8], y[8];
            if constexpr (LnAffine<CH>::kPre) {
                unpack8(p.g[i], gg);
                unpack8(p.b[i], bb);
            } else {
                if (p.gp) unpack8(*reinterpret_cast<const uint4 *>(p.gp + (size_t)c * 8), gg);
                else for (int e = 0; e < 8; ++e) gg[e] = 1.f;
                if (p.bp) unpack8(*reinterpret_cast<const uint4 *>(p.bp + (size_t)c * 8), bb);
                else for (int e = 0; e < 8; ++e) bb[e] = 0.f;
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) y[e] = (v[i][e] - mean) * rstd * gg[e] + bb[e];
            store8(dst + (size_t)c * 8, y);
        }
    }
}

}  // namespace bloom
