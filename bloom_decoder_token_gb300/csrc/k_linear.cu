// Weight-streaming linear layer for decode (and small-M prefill) on sm_103a.
//
// y[m][n] = epilogue(sum_k W[n][k] x[m][k]), W bf16 or int8 (one bf16 scale per
// output row), float32 accumulation.  At small batch the time is the time to
// read W once ("DeepSpeed Inference", III.A), so the kernel is built around one
// coalesced pass over W with as little instruction work per byte as possible:
//
//  * a CTA (8 warps) owns 8 consecutive weight rows and a tile of up to 16*MT
//    tokens; its warps split K into interleaved chunks (lane (g, q) reads 16
//    bytes of row g at offset 16q of the chunk, so each warp load covers 8 rows
//    x 64 bytes), every CTA streams its rows in order with several chunks in
//    flight per lane (output-dimension tiling plus an input-dimension split, as
//    in SBI-GeMM, "DeepSpeed Inference", III.C.1);
//  * the 16 bytes a lane loads ARE its mma.sync m16n8k16 B fragment: within a
//    chunk, logical k positions {2q, 2q+1, 2q+8, 2q+9} of mma step s are bound
//    to physical elements q*EPL + 4s + {0..3}.  The activations use the same
//    binding, so the dot product is unchanged while both operands come straight
//    from 16-byte loads (no shared-memory staging, no shuffles);
//  * int8 codes are widened exactly to bf16 (|q| <= 127) and the row scale is
//    applied once in the epilogue (y = s_n * sum q x);
//  * the 8 warps' partial tiles are summed through shared memory (a transpose
//    through shared memory instead of a shuffle tree, cf. III.C.2), then bias,
//    GeLU, the float32 residual add, the head-interleaved Q/K/V scatter into
//    the KV cache, or the LM head's logits + argmax are applied (the fusions of
//    III.D);
//  * launched with programmatic stream serialization: the weight loads of the
//    first tile are issued before griddepcontrol.wait, so they overlap the tail
//    of the kernel that produces x.
#include "common.cuh"
#include "kernels.h"

namespace bloom {

constexpr int kLinWarps = 8;
constexpr int kLinThreads = kLinWarps * kWarp;

// D[16x8] += A[16x16] * B[16x8], bf16 inputs, float32 accumulators.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two int8 codes (bytes i, i+1 of w) -> bf16x2, exactly: 2^23 + (q + 128) is an
// exact float whose low mantissa byte is q + 128; subtracting 2^23 + 128 leaves q.
__device__ __forceinline__ uint32_t i8x2_to_bf16x2(uint32_t w, int i) {
    const uint32_t b0 = ((w >> (8 * i)) & 0xffu) ^ 0x80u;
    const uint32_t b1 = ((w >> (8 * i + 8)) & 0xffu) ^ 0x80u;
    const float f0 = __uint_as_float(0x4b000000u | b0) - 8388736.0f;
    const float f1 = __uint_as_float(0x4b000000u | b1) - 8388736.0f;
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(f1), "f"(f0));
    return r;
}

template <int MT, bool INT8, int EPI>
__global__ void __launch_bounds__(kLinThreads) linear_kernel(const LinearArgs a) {
    constexpr int EPL = INT8 ? 16 : 8;   // weights per lane per chunk (16 bytes)
    constexpr int KC = 4 * EPL;          // k per chunk
    constexpr int NS = EPL / 4;          // mma k-steps per chunk
    constexpr int XW = EPL / 2;          // 32-bit words of x per lane per chunk
    constexpr int U = (MT >= 4) ? 2 : 4; // chunks in flight per warp

    __shared__ float red[kLinWarps][MT][4][kWarp];
    __shared__ unsigned long long s_best[EPI == EPI_ARGMAX ? kMaxBatch : 1];
    __shared__ int s_last;

    griddep_launch();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, q = lane & 3;
    if constexpr (EPI == EPI_ARGMAX) {
        for (int i = threadIdx.x; i < a.M; i += blockDim.x) s_best[i] = 0ull;
    }

    const int nchunks = (a.K + KC - 1) / KC;
    const int row_groups = (a.N + 7) / 8;
    const int tok_tiles = (a.M + 16 * MT - 1) / (16 * MT);
    const long long tasks = (long long)row_groups * tok_tiles;
    const size_t row_bytes = (size_t)a.K * (INT8 ? 1 : 2);
    const char *wbase = reinterpret_cast<const char *>(a.w);
    bool waited = false;

    for (long long task = blockIdx.x; task < tasks; task += gridDim.x) {
        const int rg = (int)(task / tok_tiles);
        const int tt = (int)(task - (long long)rg * tok_tiles);
        const int row0 = rg * 8, m0 = tt * 16 * MT;
        const int wrow = row0 + g;
        const bool wok = wrow < a.N;
        const char *wp = wbase + (size_t)(wok ? wrow : 0) * row_bytes + (size_t)q * 16;
        float acc[MT][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[mt][r] = 0.f;

        for (int c0 = warp; c0 < nchunks; c0 += kLinWarps * U) {
            uint4 wv[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + u * kLinWarps;
                const int k = c * KC + q * EPL;
                wv[u] = (wok && c < nchunks && k < a.K)
                            ? ld_stream(wp + (size_t)c * KC * (INT8 ? 1 : 2))
                            : make_uint4(0u, 0u, 0u, 0u);
            }
            if (!waited) {
                griddep_wait();   // x (and the residual) come from earlier kernels
                waited = true;
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + u * kLinWarps;
                if (c >= nchunks) break;
                const int k = c * KC + q * EPL;
                uint32_t xa[MT][XW], xb[MT][XW];
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    const int ma = m0 + mt * 16 + g, mb = ma + 8;
#pragma unroll
                    for (int hh = 0; hh < XW / 4; ++hh) {
                        uint4 va = make_uint4(0u, 0u, 0u, 0u), vb = va;
                        if (ma < a.M && k < a.K) va = ld_act(a.x + (size_t)ma * a.K + k + 8 * hh);
                        if (mb < a.M && k < a.K) vb = ld_act(a.x + (size_t)mb * a.K + k + 8 * hh);
                        xa[mt][4 * hh + 0] = va.x; xa[mt][4 * hh + 1] = va.y;
                        xa[mt][4 * hh + 2] = va.z; xa[mt][4 * hh + 3] = va.w;
                        xb[mt][4 * hh + 0] = vb.x; xb[mt][4 * hh + 1] = vb.y;
                        xb[mt][4 * hh + 2] = vb.z; xb[mt][4 * hh + 3] = vb.w;
                    }
                }
                const uint32_t ww[4] = {wv[u].x, wv[u].y, wv[u].z, wv[u].w};
#pragma unroll
                for (int s = 0; s < NS; ++s) {
                    uint32_t b0, b1;
                    if constexpr (INT8) {
                        b0 = i8x2_to_bf16x2(ww[s], 0);
                        b1 = i8x2_to_bf16x2(ww[s], 2);
                    } else {
                        b0 = ww[2 * s];
                        b1 = ww[2 * s + 1];
                    }
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt)
                        mma_bf16(acc[mt], xa[mt][2 * s], xb[mt][2 * s], xa[mt][2 * s + 1],
                                 xb[mt][2 * s + 1], b0, b1);
                }
            }
        }
        if (!waited) {
            griddep_wait();
            waited = true;
        }

        // sum the 8 warps' partial tiles; warp mt finishes token tile mt
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int r = 0; r < 4; ++r) red[warp][mt][r][lane] = acc[mt][r];
        __syncthreads();
        if (warp < MT) {
            const int mt = warp;
            float d[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                float t = 0.f;
#pragma unroll
                for (int w = 0; w < kLinWarps; ++w) t += red[w][mt][r][lane];
                d[r] = t;
            }
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int m = m0 + mt * 16 + g + 8 * half;
                if (m >= a.M) continue;
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int row = row0 + 2 * q + j;
                    if (row >= a.N) continue;
                    float v = d[2 * half + j];
                    if constexpr (INT8) v *= bf2f(a.scale[row]);
                    if (a.bias) v += bf2f(a.bias[row]);
                    const size_t o = (size_t)m * a.N + row;
                    if constexpr (EPI == EPI_STORE) {
                        a.out[o] = f2bf(v);
                    } else if constexpr (EPI == EPI_GELU) {
                        a.out[o] = f2bf(gelu_tanh(v));
                    } else if constexpr (EPI == EPI_RESID) {
                        a.out[o] = f2bf(bf2f(a.out[o]) + v);
                    } else if constexpr (EPI == EPI_RESID32) {
                        a.out32[o] += v;
                    } else if constexpr (EPI == EPI_QKV) {
                        const int dh = a.head_dim;
                        const int hj = row / (3 * dh);
                        const int cidx = (row / dh) % 3;
                        const int e = row % dh;
                        if (cidx == 0) {
                            a.q_out[(size_t)m * a.n_head * dh + (size_t)hj * dh + e] = f2bf(v);
                        } else {
                            int seq, slot;
                            if (a.T > 0) { seq = m / a.T; slot = m - seq * a.T; }
                            else { seq = m; slot = *a.len_ptr; }
                            if (slot >= 0 && slot < a.max_seq) {
                                uint16_t *cache = (cidx == 1) ? a.k_cache : a.v_cache;
                                cache[(((size_t)seq * a.n_head + hj) * a.max_seq + slot) * dh + e] =
                                    f2bf(v);
                            } else if (a.err) {
                                atomicOr(a.err, kErrSlot);
                            }
                        }
                    } else if constexpr (EPI == EPI_ARGMAX) {
                        if (a.logits) a.logits[o] = v;
                        atomicMax(&s_best[m], pack_argmax(v, (uint32_t)row));
                    }
                }
            }
        }
        __syncthreads();
    }

    if constexpr (EPI == EPI_ARGMAX) {
        // CTA maxima -> global; the last CTA publishes the tokens and leaves
        // the scratch zeroed for the next launch.
        if (!waited) griddep_wait();
        __syncthreads();
        for (int i = threadIdx.x; i < a.M; i += blockDim.x)
            if (s_best[i]) atomicMax(&a.best[i], s_best[i]);
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) s_last = (atomicAdd(a.ticket, 1) == (int)gridDim.x - 1);
        __syncthreads();
        if (s_last) {
            __threadfence();
            for (int i = threadIdx.x; i < a.M; i += blockDim.x) {
                const unsigned long long p = atomicExch(&a.best[i], 0ull);
                a.out_tokens[i] = (int)unpack_index(p);
                if (a.len_inc) a.next_pos[i] += 1;
            }
            if (threadIdx.x == 0) {
                *a.ticket = 0;
                if (a.len_inc) *a.len_inc += 1;
            }
        }
    }
}

template <int MT, bool INT8, int EPI>
static int occupancy() {
    static int occ = 0;
    if (occ == 0) {
        int o = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, linear_kernel<MT, INT8, EPI>,
                                                          kLinThreads, 0) != cudaSuccess || o < 1)
            o = 1;
        occ = o;
    }
    return occ;
}

template <int MT, bool INT8, int EPI>
static cudaError_t launch_t(const LinearArgs &a, int num_sms, cudaStream_t s) {
    const long long tasks = (long long)((a.N + 7) / 8) * ((a.M + 16 * MT - 1) / (16 * MT));
    long long blocks = tasks;
    const long long cap = (long long)num_sms * occupancy<MT, INT8, EPI>();
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return launch_pdl(linear_kernel<MT, INT8, EPI>, dim3((unsigned)blocks), dim3(kLinThreads), s,
                      a);
}

template <int MT, bool INT8>
static cudaError_t launch_epi(const LinearArgs &a, int num_sms, cudaStream_t s) {
    switch (a.epi) {
        case EPI_STORE: return launch_t<MT, INT8, EPI_STORE>(a, num_sms, s);
        case EPI_GELU: return launch_t<MT, INT8, EPI_GELU>(a, num_sms, s);
        case EPI_RESID: return launch_t<MT, INT8, EPI_RESID>(a, num_sms, s);
        case EPI_RESID32: return launch_t<MT, INT8, EPI_RESID32>(a, num_sms, s);
        case EPI_QKV: return launch_t<MT, INT8, EPI_QKV>(a, num_sms, s);
        default: return cudaErrorInvalidValue;
    }
}

template <bool INT8>
static cudaError_t launch_mt(const LinearArgs &a, int num_sms, cudaStream_t s) {
    if (a.M <= 16) return launch_epi<1, INT8>(a, num_sms, s);
    if (a.M <= 32) return launch_epi<2, INT8>(a, num_sms, s);
    return launch_epi<4, INT8>(a, num_sms, s);
}

template <bool INT8, int EPI>
static void prepare_mt() {
    occupancy<1, INT8, EPI>();
    occupancy<2, INT8, EPI>();
    occupancy<4, INT8, EPI>();
}

// Resolve every instance's occupancy once, outside any stream capture.
cudaError_t linear_prepare() {
    prepare_mt<false, EPI_STORE>();
    prepare_mt<false, EPI_GELU>();
    prepare_mt<false, EPI_RESID>();
    prepare_mt<false, EPI_RESID32>();
    prepare_mt<false, EPI_QKV>();
    prepare_mt<false, EPI_ARGMAX>();
    prepare_mt<true, EPI_STORE>();
    prepare_mt<true, EPI_GELU>();
    prepare_mt<true, EPI_RESID>();
    prepare_mt<true, EPI_RESID32>();
    prepare_mt<true, EPI_QKV>();
    return cudaGetLastError();
}

cudaError_t launch_linear(const LinearArgs &a, int num_sms, cudaStream_t s) {
    if (a.M <= 0 || a.N <= 0) return cudaSuccess;
    if (a.epi == EPI_ARGMAX) {
        if (a.int8 || a.M > kMaxBatch) return cudaErrorInvalidValue;
        if (a.M <= 16) return launch_t<1, false, EPI_ARGMAX>(a, num_sms, s);
        if (a.M <= 32) return launch_t<2, false, EPI_ARGMAX>(a, num_sms, s);
        return launch_t<4, false, EPI_ARGMAX>(a, num_sms, s);
    }
    return a.int8 ? launch_mt<true>(a, num_sms, s) : launch_mt<false>(a, num_sms, s);
}

}  // namespace bloom
