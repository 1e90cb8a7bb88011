// Weight-streaming linear layer (decode GEMV / small-M GEMM) for sm_103a.
//
// y[m][n] = epilogue(sum_k W[n][k] x[m][k]) with W bf16 or int8 (one bf16 scale
// per output row), float32 accumulation.  At small batch the step time is the
// time to read the weights once ("DeepSpeed Inference", III.A: small-batch
// inference is bounded by reading the parameters), so the kernel is organised
// around one pass over W:
//  * a warp owns kRows consecutive weight rows and a tile of BT tokens; lane l
//    reads 16-byte chunks l, l+32, ... of each row (full 512-byte lines per
//    warp instruction), streamed past L1, several chunks in flight per lane;
//  * the activations (BT rows) are read through L1, where all warps of the SM
//    share them;
//  * partial sums are combined with a transposing butterfly: at each shuffle
//    step a lane keeps half of its values and trades the other half, so the
//    kRows*BT sums finish in kRows*BT - 1 + (5 - log2(kRows*BT)) shuffles
//    instead of 5 per value (the same goal as SBI-GeMM's cooperative-group
//    reduction, "DeepSpeed Inference", III.C.2);
//  * bias, GeLU, the residual add (into the float32 residual stream), the head-interleaved Q/K/V scatter into the
//    KV cache, and the LM head's argmax are applied in the epilogue (the
//    fusions of "DeepSpeed Inference", III.D);
//  * the grid is sized to the SM count and warps loop over (row group, token
//    tile) tasks, token tiles fastest, so rows re-read for another token tile
//    come from L2.
#include "common.cuh"
#include "kernels.h"

namespace bloom {

constexpr int kRows = 4;
constexpr int kLinWarps = 4;
constexpr int kLinThreads = kLinWarps * kWarp;

template <int V>
struct Log2 { static constexpr int value = 1 + Log2<V / 2>::value; };
template <>
struct Log2<1> { static constexpr int value = 0; };

// Sum over the warp of acc[i] for i = lane >> (5 - log2 V); V a power of two <= 32.
template <int V>
__device__ __forceinline__ float warp_reduce_transpose(float (&acc)[V], int lane) {
#pragma unroll
    for (int n = V, off = 16; n > 1; n >>= 1, off >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float send = upper ? acc[i] : acc[i + n / 2];
            const float keep = upper ? acc[i + n / 2] : acc[i];
            acc[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
    float v = acc[0];
#pragma unroll
    for (int off = 16 / V; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// Eight weights of group g (0 or 1) of a 16-byte int8 chunk, or the 8 bf16 of a
// bf16 chunk (g = 0), as floats.
template <bool INT8>
__device__ __forceinline__ void weights8(const uint4 &v, int g, float *f) {
    if constexpr (!INT8) {
        unpack8(v, f);
    } else {
        const uint32_t a = g ? v.z : v.x;
        const uint32_t b = g ? v.w : v.y;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            f[j] = (float)(int8_t)(a >> (8 * j));
            f[4 + j] = (float)(int8_t)(b >> (8 * j));
        }
    }
}

template <int BT, bool INT8, int EPI>
__global__ void __launch_bounds__(kLinThreads) linear_kernel(const LinearArgs a) {
    constexpr int EPL = INT8 ? 16 : 8;          // elements per 16-byte chunk
    constexpr int G = EPL / 8;                  // 8-element groups per chunk
    constexpr int U = (BT >= 8) ? 2 : 4;        // chunks in flight per row per lane
    constexpr int V = kRows * BT;
    constexpr int SHIFT = 5 - Log2<V>::value;

    __shared__ unsigned long long s_best[EPI == EPI_ARGMAX ? kMaxBatch : 1];
    __shared__ int s_last;

    const int lane = threadIdx.x & 31;
    if constexpr (EPI == EPI_ARGMAX) {
        for (int i = threadIdx.x; i < a.M; i += blockDim.x) s_best[i] = 0ull;
        __syncthreads();
    }

    const long long gwarp = (long long)blockIdx.x * kLinWarps + (threadIdx.x >> 5);
    const long long nwarps = (long long)gridDim.x * kLinWarps;
    const int nchunks = a.K / EPL;
    const int row_groups = (a.N + kRows - 1) / kRows;
    const int tok_tiles = (a.M + BT - 1) / BT;
    const long long tasks = (long long)row_groups * tok_tiles;
    const size_t row_bytes = (size_t)a.K * (INT8 ? 1 : 2);
    const char *wbase = reinterpret_cast<const char *>(a.w);

    for (long long task = gwarp; task < tasks; task += nwarps) {
        const int rg = (int)(task / tok_tiles);
        const int tt = (int)(task - (long long)rg * tok_tiles);
        const int row0 = rg * kRows;
        const int m0 = tt * BT;

        const char *wr[kRows];
#pragma unroll
        for (int r = 0; r < kRows; ++r)
            wr[r] = wbase + (size_t)min(row0 + r, a.N - 1) * row_bytes;
        const uint16_t *xr[BT];
#pragma unroll
        for (int b = 0; b < BT; ++b) xr[b] = a.x + (size_t)min(m0 + b, a.M - 1) * a.K;

        float acc[V];
#pragma unroll
        for (int i = 0; i < V; ++i) acc[i] = 0.f;

        for (int c0 = lane; c0 < nchunks; c0 += kWarp * U) {
            uint4 wv[U][kRows];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + u * kWarp;
#pragma unroll
                for (int r = 0; r < kRows; ++r)
                    wv[u][r] = (c < nchunks) ? ld_stream(wr[r] + (size_t)c * 16)
                                             : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + u * kWarp;
                if (c < nchunks) {
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        const int k = c * EPL + g * 8;
                        float xf[BT][8];
#pragma unroll
                        for (int b = 0; b < BT; ++b) unpack8(ld_act(xr[b] + k), xf[b]);
#pragma unroll
                        for (int r = 0; r < kRows; ++r) {
                            float wf[8];
                            weights8<INT8>(wv[u][r], g, wf);
#pragma unroll
                            for (int b = 0; b < BT; ++b)
#pragma unroll
                                for (int e = 0; e < 8; ++e)
                                    acc[r * BT + b] = fmaf(wf[e], xf[b][e], acc[r * BT + b]);
                        }
                    }
                }
            }
        }

        const float sum = warp_reduce_transpose<V>(acc, lane);
        const int idx = lane >> SHIFT;
        const int r = idx / BT, b = idx - (idx / BT) * BT;
        const int row = row0 + r, m = m0 + b;
        if ((lane & ((1 << SHIFT) - 1)) != 0 || row >= a.N || m >= a.M) continue;

        float v = sum;
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
            const int d = a.head_dim;
            const int j = row / (3 * d);
            const int cidx = (row / d) % 3;
            const int e = row % d;
            if (cidx == 0) {
                a.q_out[(size_t)m * a.n_head * d + (size_t)j * d + e] = f2bf(v);
            } else {
                int seq, slot;
                if (a.T > 0) { seq = m / a.T; slot = m - seq * a.T; }
                else { seq = m; slot = *a.len_ptr; }
                if (slot >= 0 && slot < a.max_seq) {
                    uint16_t *cache = (cidx == 1) ? a.k_cache : a.v_cache;
                    cache[(((size_t)seq * a.n_head + j) * a.max_seq + slot) * d + e] = f2bf(v);
                } else if (a.err) {
                    atomicOr(a.err, kErrSlot);
                }
            }
        } else if constexpr (EPI == EPI_ARGMAX) {
            if (a.logits) a.logits[o] = v;
            atomicMax(&s_best[m], pack_argmax(v, (uint32_t)row));
        }
    }

    if constexpr (EPI == EPI_ARGMAX) {
        // CTA partial maxima -> global; the last CTA to finish publishes the
        // tokens and leaves the scratch zeroed for the next launch.
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

template <int BT, bool INT8, int EPI>
static int occupancy() {
    static int occ = 0;
    if (occ == 0) {
        int o = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, linear_kernel<BT, INT8, EPI>,
                                                          kLinThreads, 0) != cudaSuccess || o < 1)
            o = 1;
        occ = o;
    }
    return occ;
}

template <int BT, bool INT8, int EPI>
static cudaError_t launch_t(const LinearArgs &a, int num_sms, cudaStream_t s) {
    const long long tasks = (long long)((a.N + kRows - 1) / kRows) * ((a.M + BT - 1) / BT);
    long long blocks = (tasks + kLinWarps - 1) / kLinWarps;
    const long long cap = (long long)num_sms * occupancy<BT, INT8, EPI>();
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    linear_kernel<BT, INT8, EPI><<<(unsigned)blocks, kLinThreads, 0, s>>>(a);
    return cudaGetLastError();
}

template <int BT, bool INT8>
static cudaError_t launch_epi(const LinearArgs &a, int num_sms, cudaStream_t s) {
    switch (a.epi) {
        case EPI_STORE: return launch_t<BT, INT8, EPI_STORE>(a, num_sms, s);
        case EPI_GELU: return launch_t<BT, INT8, EPI_GELU>(a, num_sms, s);
        case EPI_RESID: return launch_t<BT, INT8, EPI_RESID>(a, num_sms, s);
        case EPI_RESID32: return launch_t<BT, INT8, EPI_RESID32>(a, num_sms, s);
        case EPI_QKV: return launch_t<BT, INT8, EPI_QKV>(a, num_sms, s);
        default: return cudaErrorInvalidValue;
    }
}

template <bool INT8>
static cudaError_t launch_bt(const LinearArgs &a, int num_sms, cudaStream_t s) {
    if (a.M <= 1) return launch_epi<1, INT8>(a, num_sms, s);
    if (a.M <= 2) return launch_epi<2, INT8>(a, num_sms, s);
    if (a.M <= 4) return launch_epi<4, INT8>(a, num_sms, s);
    return launch_epi<8, INT8>(a, num_sms, s);
}

template <bool INT8, int EPI>
static void prepare_bt() {
    occupancy<1, INT8, EPI>();
    occupancy<2, INT8, EPI>();
    occupancy<4, INT8, EPI>();
    occupancy<8, INT8, EPI>();
}

// Resolve every instance's occupancy once, outside any stream capture.
cudaError_t linear_prepare() {
    prepare_bt<false, EPI_STORE>();
    prepare_bt<false, EPI_GELU>();
    prepare_bt<false, EPI_RESID>();
    prepare_bt<false, EPI_RESID32>();
    prepare_bt<false, EPI_QKV>();
    prepare_bt<false, EPI_ARGMAX>();
    prepare_bt<true, EPI_STORE>();
    prepare_bt<true, EPI_GELU>();
    prepare_bt<true, EPI_RESID>();
    prepare_bt<true, EPI_RESID32>();
    prepare_bt<true, EPI_QKV>();
    return cudaGetLastError();
}

cudaError_t launch_linear(const LinearArgs &a, int num_sms, cudaStream_t s) {
    if (a.M <= 0 || a.N <= 0) return cudaSuccess;
    if (a.epi == EPI_ARGMAX) {
        if (a.int8 || a.M > kMaxBatch) return cudaErrorInvalidValue;
        if (a.M <= 1) return launch_t<1, false, EPI_ARGMAX>(a, num_sms, s);
        if (a.M <= 2) return launch_t<2, false, EPI_ARGMAX>(a, num_sms, s);
        if (a.M <= 4) return launch_t<4, false, EPI_ARGMAX>(a, num_sms, s);
        return launch_t<8, false, EPI_ARGMAX>(a, num_sms, s);
    }
    return a.int8 ? launch_bt<true>(a, num_sms, s) : launch_bt<false>(a, num_sms, s);
}

}  // namespace bloom
