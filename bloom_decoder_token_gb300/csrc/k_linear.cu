// Weight-streaming linear layer for decode (and small-M prefill) on sm_103a.
//
// y[m][n] = epilogue(sum_k W[n][k] x[m][k]), W bf16 or int8 (one bf16 scale per
// output row), float32 accumulation.  At small batch the time is the time to
// read W once ("DeepSpeed Inference", III.A), so the kernel is built around one
// coalesced pass over W with as little instruction work per byte as possible:
//
//  * a CTA (8 warps) owns a task of consecutive weight rows and a tile of
//    tokens; its warps split K into interleaved chunks (lane (g, q) reads 16
//    bytes of its row(s) at offset 16q of the chunk), every CTA streams its
//    rows in order with several chunks in flight per lane (output-dimension
//    tiling plus an input-dimension split, as in SBI-GeMM, "DeepSpeed
//    Inference", III.C.1);
//  * the 16 bytes a lane loads ARE an mma.sync m16n8k16 fragment: within a
//    chunk, logical k positions {2q, 2q+1, 2q+8, 2q+9} of mma step s are bound
//    to physical elements q*EPL + 4s + {0..3}.  The activations use the same
//    binding, so the dot product is unchanged while both operands come straight
//    from 16-byte loads (no shared-memory staging, no shuffles).  Two forms:
//    weights as the B operand (8-row tasks, token tiles of 16: lane g loads row
//    g) and, for wide matrices, as the A operand (16-row tasks, token tiles of
//    8: lane g loads rows g and g + 8), which halves the mma steps and the
//    activation fragments per weight byte and keeps two rows' loads in flight;
//  * int8 codes are widened exactly to bf16 (two byte permutes, a paired
//    float32 add and a pack per pair; |q| <= 128) and the row scale is applied
//    once in the epilogue (y = s_n * sum q x);
//  * the 8 warps' partial tiles are summed through shared memory (a transpose
//    through shared memory instead of a shuffle tree, cf. III.C.2), then bias,
//    GeLU, the float32 residual add, the head-interleaved Q/K/V scatter into
//    the KV cache, or the LM head's logits + argmax are applied (the fusions of
//    III.D);
//  * launched with programmatic stream serialization: the weight loads of the
//    first tile are issued before griddepcontrol.wait, so they overlap the tail
//    of the kernel that produces x;
//  * the grid is (row groups x token tiles) / w, w = the fewest waves the SMs
//    can hold, so every CTA gets w or w - 1 tasks and no partial last wave
//    leaves SMs idle;
//  * for one or two decode tokens the input LayerNorm (of the float32 residual)
//    can be fused: each CTA normalises the rows into shared memory once
//    ("DeepSpeed Inference", III.D, LN fused with the QKV / intermediate GeMM).
#include "common.cuh"
#include "kernels.h"
#include "tile_ops.cuh"

namespace bloom {

constexpr int kLinWarps = 8;
constexpr int kLinThreads = kLinWarps * kWarp;

// Output element e (0..3) of lane (g, q)'s accumulator tile mt: token m and
// weight row n.  Weights as the B operand (WA = false): 8 rows x 16 tokens;
// as the A operand (WA = true): 16 rows x 8 tokens.
template <bool WA>
__device__ __forceinline__ void tile_elem(int e, int mt, int m0, int row0, int g, int q, int &m,
                                          int &n) {
    if constexpr (WA) {
        m = m0 + mt * 8 + 2 * q + (e & 1);
        n = row0 + g + 8 * (e >> 1);
    } else {
        m = m0 + mt * 16 + g + 8 * (e >> 1);
        n = row0 + 2 * q + (e & 1);
    }
}

template <int MT, bool INT8, int EPI, bool LNF, bool WA>
__global__ void __launch_bounds__(kLinThreads) linear_kernel(const LinearArgs a) {
    constexpr int EPL = INT8 ? 16 : 8;   // weights per lane per chunk (16 bytes)
    constexpr int KC = 4 * EPL;          // k per chunk
    constexpr int NS = EPL / 4;          // mma k-steps per chunk
    constexpr int XW = EPL / 2;          // 32-bit words of x per lane per chunk
    constexpr int U = (MT >= 4) ? 2 : 4; // chunks in flight per warp
    constexpr int RG = WA ? 16 : 8;      // weight rows per task
    constexpr int TT = WA ? 8 * MT : 16 * MT;   // tokens per task
    constexpr int NR = WA ? 2 : 1;       // weight rows a lane loads (g, g + 8)
    // int8 as the A operand: weights a few batches ahead are pulled towards L2
    constexpr int PF = (WA && INT8) ? 2 : 0;

    extern __shared__ __align__(16) unsigned char xs[];   // LNF: [M][K*2 + 64] bf16
    __shared__ float red[kLinWarps][MT][4][kWarp];
    __shared__ unsigned long long s_best[EPI == EPI_ARGMAX ? kMaxBatch : 1];
    __shared__ float s_sum[3 * kLinWarps];
    __shared__ int s_last;

    griddep_launch();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, q = lane & 3;
    if constexpr (EPI == EPI_ARGMAX) {
        for (int i = threadIdx.x; i < a.M; i += blockDim.x) s_best[i] = 0ull;
    }

    const int nchunks = (a.K + KC - 1) / KC;
    const int row_groups = (a.N + RG - 1) / RG;
    const int tok_tiles = (a.M + TT - 1) / TT;
    const long long tasks = (long long)row_groups * tok_tiles;
    const size_t row_bytes = (size_t)a.K * (INT8 ? 1 : 2);
    const char *wbase = reinterpret_cast<const char *>(a.w);
    const int PX = a.K * 2 + 64;   // 64 mod 128: two rows' fragments hit disjoint banks
    bool waited = false;
    if constexpr (LNF) {
        // pull the first task's weight chunks towards L2 (they depend on no
        // earlier kernel), then wait for x and normalise its rows once
        if (blockIdx.x < tasks && q == 0) {
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                const int wrow = (int)(blockIdx.x / tok_tiles) * RG + g + 8 * r;
                if (wrow < a.N)
                    for (int c = warp; c < nchunks && c < 2 * U * kLinWarps; c += kLinWarps)
                        asm volatile("prefetch.global.L2 [%0];" ::"l"(
                            wbase + (size_t)wrow * row_bytes + (size_t)c * KC * (INT8 ? 1 : 2)));
            }
        }
        griddep_wait();
        waited = true;
        layernorm_rows_to_smem_shifted(a, xs, PX, s_sum, threadIdx.x, warp, lane);
    }

    for (long long task = blockIdx.x; task < tasks; task += gridDim.x) {
        const int rg = (int)(task / tok_tiles);
        const int tt = (int)(task - (long long)rg * tok_tiles);
        const int row0 = rg * RG, m0 = tt * TT;
        bool wok[NR];
        const char *wp[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            const int wrow = row0 + g + 8 * r;
            wok[r] = wrow < a.N;
            wp[r] = wbase + (size_t)(wok[r] ? wrow : 0) * row_bytes + (size_t)q * 16;
        }
        float acc[MT][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[mt][r] = 0.f;

        for (int c0 = warp; c0 < nchunks; c0 += kLinWarps * U) {
            uint4 wv[NR][U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + u * kLinWarps;
                const int k = c * KC + q * EPL;
#pragma unroll
                for (int r = 0; r < NR; ++r)
                    wv[r][u] = (wok[r] && c < nchunks && k < a.K)
                                   ? ld_stream(wp[r] + (size_t)c * KC * (INT8 ? 1 : 2))
                                   : make_uint4(0u, 0u, 0u, 0u);
            }
            if constexpr (PF > 0) {
                if (q == 0) {
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const int c = c0 + u * kLinWarps + PF * kLinWarps * U;
                        if (c < nchunks)
#pragma unroll
                            for (int r = 0; r < NR; ++r)
                                if (wok[r])
                                    asm volatile("prefetch.global.L2 [%0];" ::"l"(
                                        wp[r] + (size_t)c * KC * (INT8 ? 1 : 2)));
                    }
                }
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
                // activation fragments: tokens g (WA) or g, g + 8 of each tile
                uint32_t xa[MT][XW], xb[MT][WA ? 1 : XW];
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    const int ma = m0 + mt * (WA ? 8 : 16) + g, mb = ma + 8;
#pragma unroll
                    for (int hh = 0; hh < XW / 4; ++hh) {
                        uint4 va = make_uint4(0u, 0u, 0u, 0u), vb = va;
                        if constexpr (LNF) {
                            if (ma < a.M && k < a.K)
                                va = *reinterpret_cast<const uint4 *>(xs + (size_t)ma * PX +
                                                                      (size_t)(k + 8 * hh) * 2);
                            if (!WA && mb < a.M && k < a.K)
                                vb = *reinterpret_cast<const uint4 *>(xs + (size_t)mb * PX +
                                                                      (size_t)(k + 8 * hh) * 2);
                        } else {
                            if (ma < a.M && k < a.K) va = ld_act(a.x + (size_t)ma * a.K + k + 8 * hh);
                            if (!WA && mb < a.M && k < a.K)
                                vb = ld_act(a.x + (size_t)mb * a.K + k + 8 * hh);
                        }
                        xa[mt][4 * hh + 0] = va.x; xa[mt][4 * hh + 1] = va.y;
                        xa[mt][4 * hh + 2] = va.z; xa[mt][4 * hh + 3] = va.w;
                        if constexpr (!WA) {
                            xb[mt][4 * hh + 0] = vb.x; xb[mt][4 * hh + 1] = vb.y;
                            xb[mt][4 * hh + 2] = vb.z; xb[mt][4 * hh + 3] = vb.w;
                        }
                    }
                }
                const uint32_t w0[4] = {wv[0][u].x, wv[0][u].y, wv[0][u].z, wv[0][u].w};
                const uint32_t w1[4] = {wv[NR - 1][u].x, wv[NR - 1][u].y, wv[NR - 1][u].z,
                                        wv[NR - 1][u].w};
#pragma unroll
                for (int s = 0; s < NS; ++s) {
                    // the 16 bytes of row g (and g + 8) are the lane's fragment:
                    // words (2s, 2s+1), or int8 word s widened in two halves
                    uint32_t lo0, hi0, lo1, hi1;
                    if constexpr (INT8) {
                        lo0 = i8x2_to_bf16x2(w0[s], 0);
                        hi0 = i8x2_to_bf16x2(w0[s], 2);
                        lo1 = WA ? i8x2_to_bf16x2(w1[s], 0) : 0u;
                        hi1 = WA ? i8x2_to_bf16x2(w1[s], 2) : 0u;
                    } else {
                        lo0 = w0[2 * s];
                        hi0 = w0[2 * s + 1];
                        lo1 = w1[2 * s];
                        hi1 = w1[2 * s + 1];
                    }
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt) {
                        if constexpr (WA)
                            mma_bf16_16816(acc[mt], lo0, lo1, hi0, hi1, xa[mt][2 * s],
                                           xa[mt][2 * s + 1]);
                        else
                            mma_bf16_16816(acc[mt], xa[mt][2 * s], xb[mt][2 * s],
                                           xa[mt][2 * s + 1], xb[mt][2 * s + 1], lo0, hi0);
                    }
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
            for (int e = 0; e < 4; ++e) {
                int m, row;
                tile_elem<WA>(e, mt, m0, row0, g, q, m, row);
                if (m >= a.M || row >= a.N) continue;
                float v = d[e];
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
                    const int e2 = row % dh;
                    if (cidx == 0) {
                        a.q_out[(size_t)m * a.n_head * dh + (size_t)hj * dh + e2] = f2bf(v);
                    } else {
                        int seq, slot;
                        if (a.T > 0) {
                            const int i = m / a.T;
                            seq = a.row_map ? a.row_map[i] : i;
                            slot = m - i * a.T;
                        } else {
                            seq = m;
                            slot = a.len_ptr[m];
                            if (a.active && !a.active[m]) continue;   // idle row: no append
                        }
                        if (slot >= 0 && slot < a.max_seq) {
                            uint16_t *cache = (cidx == 1) ? a.k_cache : a.v_cache;
                            cache[(((size_t)seq * a.n_head + hj) * a.max_seq + slot) * dh + e2] =
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
                const bool act = !a.active || a.active[i];
                a.out_tokens[i] = act ? (int)unpack_index(p) : -1;
                if (a.len_inc && act) {
                    a.len_inc[i] += 1;
                    a.next_pos[i] += 1;
                }
            }
            if (threadIdx.x == 0) *a.ticket = 0;
        }
    }
}

template <int MT, bool INT8, int EPI, bool LNF, bool WA>
static int occupancy(size_t smem) {
    // cached per instance and dynamic shared-memory size (a few sizes per model)
    static size_t keys[8];
    static int vals[8];
    static int n = 0;
    for (int i = 0; i < n; ++i)
        if (keys[i] == smem) return vals[i];
    int o = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, linear_kernel<MT, INT8, EPI, LNF, WA>,
                                                      kLinThreads, smem) != cudaSuccess || o < 1)
        o = 1;
    if (n < 8) {
        keys[n] = smem;
        vals[n] = o;
        ++n;
    }
    return o;
}

template <int MT, bool INT8, int EPI, bool LNF, bool WA>
static cudaError_t launch_t(const LinearArgs &a, int num_sms, cudaStream_t s) {
    constexpr int RG = WA ? 16 : 8, TT = WA ? 8 * MT : 16 * MT;
    const size_t smem = LNF ? (size_t)a.M * (a.K * 2 + 64) : 0;
    const long long tasks = (long long)((a.N + RG - 1) / RG) * ((a.M + TT - 1) / TT);
    const long long cap = (long long)num_sms * occupancy<MT, INT8, EPI, LNF, WA>(smem);
    // the fewest waves the SMs can hold, then just enough CTAs for that many
    const long long waves = (tasks + cap - 1) / cap;
    long long blocks = (tasks + waves - 1) / waves;
    if (blocks < 1) blocks = 1;
    return launch_pdl_smem(linear_kernel<MT, INT8, EPI, LNF, WA>, dim3((unsigned)blocks),
                           dim3(kLinThreads), smem, s, a);
}

// Weights as the A operand (16-row tasks, MTA token tiles of 8) when those
// tasks fill at least one wave of the SMs: half the mma steps and half the
// activation fragments per weight byte, two rows' loads in flight per lane.
// Fewer, larger tasks lose when they leave SMs idle (4096-row matrices), so
// those keep the B-operand form (8-row tasks, MTB token tiles of 16); so do
// more than 32 tokens (MTA = 0).
template <int MTA, int MTB, bool INT8, int EPI, bool LNF>
static cudaError_t launch_o(const LinearArgs &a, int num_sms, cudaStream_t s) {
    if constexpr (MTA > 0) {
        const size_t smem = LNF ? (size_t)a.M * (a.K * 2 + 64) : 0;
        const long long cap = (long long)num_sms * occupancy<MTA, INT8, EPI, LNF, true>(smem);
        if ((a.N + 15) / 16 >= cap) return launch_t<MTA, INT8, EPI, LNF, true>(a, num_sms, s);
    }
    return launch_t<MTB, INT8, EPI, LNF, false>(a, num_sms, s);
}

template <int MTA, int MTB, bool INT8, bool LNF>
static cudaError_t launch_epi(const LinearArgs &a, int num_sms, cudaStream_t s) {
    switch (a.epi) {
        case EPI_STORE: return launch_o<MTA, MTB, INT8, EPI_STORE, LNF>(a, num_sms, s);
        case EPI_GELU: return launch_o<MTA, MTB, INT8, EPI_GELU, LNF>(a, num_sms, s);
        case EPI_RESID: return launch_o<MTA, MTB, INT8, EPI_RESID, LNF>(a, num_sms, s);
        case EPI_RESID32: return launch_o<MTA, MTB, INT8, EPI_RESID32, LNF>(a, num_sms, s);
        case EPI_QKV: return launch_o<MTA, MTB, INT8, EPI_QKV, LNF>(a, num_sms, s);
        case EPI_ARGMAX:
            if constexpr (!INT8) return launch_o<MTA, MTB, false, EPI_ARGMAX, LNF>(a, num_sms, s);
            return cudaErrorInvalidValue;
        default: return cudaErrorInvalidValue;
    }
}

template <bool INT8, bool LNF>
static cudaError_t launch_mt(const LinearArgs &a, int num_sms, cudaStream_t s) {
    if (a.M <= 8) return launch_epi<1, 1, INT8, LNF>(a, num_sms, s);
    if (a.M <= 16) return launch_epi<2, 1, INT8, LNF>(a, num_sms, s);
    if (a.M <= 32) return launch_epi<4, 2, INT8, LNF>(a, num_sms, s);
    return launch_epi<0, 4, INT8, LNF>(a, num_sms, s);
}

template <bool INT8, int EPI, bool WA>
static cudaError_t prepare_mt_o() {
    occupancy<1, INT8, EPI, false, WA>(0);
    occupancy<2, INT8, EPI, false, WA>(0);
    occupancy<4, INT8, EPI, false, WA>(0);
    // only the fused-LayerNorm instance (one token tile) uses dynamic shared memory
    return cudaFuncSetAttribute(linear_kernel<1, INT8, EPI, true, WA>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, kLnFuseSmemMax);
}

template <bool INT8, int EPI>
static cudaError_t prepare_mt() {
    const cudaError_t e = prepare_mt_o<INT8, EPI, false>();
    return e ? e : prepare_mt_o<INT8, EPI, true>();
}

// Occupancies and shared-memory limits of every instance, outside any capture.
cudaError_t linear_prepare() {
    cudaError_t e;
    if ((e = prepare_mt<false, EPI_STORE>())) return e;
    if ((e = prepare_mt<false, EPI_GELU>())) return e;
    if ((e = prepare_mt<false, EPI_RESID>())) return e;
    if ((e = prepare_mt<false, EPI_RESID32>())) return e;
    if ((e = prepare_mt<false, EPI_QKV>())) return e;
    if ((e = prepare_mt<false, EPI_ARGMAX>())) return e;
    if ((e = prepare_mt<true, EPI_STORE>())) return e;
    if ((e = prepare_mt<true, EPI_GELU>())) return e;
    if ((e = prepare_mt<true, EPI_RESID>())) return e;
    if ((e = prepare_mt<true, EPI_RESID32>())) return e;
    return prepare_mt<true, EPI_QKV>();
}

bool linear_can_fuse_ln(const LinearArgs &a) {
    return a.T == 0 && a.M >= 1 && a.M <= kLnFuseMaxM &&
           (size_t)a.M * (a.K * 2 + 64) <= (size_t)kLnFuseSmemMax &&
           !(a.int8 && a.epi == EPI_ARGMAX);
}

cudaError_t launch_linear(const LinearArgs &a, int num_sms, cudaStream_t s) {
    if (a.M <= 0 || a.N <= 0) return cudaSuccess;
    if (a.epi == EPI_ARGMAX && (a.int8 || a.M > kMaxBatch)) return cudaErrorInvalidValue;
    if (a.ln_x) {
        if (!linear_can_fuse_ln(a)) return cudaErrorInvalidValue;
        return a.int8 ? launch_epi<1, 1, true, true>(a, num_sms, s)
                      : launch_epi<1, 1, false, true>(a, num_sms, s);
    }
    return a.int8 ? launch_mt<true, false>(a, num_sms, s) : launch_mt<false, false>(a, num_sms, s);
}

}  // namespace bloom
