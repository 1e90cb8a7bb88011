// Prefill attention on the tensor cores (sm_103a): causal, pad-masked ALiBi
// attention of every prompt slot, as tiles of queries against tiles of keys.
//
// Score of key k for query t of head j: s = (q_t . k_k) / sqrt(d) + slope_j * pos_k,
// for keys k <= t that are tokens (pos_k >= 0); other keys take no part (their
// probability is exactly 0).  That is the masked_fill + float32 softmax of
// "Hugging Face BLOOM Inference Optimization" (Custom CUDA Kernels); the
// probabilities are then rounded to bf16 for the product with V, as that fused
// kernel hands its float32 softmax back in the activations' type.
//
// One CTA takes 64 queries of one (sequence, head), 16 per warp, and walks the
// key tiles of 64 that causality lets them see (the pages' batched-GeMM form of
// attention, "DeepSpeed Inference", III.D, on the tensor cores):
//  * Q, K and V tiles sit in shared memory with a 16-byte-chunk XOR swizzle
//    (chunk c of row r at c ^ (r & 7)), so the ldmatrix fragment loads of eight
//    rows hit eight different bank groups; K / V / position tiles of the next
//    key tile are copied (cp.async, zero-filled past the prompt) while the
//    current one is computed;
//  * S = Q K^T on mma.sync m16n8k16 (bf16 in, float32 accumulate); scale, ALiBi
//    bias and masks applied in registers; an online softmax (running max and
//    sum per row, the sum reduced over the row's four lanes only at the end);
//  * O += P V on the same instruction, P taken straight from the S registers
//    (the accumulator layout of two 8-key blocks is the A-operand layout of one
//    16-key step), V fragments by a transposing ldmatrix.
// A query at a pad slot has no defined output; the kernel writes zeros there.
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "tile_ops.cuh"

namespace bloom {

constexpr int kFaQ = 64;        // queries per CTA
constexpr int kFaK = 64;        // keys per tile
constexpr int kFaThreads = 128; // 4 warps x 16 queries

template <int D>
struct FaSmem {
    static constexpr int Row = D * 2;               // bytes per row
    static constexpr int Tile = kFaK * Row;         // one Q / K / V tile
    static constexpr int Q = 0;
    static constexpr int K0 = Tile;                 // K tiles [2]
    static constexpr int V0 = 3 * Tile;             // V tiles [2]
    static constexpr int P0 = 5 * Tile;             // positions [2][64] int
    static constexpr int Bytes = 5 * Tile + 2 * kFaK * 4;
};

// Byte offset of 16-byte chunk c of row r in a swizzled tile.
template <int D>
__device__ __forceinline__ uint32_t fa_off(int r, int c) {
    return (uint32_t)(r * (D * 2) + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
// 16-byte asynchronous copy that reads `valid` ? 16 : 0 bytes and zero-fills the rest.
__device__ __forceinline__ void cp16(uint32_t dst, const void *src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}

// The same for 4 bytes.
__device__ __forceinline__ void cp4(uint32_t dst, const void *src, bool valid) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src),
                 "r"(valid ? 4 : 0)
                 : "memory");
}

template <int D>
__global__ void __launch_bounds__(kFaThreads) attn_prefill_tc_kernel(const AttnPrefillArgs a) {
    using L = FaSmem<D>;
    constexpr int CH = D / 8;    // 16-byte chunks per row
    constexpr int NJ = D / 8;    // 8-wide output column blocks
    extern __shared__ __align__(128) unsigned char fsm[];
    griddep_launch();
    griddep_wait();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, q4 = lane & 3;
    // the longest query tiles (most key tiles) first
    const int qt = gridDim.x - 1 - blockIdx.x;
    const int j = blockIdx.y, b = blockIdx.z;   // head, prompt
    const int q0 = qt * kFaQ;
    const int T = a.T;
    const int row = a.row_map ? a.row_map[b] : b;   // the prompt's cache row
    const size_t bh = (size_t)row * a.n + j;
    const uint16_t *kb = a.k + bh * a.max_seq * D;
    const uint16_t *vb = a.v + bh * a.max_seq * D;
    const int *posb = a.pos + (size_t)row * a.max_seq;
    const float slope = a.slopes[j];
    const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(fsm);
    int *spos = reinterpret_cast<int *>(fsm + L::P0);

    // ---- Q tile (rows past the prompt zero-filled), key tile 0
    for (int i = tid; i < kFaQ * CH; i += kFaThreads) {
        const int r = i / CH, c = i % CH;
        const int t = q0 + r;
        const uint16_t *src = a.q + ((size_t)(b * T + (t < T ? t : 0)) * a.n + j) * D + c * 8;
        cp16(sbase + L::Q + fa_off<D>(r, c), src, t < T);
    }
    const int kend = min(q0 + kFaQ, T);          // keys [0, kend) can be seen
    const int ntiles = (kend + kFaK - 1) / kFaK;
    auto load_kv = [&](int kt, int buf) {
        for (int i = tid; i < kFaK * CH; i += kFaThreads) {
            const int r = i / CH, c = i % CH;
            const int key = kt * kFaK + r;
            const bool ok = key < T;
            const size_t off = (size_t)(ok ? key : 0) * D + c * 8;
            cp16(sbase + L::K0 + buf * L::Tile + fa_off<D>(r, c), kb + off, ok);
            cp16(sbase + L::V0 + buf * L::Tile + fa_off<D>(r, c), vb + off, ok);
        }
        if (tid < kFaK) {   // one position per 4-byte copy (a row need not be 16-byte aligned)
            const int key = kt * kFaK + tid;
            cp4(sbase + L::P0 + (buf * kFaK + tid) * 4, posb + (key < T ? key : 0), key < T);
        }
    };
    load_kv(0, 0);
    cp_async_commit();

    // ---- this warp's 16 queries
    const int qw = 16 * warp;
    uint32_t qa[D / 16][4];
    float o[NJ][4];
#pragma unroll
    for (int n = 0; n < NJ; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
    const int tq[2] = {q0 + qw + g, q0 + qw + g + 8};

    for (int kt = 0; kt < ntiles; ++kt) {
        const int buf = kt & 1;
        cp_async_wait<0>();
        __syncthreads();   // tile kt (and Q) landed for all; buffer buf ^ 1 is free
        if (kt + 1 < ntiles) {
            load_kv(kt + 1, buf ^ 1);
            cp_async_commit();
        }
        if (kt == 0) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const int r = qw + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int c = 2 * kk + (lane >> 4);
                ldsm_x4(sbase + L::Q + fa_off<D>(r, c), qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
            }
        }
        // a tile entirely after this warp's last query adds nothing
        if (kt * kFaK > q0 + qw + 15) continue;
        // ---- S = Q K^T: 8 blocks of 8 keys
        float sc[8][4];
#pragma unroll
        for (int nb = 0; nb < 8; ++nb) {
            sc[nb][0] = sc[nb][1] = sc[nb][2] = sc[nb][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < D / 16; kk += 2) {
                uint32_t b0, b1, b2, b3;
                const int r = nb * 8 + (lane & 7);
                const int c = 2 * kk + (lane >> 3);
                ldsm_x4(sbase + L::K0 + buf * L::Tile + fa_off<D>(r, c), b0, b1, b2, b3);
                mma_bf16_16816(sc[nb], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
                mma_bf16_16816(sc[nb], qa[kk + 1][0], qa[kk + 1][1], qa[kk + 1][2], qa[kk + 1][3],
                               b2, b3);
            }
        }
        // ---- scale, ALiBi bias, masks; online softmax
        const int *tpos = spos + buf * kFaK;
        float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int nb = 0; nb < 8; ++nb)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int kl = nb * 8 + 2 * q4 + (e & 1);
                const int key = kt * kFaK + kl;
                const int h = e >> 1;
                const int pk = tpos[kl];
                const bool valid = key <= tq[h] && key < T && pk >= 0;
                const float s = valid ? sc[nb][e] * a.scale + slope * (float)pk : -INFINITY;
                sc[nb][e] = s;
                tmax[h] = fmaxf(tmax[h], s);
            }
        float corr[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            tmax[h] = fmaxf(tmax[h], __shfl_xor_sync(0xffffffffu, tmax[h], 1));
            tmax[h] = fmaxf(tmax[h], __shfl_xor_sync(0xffffffffu, tmax[h], 2));
            const float mn = fmaxf(mrow[h], tmax[h]);
            corr[h] = (mrow[h] == -INFINITY) ? 0.f : expf(mrow[h] - mn);
            mrow[h] = mn;
            lrow[h] *= corr[h];
        }
#pragma unroll
        for (int n = 0; n < NJ; ++n) {
            o[n][0] *= corr[0];
            o[n][1] *= corr[0];
            o[n][2] *= corr[1];
            o[n][3] *= corr[1];
        }
#pragma unroll
        for (int nb = 0; nb < 8; ++nb)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int h = e >> 1;
                const float p = (sc[nb][e] == -INFINITY) ? 0.f : expf(sc[nb][e] - mrow[h]);
                sc[nb][e] = p;
                lrow[h] += p;
            }
        // ---- O += P V: 4 steps of 16 keys
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            const uint32_t pa0 = pack_bf2(sc[2 * ks][0], sc[2 * ks][1]);
            const uint32_t pa1 = pack_bf2(sc[2 * ks][2], sc[2 * ks][3]);
            const uint32_t pa2 = pack_bf2(sc[2 * ks + 1][0], sc[2 * ks + 1][1]);
            const uint32_t pa3 = pack_bf2(sc[2 * ks + 1][2], sc[2 * ks + 1][3]);
#pragma unroll
            for (int n = 0; n < NJ; n += 2) {
                uint32_t b0, b1, b2, b3;
                const int r = 16 * ks + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int c = n + (lane >> 4);
                ldsm_x4_t(sbase + L::V0 + buf * L::Tile + fa_off<D>(r, c), b0, b1, b2, b3);
                mma_bf16_16816(o[n], pa0, pa1, pa2, pa3, b0, b1);
                mma_bf16_16816(o[n + 1], pa0, pa1, pa2, pa3, b2, b3);
            }
        }
    }
    // ---- normalise and store (rows g and g + 8 of this warp; pad queries -> 0)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        float l = lrow[h];
        l += __shfl_xor_sync(0xffffffffu, l, 1);
        l += __shfl_xor_sync(0xffffffffu, l, 2);
        const int t = tq[h];
        if (t >= T) continue;
        const bool qok = posb[t] >= 0 && l > 0.f;
        const float inv = qok ? 1.f / l : 0.f;
        uint16_t *dst = a.o + ((size_t)(b * T + t) * a.n + j) * D + 2 * q4;
#pragma unroll
        for (int n = 0; n < NJ; ++n)
            *reinterpret_cast<uint32_t *>(dst + n * 8) =
                pack_bf2(o[n][2 * h] * inv, o[n][2 * h + 1] * inv);
    }
}

cudaError_t attn_prefill_tc_prepare() {
    cudaError_t e = cudaFuncSetAttribute(attn_prefill_tc_kernel<64>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         FaSmem<64>::Bytes);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(attn_prefill_tc_kernel<128>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, FaSmem<128>::Bytes);
}

cudaError_t launch_attn_prefill_tc(const AttnPrefillArgs &a, cudaStream_t s) {
    if (a.T <= 0) return cudaSuccess;
    static bool prepared = false;
    if (!prepared) {
        cudaError_t e = attn_prefill_tc_prepare();
        if (e != cudaSuccess) return e;
        prepared = true;
    }
    dim3 grid((a.T + kFaQ - 1) / kFaQ, a.n, a.B);
    if (a.d == 64)
        return launch_pdl_smem(attn_prefill_tc_kernel<64>, grid, dim3(kFaThreads), FaSmem<64>::Bytes,
                               s, a);
    if (a.d == 128)
        return launch_pdl_smem(attn_prefill_tc_kernel<128>, grid, dim3(kFaThreads),
                               FaSmem<128>::Bytes, s, a);
    return cudaErrorInvalidValue;
}

}  // namespace bloom
