// Persistent decode step: the whole token step -- embedding, every decoder
// layer, ln_f and the LM head with its argmax -- as one cooperative launch with
// one 8-warp block per SM.
//
// At small batch a decode step is the time to read every weight once
// ("DeepSpeed Inference", III.A), but a step of one kernel per operation pays
// a ramp-up and a tail at each of the ~7 launches per layer, during which HBM
// idles (CUDA graphs, III.D, remove the CPU side of that cost, not the GPU
// side).  Here the operations become phases of one kernel separated by grid
// barriers, and the weight stream does not stop at a barrier:
//
//  * every lane streams its 16-byte weight fragments (the mma.sync B fragment
//    binding of the weight-streaming linear kernel) through a private ring in
//    shared memory with cp.async: 8 batches of 4 chunks, one cp.async group
//    per batch.  The ring is filled ahead in the order the lane will consume
//    it, across phase boundaries: while a block waits at a barrier, or runs a
//    LayerNorm or attention phase, the loads of the next linear phase's
//    weights are already in flight;
//  * the weights do not depend on the activations, so nothing but the small
//    activation vectors waits for a barrier;
//  * activations written by other blocks in an earlier phase are read with
//    coherent loads (never the non-coherent path); the barrier's
//    release / acquire fences order them;
//  * linear phases split the weight rows in groups of 8 over the blocks
//    (strided) and K over the 8 warps, reduce through shared memory and apply
//    the same fused epilogues as the per-launch kernel (Q/K/V scatter into the
//    cache, GeLU, float32 residual add, LM-head argmax);
//  * LayerNorm, embedding and attention phases reuse the per-launch kernels'
//    block-level device functions.
// Every barrier wait is bounded (about two seconds of SM clock): on expiry the
// block records kErrTimeout in the device flag, raises an abort flag that
// every other waiting block sees, waits for its own copies in flight, and
// returns.  The last block to exit leaves the barrier words at zero.
#include "attn_ops.cuh"
#include "common.cuh"
#include "kernels.h"
#include "norm_ops.cuh"
#include "tile_ops.cuh"

namespace bloom {

constexpr int kPWarps = 8;
constexpr int kPThreads = kPWarps * kWarp;
constexpr int kPU = 4;                        // chunks per batch (one cp.async group)
constexpr int kPNB = 8;                       // batches in a warp's ring
constexpr int kPChunk = kWarp * 16;           // bytes of one warp chunk (16 per lane)
constexpr int kPRingBytes = kPWarps * kPNB * kPU * kPChunk;   // 128 KB
constexpr long long kPWaitCycles = 4000000000ll;

static_assert(kLnThreads == kPThreads, "LayerNorm rows are normalised by one whole block");

__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                     (uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// Activations written by other blocks of this launch: coherent (L1-cached,
// invalidated by the barrier's acquire fence), never ld.global.nc.
__device__ __forceinline__ uint4 ld_coherent(const void *p) {
    return *reinterpret_cast<const uint4 *>(p);
}

// Position of a warp in its weight stream: phase, task (row group), batch.
struct Cursor {
    int p, t, b;
};

// Moves c to the next batch this block streams (c itself if it is one).
__device__ __forceinline__ void cursor_settle(const PersistArgs &pa, Cursor &c) {
    while (c.p < pa.nphases) {
        const PersistPhase &ph = pa.phases[c.p];
        if (ph.kind == PH_LINEAR) {
            if (c.b >= ph.nbt) {
                c.b = 0;
                c.t += gridDim.x;
            }
            if (c.t < ph.tasks) return;
        }
        ++c.p;
        c.t = blockIdx.x;
        c.b = 0;
    }
}

// Issue the cp.async copies of the batch at c into this lane's ring slot
// (one group, possibly empty), then advance c.
__device__ __forceinline__ void issue_batch(const PersistArgs &pa, Cursor &c, unsigned char *slot,
                                            int warp, int lane) {
    if (c.p < pa.nphases) {
        const PersistPhase &ph = pa.phases[c.p];
        const LinearArgs &a = ph.lin;
        const int eb = a.int8 ? 1 : 2;
        const int epl = 16 / eb, kc = 4 * epl;
        const int g = lane >> 2, q = lane & 3;
        const int row = c.t * 8 + g;
        const char *wrow = reinterpret_cast<const char *>(a.w) + (size_t)row * a.K * eb;
#pragma unroll
        for (int u = 0; u < kPU; ++u) {
            const int ch = warp + kPWarps * (c.b * kPU + u);
            const int k = ch * kc + q * epl;
            if (row < a.N && ch < ph.nchunks && k < a.K)
                cp_async16(slot + u * kPChunk + lane * 16, wrow + (size_t)k * eb);
        }
        ++c.b;
        cursor_settle(pa, c);
    }
    cp_async_commit();
}

// Grid-wide barrier number `idx` (0-based) of this launch.  Returns false if
// the launch is aborting.
__device__ __forceinline__ bool grid_barrier(const PersistArgs &pa, unsigned idx, int *s_flag) {
    __syncthreads();
    if (threadIdx.x == 0) {
        int ok = 1;
        const unsigned target = gridDim.x * (idx + 1);
        __threadfence();   // release this block's writes
        atomicAdd(pa.bar, 1u);
        const long long t0 = clock64();
        for (unsigned spin = 0;; ++spin) {
            unsigned v;
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(pa.bar) : "memory");
            if (v >= target) break;
            if (*reinterpret_cast<volatile unsigned *>(pa.bar + 2)) {
                ok = 0;
                break;
            }
            if ((spin & 31u) == 31u && clock64() - t0 > kPWaitCycles) {
                atomicOr(pa.err, kErrTimeout);
                atomicExch(pa.bar + 2, 1u);
                ok = 0;
                break;
            }
            __nanosleep(20);
        }
        __threadfence();   // acquire: later loads see the other blocks' writes
        *s_flag = ok;
    }
    __syncthreads();
    return *s_flag != 0;
}

// One linear phase: this block's row groups, K split over the warps, every
// weight fragment taken from the lane's ring slot.
template <bool INT8>
__device__ __forceinline__ void linear_phase(const PersistArgs &pa, const PersistPhase &ph,
                                             unsigned char *ring, Cursor &prod, unsigned &seq,
                                             float (*red)[kPWarps][4][kWarp], int &par,
                                             unsigned long long *s_best, int *s_last) {
    constexpr int EPL = INT8 ? 16 : 8;
    constexpr int KC = 4 * EPL;
    constexpr int NS = EPL / 4;
    constexpr int XW = EPL / 2;
    const LinearArgs &a = ph.lin;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, q = lane & 3;
    const int M = a.M, N = a.N, K = a.K, epi = a.epi;
    const uint16_t *x = a.x;
    unsigned char *wring = ring + (size_t)warp * kPNB * kPU * kPChunk;

    if (epi == EPI_ARGMAX) {
        for (int i = threadIdx.x; i < M; i += blockDim.x) s_best[i] = 0ull;
        __syncthreads();
    }
    for (int t = blockIdx.x; t < ph.tasks; t += gridDim.x) {
        const int row0 = t * 8;
        const bool wok = row0 + g < N;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int bt = 0; bt < ph.nbt; ++bt) {
            cp_async_wait<kPNB - 1>();   // this lane's batch `seq` has landed
            unsigned char *slot = wring + (size_t)(seq % kPNB) * kPU * kPChunk + lane * 16;
#pragma unroll
            for (int u = 0; u < kPU; ++u) {
                const int ch = warp + kPWarps * (bt * kPU + u);
                if (ch >= ph.nchunks) break;   // warp-uniform
                const int k = ch * KC + q * EPL;
                const bool kok = k < K;
                uint4 wv = make_uint4(0u, 0u, 0u, 0u);
                if (wok && kok) wv = *reinterpret_cast<const uint4 *>(slot + u * kPChunk);
                uint32_t xa[XW], xb[XW];
#pragma unroll
                for (int hh = 0; hh < XW / 4; ++hh) {
                    uint4 va = make_uint4(0u, 0u, 0u, 0u), vb = va;
                    if (g < M && kok) va = ld_coherent(x + (size_t)g * K + k + 8 * hh);
                    if (g + 8 < M && kok) vb = ld_coherent(x + (size_t)(g + 8) * K + k + 8 * hh);
                    xa[4 * hh + 0] = va.x; xa[4 * hh + 1] = va.y;
                    xa[4 * hh + 2] = va.z; xa[4 * hh + 3] = va.w;
                    xb[4 * hh + 0] = vb.x; xb[4 * hh + 1] = vb.y;
                    xb[4 * hh + 2] = vb.z; xb[4 * hh + 3] = vb.w;
                }
                const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
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
                    mma_bf16_16816(acc, xa[2 * s], xb[2 * s], xa[2 * s + 1], xb[2 * s + 1], b0, b1);
                }
            }
            // the slot is consumed: refill it with the batch kPNB ahead
            issue_batch(pa, prod, wring + (size_t)(seq % kPNB) * kPU * kPChunk, warp, lane);
            ++seq;
        }
        // sum the 8 warps' partial tiles (double-buffered: one barrier per task)
#pragma unroll
        for (int r = 0; r < 4; ++r) red[par][warp][r][lane] = acc[r];
        __syncthreads();
        if (warp == 0) {
            float d[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                float s = 0.f;
#pragma unroll
                for (int w = 0; w < kPWarps; ++w) s += red[par][w][r][lane];
                d[r] = s;
            }
            switch (epi) {
                case EPI_QKV: tile_epilogue<INT8, EPI_QKV>(a, d, 0, row0, lane, s_best); break;
                case EPI_RESID32: tile_epilogue<INT8, EPI_RESID32>(a, d, 0, row0, lane, s_best); break;
                case EPI_GELU: tile_epilogue<INT8, EPI_GELU>(a, d, 0, row0, lane, s_best); break;
                case EPI_STORE: tile_epilogue<INT8, EPI_STORE>(a, d, 0, row0, lane, s_best); break;
                case EPI_RESID: tile_epilogue<INT8, EPI_RESID>(a, d, 0, row0, lane, s_best); break;
                case EPI_ARGMAX: tile_epilogue<INT8, EPI_ARGMAX>(a, d, 0, row0, lane, s_best); break;
                default: break;
            }
        }
        par ^= 1;
    }
    if (epi == EPI_ARGMAX) argmax_publish(a, s_best, s_last, threadIdx.x, gridDim.x);
}

template <bool INT8>
__global__ void __launch_bounds__(kPThreads, 1) decode_persistent_kernel(const PersistArgs pa) {
    extern __shared__ __align__(16) unsigned char ring[];   // kPRingBytes
    __shared__ float red[2][kPWarps][4][kWarp];
    __shared__ unsigned long long s_best[kMaxBatch];
    __shared__ float s_ln[kLnWarps];
    __shared__ int s_flag, s_last;
    __shared__ __align__(16) unsigned char s_attn[sizeof(AttnSmem<128, kPThreads>)];

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned char *wring = ring + (size_t)warp * kPNB * kPU * kPChunk;

    // fill the ring: the first kPNB batches of this warp's weight stream
    Cursor prod = {0, (int)blockIdx.x, 0};
    cursor_settle(pa, prod);
    for (int i = 0; i < kPNB; ++i) issue_batch(pa, prod, wring + (size_t)i * kPU * kPChunk, warp, lane);
    unsigned seq = 0;
    int par = 0;
    unsigned nbar = 0;
    bool ok = true;

    for (int p = 0; p < pa.nphases && ok; ++p) {
        const PersistPhase &ph = pa.phases[p];
        if (ph.kind == PH_LINEAR) {
            if (ph.lin.int8) {
                if constexpr (INT8)
                    linear_phase<true>(pa, ph, ring, prod, seq, red, par, s_best, &s_last);
            } else {
                linear_phase<false>(pa, ph, ring, prod, seq, red, par, s_best, &s_last);
            }
        } else if (ph.kind == PH_LN) {
            for (int r = blockIdx.x; r < ph.rows; r += gridDim.x)
                ln_row(ph.ln_src + (size_t)r * ph.h, ph.g, ph.b, ph.h, ph.eps,
                       ph.ln_dst + (size_t)r * ph.h, s_ln);
        } else if (ph.kind == PH_EMBED) {
            for (int r = blockIdx.x; r < ph.rows; r += gridDim.x) {
                int tok = ph.tokens[r];
                if (tok < 0 || tok >= ph.vocab) {
                    if (threadIdx.x == 0) atomicOr(pa.err, kErrToken);
                    tok = 0;
                }
                if (threadIdx.x == 0) {
                    const int slot = *ph.len;
                    if (slot >= 0 && slot < ph.max_seq)
                        ph.pos[(size_t)r * ph.max_seq + slot] = ph.next_pos[r];
                    else
                        atomicOr(pa.err, kErrSlot);
                }
                ln_row(ph.emb + (size_t)tok * ph.h, ph.g, ph.b, ph.h, ph.eps,
                       ph.emb_dst + (size_t)r * ph.h, s_ln);
            }
        } else if (ph.kind == PH_ATTN) {
            const AttnDecodeArgs &at = ph.at;
            const int units = at.B * at.n * at.splits;
            for (int u = blockIdx.x; u < units; u += gridDim.x) {
                const int split = u % at.splits, j = (u / at.splits) % at.n;
                const int b = u / (at.splits * at.n);
                if (at.d == 64)
                    attn_decode_block<64, kPThreads>(
                        at, split, j, b, *reinterpret_cast<AttnSmem<64, kPThreads> *>(s_attn));
                else
                    attn_decode_block<128, kPThreads>(
                        at, split, j, b, *reinterpret_cast<AttnSmem<128, kPThreads> *>(s_attn));
            }
        }
        if (p + 1 < pa.nphases) ok = grid_barrier(pa, nbar++, &s_flag);
    }

    cp_async_wait_all();   // no copy of this block may land after it exits
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(pa.bar + 1, 1u) == gridDim.x - 1) {
            // every block has left every barrier: reset for the next launch
            pa.bar[0] = 0u;
            pa.bar[2] = 0u;
            __threadfence();
            pa.bar[1] = 0u;
        }
    }
}

// ---------------------------------------------------------------- host side
void persist_linear_geometry(PersistPhase &ph) {
    const LinearArgs &a = ph.lin;
    const int kc = a.int8 ? 64 : 32;
    ph.tasks = (a.N + 7) / 8;
    ph.nchunks = (a.K + kc - 1) / kc;
    const int per_warp = (ph.nchunks + kPWarps - 1) / kPWarps;
    ph.nbt = (per_warp + kPU - 1) / kPU;
    if (ph.nbt < 1) ph.nbt = 1;
}

cudaError_t persist_prepare() {
    cudaError_t e = cudaFuncSetAttribute(decode_persistent_kernel<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kPRingBytes);
    if (e) return e;
    return cudaFuncSetAttribute(decode_persistent_kernel<true>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, kPRingBytes);
}

int persist_grid(int int8) {
    int dev = 0, sms = 0, coop = 0, per_sm = 0;
    if (cudaGetDevice(&dev) || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) ||
        cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev))
        return 0;
    if (!coop || persist_prepare()) return 0;
    const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &per_sm, int8 ? decode_persistent_kernel<true> : decode_persistent_kernel<false>,
        kPThreads, kPRingBytes);
    if (e || per_sm < 1) return 0;
    return sms;   // one block per SM
}

cudaError_t launch_decode_persistent(const PersistArgs &pa, int int8, int grid, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kPThreads);
    cfg.dynamicSmemBytes = kPRingBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (int8) return cudaLaunchKernelEx(&cfg, decode_persistent_kernel<true>, pa);
    return cudaLaunchKernelEx(&cfg, decode_persistent_kernel<false>, pa);
}

}  // namespace bloom
