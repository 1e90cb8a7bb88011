// Prefill GEMM on the 5th-generation tensor cores (tcgen05 + TMEM + TMA), sm_103a.
//
// Y[m][n] = epilogue(sum_k X[m][k] W[n][k]) for the B*T prompt tokens of a
// prefill: the linear layers there are real dense contractions (compute-bound,
// "DeepSpeed Inference", III.A / IV.C.1: prompt processing saturates compute),
// so they run as 128 x 256 output tiles on the tensor cores instead of
// streaming the weights per token tile.
//
// One CTA per SM walks the 128 (tokens) x 256 (features) output tiles
// (persistent), with two accumulators in TMEM so that the epilogue of one tile
// overlaps the main loop of the next:
//  * warp 0, one lane: TMA producer.  Two 2-D tensor maps (128B swizzle) move
//    a 128 x 64 tile of X and a 256 x 64 tile of W per k-block into a 4-stage
//    shared-memory ring, completing an mbarrier per stage;
//  * warp 1, one lane: issues tcgen05.mma (kind::f16, bf16 x bf16 -> f32,
//    M = 128, N = 256, K = 16 per instruction, 4 per k-block) into one of two
//    TMEM accumulators of 256 columns (the SM's 512), once the epilogue has
//    drained it; tcgen05.commit frees each stage when its MMAs are done and
//    signals each tile's accumulator complete;
//  * warps 2-5: epilogue.  Each warp reads its 32-lane quarter of the
//    accumulator with tcgen05.ld (lane = token row, 32 columns at a time),
//    adds the bias and applies GeLU, the float32 residual add or the
//    head-interleaved Q/K/V scatter into the KV cache ("DeepSpeed Inference",
//    III.D fusions), stores, and hands the accumulator back to the MMA lane.
// Warp 0 also allocates and frees the TMEM columns.  Every wait is bounded
// (about two seconds of SM clock); on expiry the kernel records kErrTimeout,
// skips its stores, and still frees TMEM.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_ops.cuh"

namespace bloom {

constexpr int kTcBM = 128;          // tokens per tile (MMA M)
constexpr int kTcBN = 256;          // features per tile (MMA N)
constexpr int kTcBK = 64;           // k per stage: 64 bf16 = one 128-byte swizzle row
constexpr int kTcStages = 4;
constexpr int kTcThreads = 192;     // 6 warps
constexpr int kTcABytes = kTcBM * kTcBK * 2;     // 16 KB
constexpr int kTcBBytes = kTcBN * kTcBK * 2;     // 32 KB
constexpr int kTcStageBytes = kTcABytes + kTcBBytes;
constexpr size_t kTcSmem = (size_t)kTcStages * kTcStageBytes + 1024;   // + 1 KB alignment slack
// Epilogue of 32 consecutive features [nb, nb + 32) of token row m (v = the
// accumulators; bias: those features' bias in shared memory, or null);
// features >= a.N are dropped.
template <int EPI>
__device__ __forceinline__ void tc_store_chunk(const LinearArgs &a, float (&v)[32], int m, int nb,
                                               const uint16_t *bias, const float (&res)[32]) {
    const int nv = min(32, a.N - nb);
    if (bias) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] += bf2f(bias[i]);
    }
    if constexpr (EPI == EPI_GELU) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = gelu_tanh(v[i]);
    }
    if constexpr (EPI == EPI_RESID32) {
        // res: the residual of these features, loaded a chunk ahead (tc_load_res)
        float *o = a.out32 + (size_t)m * a.N + nb;
        if (nv == 32 && ((uintptr_t)o & 15u) == 0) {
#pragma unroll
            for (int i = 0; i < 32; i += 4)
                *reinterpret_cast<float4 *>(o + i) =
                    make_float4(res[i] + v[i], res[i + 1] + v[i + 1], res[i + 2] + v[i + 2],
                                res[i + 3] + v[i + 3]);
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (i < nv) o[i] = res[i] + v[i];
        }
    } else {
        uint16_t *o;
        if constexpr (EPI == EPI_QKV) {
            // 32 consecutive features lie inside one head's q, k or v (d % 32 == 0)
            const int dh = a.head_dim;
            const int hj = nb / (3 * dh);
            const int cidx = (nb / dh) % 3;
            const int e0 = nb % dh;
            if (cidx == 0) {
                o = a.q_out + (size_t)m * a.n_head * dh + (size_t)hj * dh + e0;
            } else {
                const int i = m / a.T, slot = m - i * a.T;
                const int seq = a.row_map ? a.row_map[i] : i;   // the prompt's cache row
                if (slot >= a.max_seq) {
                    if (a.err) atomicOr(a.err, kErrSlot);
                    return;
                }
                uint16_t *cache = (cidx == 1) ? a.k_cache : a.v_cache;
                o = cache + (((size_t)seq * a.n_head + hj) * a.max_seq + slot) * dh + e0;
            }
        } else {
            o = a.out + (size_t)m * a.N + nb;
        }
        if constexpr (EPI == EPI_RESID) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (i < nv) v[i] += bf2f(o[i]);
        }
        if (nv == 32 && ((uintptr_t)o & 15u) == 0) {
#pragma unroll
            for (int i = 0; i < 32; i += 8) {
                uint4 p;
                p.x = pack_bf2(v[i], v[i + 1]);
                p.y = pack_bf2(v[i + 2], v[i + 3]);
                p.z = pack_bf2(v[i + 4], v[i + 5]);
                p.w = pack_bf2(v[i + 6], v[i + 7]);
                *reinterpret_cast<uint4 *>(o + i) = p;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (i < nv) o[i] = f2bf(v[i]);
        }
    }
}

// The float32 residual of features [nb, nb + 32) of row m (EPI_RESID32), for
// the chunk after the one being stored: its loads overlap that chunk's work.
template <int EPI>
__device__ __forceinline__ void tc_load_res(const LinearArgs &a, float (&r)[32], int m, int nb,
                                            bool live) {
    if constexpr (EPI == EPI_RESID32) {
        if (!live) return;
        const int nv = min(32, a.N - nb);
        const float *o = a.out32 + (size_t)m * a.N + nb;
        if (nv == 32 && ((uintptr_t)o & 15u) == 0) {
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
                const float4 x = *reinterpret_cast<const float4 *>(o + i);
                r[i] = x.x;
                r[i + 1] = x.y;
                r[i + 2] = x.z;
                r[i + 3] = x.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = i < nv ? o[i] : 0.f;
        }
    }
}

// Tile order: groups of kTcGroupM row blocks, row block fastest inside a group,
// so that the tiles running at once share a few X row blocks and each W tile
// is used by kTcGroupM neighbouring tiles while it is still in L2.
constexpr int kTcGroupM = 8;

__device__ __forceinline__ void tc_tile_coords(int t, int tiles_m, int tiles_n, int &m0, int &n0) {
    const int per_group = kTcGroupM * tiles_n;
    const int group = t / per_group;
    const int first = group * kTcGroupM;
    const int gm = min(kTcGroupM, tiles_m - first);
    const int r = t - group * per_group;
    m0 = (first + r % gm) * kTcBM;
    n0 = (r / gm) * kTcBN;
}

template <int EPI>
__global__ void __launch_bounds__(kTcThreads, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
               const LinearArgs a) {
    extern __shared__ unsigned char smem_raw[];
    // 1024-byte alignment for the 128B-swizzled tiles
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        ((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    __shared__ uint64_t full[kTcStages], empty[kTcStages], acc_full[2], acc_empty[2], drained;
    __shared__ uint32_t tmem_base;
    __shared__ int s_abort;
    __shared__ uint16_t s_bias[4][kTcBN];   // the tile's bias, one copy per epilogue warp

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nkb = (a.K + kTcBK - 1) / kTcBK;
    const int tiles_n = (a.N + kTcBN - 1) / kTcBN;
    const int tiles_m = (a.M + kTcBM - 1) / kTcBM;
    const int tiles = tiles_m * tiles_n;

    if (tid == 0) {
        for (int s = 0; s < kTcStages; ++s) {
            tc_mbar_init(&full[s], 1);
            tc_mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            tc_mbar_init(&acc_full[b], 1);
            tc_mbar_init(&acc_empty[b], 4);   // one arrival per epilogue warp
        }
        tc_mbar_init(&drained, 1);
        s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tm_x) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tm_w) : "memory");
    }
    if (warp == 0) {
        // two accumulators of 256 columns: the whole TMEM of the SM (one CTA per SM)
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         tc_smem(&tmem_base)),
                     "n"(2 * kTcBN));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = tmem_base;
    griddep_launch();
    volatile int *abort_flag = &s_abort;

    if (warp == 0) {
        if (lane == 0) {
            // ---- TMA producer: this CTA's tiles back to back through one ring
            griddep_wait();   // X comes from the previous kernel
            long long it = 0;   // ring position over all tiles
            for (int t = blockIdx.x; t < tiles && !*abort_flag; t += gridDim.x) {
                int m0, n0;
                tc_tile_coords(t, tiles_m, tiles_n, m0, n0);
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    const int s = (int)(it % kTcStages);
                    const uint32_t par = (uint32_t)((it / kTcStages) & 1);
                    if (!tc_mbar_wait(&empty[s], par ^ 1u, a.wait_ns)) {
                        *abort_flag = 1;
                        if (a.err) atomicOr(a.err, kErrTimeout);
                        break;
                    }
                    unsigned char *sa = smem + (size_t)s * kTcStageBytes;
                    unsigned char *sb = sa + kTcABytes;
                    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
                                     tc_smem(&full[s])),
                                 "r"(kTcStageBytes)
                                 : "memory");
                    tc_tma_2d(sa, &tm_x, kb * kTcBK, m0, &full[s]);
                    tc_tma_2d(sb, &tm_w, kb * kTcBK, n0, &full[s]);
                }
            }
            // no copy of ours may still be landing when the CTA exits
            for (int i = 0; i < kTcStages && i < it; ++i) {
                const long long j = it - 1 - i;
                if (!tc_mbar_wait(&full[j % kTcStages], (uint32_t)((j / kTcStages) & 1), kTcWaitNs))
                    if (a.err) atomicOr(a.err, kErrTimeout);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---- MMA issuer: tile i accumulates into TMEM buffer i % 2 once the
            // epilogue has drained that buffer's previous tile
            constexpr uint32_t idesc = tc_idesc(kTcBM, kTcBN);
            long long it = 0;
            int lt = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < tiles && ok && !*abort_flag; t += gridDim.x, ++lt) {
                const int b = lt & 1;
                if (!tc_mbar_wait(&acc_empty[b], (uint32_t)(((lt >> 1) & 1) ^ 1), a.wait_ns)) {
                    ok = false;
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t acc = tmem + (uint32_t)(b * kTcBN);
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    const int s = (int)(it % kTcStages);
                    if (!tc_mbar_wait(&full[s], (uint32_t)((it / kTcStages) & 1), a.wait_ns)) {
                        ok = false;
                        break;
                    }
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const uint32_t sa = tc_smem(smem + (size_t)s * kTcStageBytes);
                    const uint32_t sb = sa + kTcABytes;
                    const uint64_t da = tc_desc(sa), db = tc_desc(sb);
#pragma unroll
                    for (int k = 0; k < kTcBK / 16; ++k)   // 16 bf16 = 32 bytes per step
                        tc_mma(acc, da + (uint64_t)(2 * k), db + (uint64_t)(2 * k), idesc,
                               (kb > 0 || k > 0) ? 1u : 0u);
                    tc_commit(&empty[s]);   // stage free once these MMAs have read it
                }
                tc_commit(&acc_full[b]);    // this tile's accumulator complete (or abandoned)
            }
            if (!ok) {
                *abort_flag = 1;
                if (a.err) atomicOr(a.err, kErrTimeout);
            }
            // every MMA of ours has finished before TMEM is freed, on every path
            tc_commit(&drained);
            if (!tc_mbar_wait(&drained, 0, kTcWaitNs) && a.err) atomicOr(a.err, kErrTimeout);
        }
    } else {
        // ---- epilogue: warps 2..5 -> TMEM lane quarters (warp % 4)
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        griddep_wait();   // the residual and the cache belong to earlier kernels too
        int lt = 0;
        for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++lt) {
            const int b = lt & 1;
            int m0, n0;
            tc_tile_coords(t, tiles_m, tiles_n, m0, n0);
            const int m = m0 + row;
            // the tile's bias into this warp's copy while the main loop runs: eight
            // independent loads per lane instead of a round trip per 32-feature chunk
            if (a.bias) {
                __syncwarp();   // the previous tile's reads are done
#pragma unroll
                for (int j = 0; j < kTcBN / 32; ++j) {
                    const int f = lane * (kTcBN / 32) + j;
                    s_bias[quarter][f] = n0 + f < a.N ? a.bias[n0 + f] : (uint16_t)0;
                }
                __syncwarp();
            }
            // longer limit than the MMA issuer's, so that its commits arrive first
            const bool ok = tc_mbar_wait(&acc_full[b], (uint32_t)((lt >> 1) & 1),
                                         3 * (a.wait_ns ? a.wait_ns : kTcWaitNs));
            if (!ok) {
                if (a.err) atomicOr(a.err, kErrTimeout);
                *abort_flag = 1;
                break;
            }
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const bool store = !*abort_flag && m < a.M;
            const uint32_t acc = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(b * kTcBN);
            float res[32], res_next[32];
            tc_load_res<EPI>(a, res, m, n0, store && n0 < a.N);
#pragma unroll 1
            for (int c = 0; c < kTcBN; c += 32) {
                float v[32];
                tc_ld32(acc + (uint32_t)c, v);   // whole warp
                const bool more = c + 32 < kTcBN;
                tc_load_res<EPI>(a, res_next, m, n0 + c + 32, store && more && n0 + c + 32 < a.N);
                if (store && n0 + c < a.N)
                    tc_store_chunk<EPI>(a, v, m, n0 + c, a.bias ? &s_bias[quarter][c] : nullptr, res);
                if constexpr (EPI == EPI_RESID32) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) res[i] = res_next[i];
                }
            }
            // buffer b drained: the MMA issuer may start the tile after next in it
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0)
                asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc_smem(&acc_empty[b]))
                             : "memory");
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "n"(2 * kTcBN));
    }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPoint("cuTensorMapEncodeTiled", &p, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (EncodeTiledFn)p;
    }
    return fn;
}

// 2-D bf16 tensor map over rows x K (row-major), boxes of box_rows x 64, 128B swizzle.
bool gemm_make_map(void *map, const void *base, long long rows, long long K, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || ((uintptr_t)base & 15u) || (K * 2) % 16) return false;
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {(cuuint32_t)kTcBK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(reinterpret_cast<CUtensorMap *>(map), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
              const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D uint8 tensor map over rows x K bytes (row-major int8 weights), boxes of
// box_rows x 128 bytes, 128B swizzle.
bool gemm_make_map_u8(void *map, const void *base, long long rows, long long K, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || ((uintptr_t)base & 15u) || K % 16) return false;
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)K};
    cuuint32_t box[2] = {128u, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(reinterpret_cast<CUtensorMap *>(map), CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
              const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t gemm_map_bytes() { return sizeof(CUtensorMap); }
int gemm_box_rows_x() { return kTcBM; }
int gemm_box_rows_w() { return kTcBN; }

template <int EPI>
static cudaError_t gemm_launch_t(const void *mx, const void *mw, const LinearArgs &a,
                                 cudaStream_t s) {
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<EPI>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kTcSmem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const CUtensorMap &tx = *reinterpret_cast<const CUtensorMap *>(mx);
    const CUtensorMap &tw = *reinterpret_cast<const CUtensorMap *>(mw);
    // persistent: one CTA per SM walks the tiles
    static int sms = 0;
    if (!sms) {
        int dev = 0;
        if (cudaGetDevice(&dev) || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) ||
            sms < 1)
            sms = 1;
    }
    const long long tiles = (long long)((a.M + kTcBM - 1) / kTcBM) * ((a.N + kTcBN - 1) / kTcBN);
    dim3 grid((unsigned)(tiles < sms ? tiles : sms));
    return launch_pdl_smem(gemm_tc_kernel<EPI>, grid, dim3(kTcThreads), kTcSmem, s, tx, tw, a);
}

cudaError_t gemm_prepare() {
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(gemm_tc_kernel<EPI_STORE>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTcSmem)))
        return e;
    if ((e = cudaFuncSetAttribute(gemm_tc_kernel<EPI_GELU>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTcSmem)))
        return e;
    if ((e = cudaFuncSetAttribute(gemm_tc_kernel<EPI_RESID>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTcSmem)))
        return e;
    if ((e = cudaFuncSetAttribute(gemm_tc_kernel<EPI_RESID32>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTcSmem)))
        return e;
    return cudaFuncSetAttribute(gemm_tc_kernel<EPI_QKV>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTcSmem);
}

// X [M][K] and W [N][K] described by maps from gemm_make_map (box rows 128 and
// 256).  K % 8 == 0; bf16 weights only.
cudaError_t launch_gemm_tc(const void *map_x, const void *map_w, const LinearArgs &a,
                           cudaStream_t s) {
    if (a.M <= 0 || a.N <= 0) return cudaSuccess;
    if (a.int8 || a.K % 8) return cudaErrorInvalidValue;
    if (a.epi == EPI_QKV && (a.head_dim % 32 || a.T < 1)) return cudaErrorInvalidValue;
    switch (a.epi) {
        case EPI_STORE: return gemm_launch_t<EPI_STORE>(map_x, map_w, a, s);
        case EPI_GELU: return gemm_launch_t<EPI_GELU>(map_x, map_w, a, s);
        case EPI_RESID: return gemm_launch_t<EPI_RESID>(map_x, map_w, a, s);
        case EPI_RESID32: return gemm_launch_t<EPI_RESID32>(map_x, map_w, a, s);
        case EPI_QKV: return gemm_launch_t<EPI_QKV>(map_x, map_w, a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace bloom
